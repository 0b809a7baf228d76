/*
 * CPU oracle for the DeepSeek-V4 C128 KV compressor:
 *   window gather -> per-column softmax -> weighted sum -> RMSNorm
 *   -> FP8 e4m3 / UE8M0 quant (nope 448) + GPT-J RoPE (rope 64, bf16) -> paged k_cache store.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously-correct statement of what
 * the op computes. Only the tests, the package smoke check and the benchmark's CPU-baseline leg
 * may load it. The CUDA library shares no code with it.
 *
 * Source of the semantics: vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache,
 * kernel _fused_kv_compress_norm_rope_insert_sparse_attn (docs.vllm.ai API page, sections
 * "Gather state cache entries", "Softmax + weighted sum", "RMSNorm", "KV cache pointers",
 * "FP8 UE8M0 quant", "GPT-J RoPE"), and vLLM PR #44230 (Summary: head 512, state width 512,
 * compress ratio 128, no overlap, state block 8).
 *
 * Readings taken where the pages leave a step open. The fused kernel's listing on the API page
 * states the operations in Triton (`%`, tl.softmax, tl.sum, tl.rsqrt, .to(bfloat16) and
 * .to(float8e4nv)) but not their precision, rounding or evaluation order, so:
 *   - positions < 0 are inactive: the page's window-end test uses a modulo under which p = -1
 *     would count as a window end whose rows are all masked ("Gather state cache entries",
 *     mask_pos = pos >= 0), a window with no row to weight;
 *   - softmax and weighted sum ("Gather state cache entries", tl.softmax then tl.sum) are
 *     evaluated in binary64 and rounded once to fp32 (comp32); their summation order is free,
 *     and the GPU is held to a tolerance on comp32, not to its bits;
 *   - variance = RN32( exact(sum c^2) / 512 ) ("RMSNorm": tl.sum of the squares over HEAD_SIZE),
 *     the sum taken exactly (big-integer accumulator) so that its order cannot matter;
 *   - rrms = the correctly rounded fp32 1/sqrt(RN32(var + eps)) (tl.rsqrt's accuracy is not
 *     stated; the correctly rounded value is the one precision-free reading), computed in binary64;
 *   - every other fp32 product / sum is one IEEE fp32 operation, left to right as printed
 *     ("RMSNorm": compressed_kv * rrms * rms_w; "GPT-J RoPE": even*cos - odd*sin), no FMA;
 *   - fp32 -> bf16 and fp32 -> e4m3 round to nearest, ties to even (the casts' default mode);
 *     e4m3 saturates at FP8_MAX = 448 after the page's clamp and keeps the sign (so -0 and
 *     negative underflow give 0x80);
 *   - the UE8M0 exponent is the exact ceil(log2(raw)), raw = RN32(absmax * RN32(1/448))
 *     ("FP8 UE8M0 quant" multiplies by the reciprocal and takes ceil of log2; for every
 *     positive bf16 absmax at or above the 1e-4 floor the exact and the approximate log2 give the
 *     same integer, so the exact one is used).
 *
 * Build: cc -O2 -ffp-contract=off -fPIC -shared c128_oracle.c -lm
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define HEAD 512          /* head size */
#define NOPE 448          /* fp8 columns */
#define ROPE 64           /* bf16 rope columns */
#define STATE_WIDTH 512   /* kv columns; score columns follow */
#define ROW 1024          /* fp32 values per state row */
#define SBLK 8            /* state-cache block size (rows) */
#define RATIO 128         /* compress ratio */
#define QBLK 64           /* quant block (columns per UE8M0 scale) */
#define NQ 7              /* nope quant blocks */
#define TOKEN_STRIDE 576  /* bytes of token data per k_cache slot */
#define SCALE_DIM 8       /* scale bytes per slot: 7 real + 1 zero pad */
#define FP8_MAX 448.0f

/* error bits, same meaning as the device error word of the CUDA library */
#define ORC_BAD_REQ 1
#define ORC_BAD_BT_COL 2
#define ORC_BAD_BLOCK 4
#define ORC_BAD_COS_ROW 8
#define ORC_BAD_KV_SLOT 16

static uint32_t f2u(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float u2f(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* ---------------------------------------------------------------------------------------- */
/* fp32 -> bf16, round to nearest, ties to even (bf16 = the upper 16 bits of binary32).       */
uint16_t c128o_bf16(float x) {
    uint32_t u = f2u(x);
    uint32_t upper = u >> 16, rem = u & 0xFFFFu;
    if (rem > 0x8000u || (rem == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}
static float bf16_value(float x) { return u2f((uint32_t)c128o_bf16(x) << 16); }

/* ---------------------------------------------------------------------------------------- */
/* e4m3fn (OCP FP8): sign, 4 exponent bits (bias 7), 3 mantissa bits; no infinity; 0x7F/0xFF  */
/* are NaN, so the largest finite magnitude is code 0x7E = 1.75 * 2^8 = 448.                  */
static double e4m3_magnitude(int code) { /* code in [0, 126] */
    int E = (code >> 3) & 15, m = code & 7;
    if (E == 0) return ldexp((double)m / 8.0, -6);
    return ldexp(1.0 + (double)m / 8.0, E - 7);
}
/* Nearest finite code by exhaustive search, ties to the even code (even mantissa LSB);       */
/* magnitudes above 448 saturate to 0x7E. The sign bit of x is kept.                           */
uint8_t c128o_e4m3(float x) {
    double a = fabs((double)x);
    int best = 0;
    double bestd = a;  /* distance to code 0 */
    for (int c = 1; c <= 126; ++c) {
        double d = fabs(e4m3_magnitude(c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) { best = c; bestd = d; }
    }
    return (uint8_t)(best | ((f2u(x) >> 31) ? 0x80 : 0));
}

/* ---------------------------------------------------------------------------------------- */
/* Smallest integer e with 2^e >= r, for a positive finite r (exact, via frexp).                */
int c128o_ceil_log2(float r) {
    int k;
    double f = frexp((double)r, &k); /* r = f * 2^k, f in [0.5, 1) */
    return (f == 0.5) ? k - 1 : k;
}

/* ---------------------------------------------------------------------------------------- */
/* RN32( (sum_i c_i^2) / 512 ) with the sum taken exactly.                                     */
/* Every c = M * 2^(e-24) with M < 2^24 an integer, so c^2 = M^2 * 2^(2e-48) and the sum is an */
/* integer multiple of 2^-344 (smallest fp32 magnitude 2^-149 has e = -148). A 640-bit         */
/* accumulator of 32-bit limbs holds every term and the 512-term sum without loss.              */
#define NLIMB 20
/* RN32( (sum_i c_i^2) / 2^log2n ) over n = 2^log2n <= 512 values, the sum taken exactly. */
static float exact_mean_square(const float* c, int n, int log2n) {
    uint32_t acc[NLIMB];
    memset(acc, 0, sizeof acc);
    for (int i = 0; i < n; ++i) {
        float x = fabsf(c[i]);
        if (x == 0.0f) continue;
        if (!isfinite(x)) return isnan(x) ? NAN : INFINITY; /* not reached by finite inputs */
        int e;
        float f = frexpf(x, &e);
        uint64_t M = (uint64_t)ldexpf(f, 24);          /* exact: 24-bit integer */
        uint64_t sq = M * M;                            /* < 2^48 */
        int shift = 2 * e - 48 + 344;                   /* bit offset of sq's LSB */
        /* add sq << shift into the limb array */
        int limb = shift / 32, bit = shift % 32;
        uint64_t carry = 0;
        uint32_t parts[3] = {
            (uint32_t)(sq << bit),
            (uint32_t)((sq << bit) >> 32),
            (uint32_t)(bit ? (sq >> (64 - bit)) : 0)};
        for (int j = 0; j < NLIMB - limb; ++j) {
            uint64_t add = (j < 3) ? parts[j] : 0;
            if (j >= 3 && carry == 0) break;
            uint64_t s = (uint64_t)acc[limb + j] + add + carry;
            acc[limb + j] = (uint32_t)s;
            carry = s >> 32;
        }
    }
    /* value = acc * 2^-344 / 2^log2n; round to fp32 (normal or subnormal), RNE. */
    int msb = -1;
    for (int j = NLIMB - 1; j >= 0 && msb < 0; --j)
        if (acc[j]) for (int b = 31; b >= 0; --b) if (acc[j] >> b & 1u) { msb = 32 * j + b; break; }
    if (msb < 0) return 0.0f;
    const int k = -344 - log2n;
    int lsb = msb - 23;
    if (lsb < -149 - k) lsb = -149 - k;               /* subnormal results keep fewer bits */
    /* lsb >= 195 + log2n > 0 here, so there is always a round bit below it */
    uint64_t q = 0;
    int round_up = 0;
    for (int b = msb; b >= lsb; --b) q = (q << 1) | (acc[b / 32] >> (b % 32) & 1u);
    int rbit = acc[(lsb - 1) / 32] >> ((lsb - 1) % 32) & 1u;
    int sticky = 0;
    for (int b = lsb - 2; b >= 0 && !sticky; --b) sticky = acc[b / 32] >> (b % 32) & 1u;
    if (rbit && (sticky || (q & 1u))) round_up = 1;
    q += (uint64_t)round_up;
    return (float)ldexp((double)q, lsb + k);         /* exact; >= 2^128 becomes +inf */
}
float c128o_mean_square_512(const float* c) { return exact_mean_square(c, HEAD, 9); }
float c128o_mean_square_128(const float* c) { return exact_mean_square(c, 128, 7); }

/* ---------------------------------------------------------------------------------------- */
/* rrms = RN32(1 / sqrt(v)), evaluated as IEEE binary64 sqrt and division rounded once to fp32. */
/* For every positive finite fp32 v this is the correctly rounded reciprocal square root       */
/* (checked exhaustively over all 2^31 - 2^23 - 1 such v by tests/rsqrt_exhaustive.c).         */
float c128o_rsqrt(float v) { return (float)(1.0 / sqrt((double)v)); }

/* ---------------------------------------------------------------------------------------- */
/* RMSNorm -> quant -> RoPE on one compressed vector, producing the 576 token bytes and the   */
/* 8 scale bytes of one k_cache slot.                                                          */
void c128o_epilogue(const float* comp32, const float* rms_w, float eps, const float* cos_sin_row,
                    uint8_t* token_bytes, uint8_t* scale_bytes) {
    /* RMSNorm: variance = sum(c^2)/512, rrms = rsqrt(variance + eps), normed = c * rrms * w */
    float var32 = c128o_mean_square_512(comp32);
    float v = var32 + eps;
    float rrms = c128o_rsqrt(v);
    float normed[HEAD];
    for (int c = 0; c < HEAD; ++c) {
        float t = comp32[c] * rrms;
        normed[c] = t * rms_w[c];
    }
    /* nope: bf16 round, per-64-column absmax (floor 1e-4), UE8M0 exponent, scale, clamp, e4m3 */
    const float inv_fp8_max = (float)(1.0 / 448.0);
    const float floor_amax = (float)1e-4;
    for (int b = 0; b < NQ; ++b) {
        float x[QBLK];
        float amax = 0.0f;
        for (int i = 0; i < QBLK; ++i) {
            x[i] = bf16_value(normed[b * QBLK + i]);
            float a = fabsf(x[i]);
            if (a > amax) amax = a;
        }
        if (amax < floor_amax) amax = floor_amax;
        float raw = amax * inv_fp8_max;
        int e = c128o_ceil_log2(raw);
        float inv_scale = (float)ldexp(1.0, -e);
        for (int i = 0; i < QBLK; ++i) {
            float y = x[i] * inv_scale;
            if (y > FP8_MAX) y = FP8_MAX;
            if (y < -FP8_MAX) y = -FP8_MAX;
            token_bytes[b * QBLK + i] = c128o_e4m3(y);
        }
        int enc = e + 127;
        if (enc > 255) enc = 255;
        if (enc < 0) enc = 0;
        scale_bytes[b] = (uint8_t)enc;
    }
    scale_bytes[NQ] = 0;
    /* rope: pair j = (448+2j, 449+2j); cos at [j], sin at [32+j]; stored as bf16 LE */
    for (int j = 0; j < ROPE / 2; ++j) {
        float ev = normed[NOPE + 2 * j], od = normed[NOPE + 2 * j + 1];
        float C = cos_sin_row[j], S = cos_sin_row[ROPE / 2 + j];
        float ec = ev * C, os = od * S, oc = od * C, es = ev * S;
        float ne = ec - os;
        float no = oc + es;
        uint16_t be = c128o_bf16(ne), bo = c128o_bf16(no);
        token_bytes[NOPE + 4 * j + 0] = (uint8_t)(be & 0xFF);
        token_bytes[NOPE + 4 * j + 1] = (uint8_t)(be >> 8);
        token_bytes[NOPE + 4 * j + 2] = (uint8_t)(bo & 0xFF);
        token_bytes[NOPE + 4 * j + 3] = (uint8_t)(bo >> 8);
    }
}

/* ---------------------------------------------------------------------------------------- */
/* Per-column softmax over the 128 window rows of score, weighted sum of kv, in binary64,    */
/* rounded once to fp32. rows[i] points at the 1024 floats of window row i.                   */
void c128o_compress_window(const float* const* rows, float* comp32) {
    for (int c = 0; c < HEAD; ++c) {
        double m = -INFINITY;
        for (int i = 0; i < RATIO; ++i) {
            double s = rows[i][STATE_WIDTH + c];
            if (s > m) m = s;
        }
        double w[RATIO], Z = 0.0;
        for (int i = 0; i < RATIO; ++i) {
            w[i] = exp((double)rows[i][STATE_WIDTH + c] - m);
            Z += w[i];
        }
        double acc = 0.0;
        for (int i = 0; i < RATIO; ++i) acc += (w[i] / Z) * (double)rows[i][c];
        comp32[c] = (float)acc;
    }
}

/* ---------------------------------------------------------------------------------------- */
/* The whole op over tokens (all of them, or the listed subset), in token order.               */
/* Index arguments follow the CUDA library's boundary: block table rows of bt_cols int32      */
/* entries at bt_row_stride; state [num_blocks, 8, 1024] fp32 with element strides st_s0,      */
/* st_s1 (innermost contiguous); cos_sin [max_pos, 64] fp32 with row stride cs_stride;         */
/* k_cache blocks of kv_block_size slots at kc_block_stride bytes.                             */
/* Returns the OR of error bits of tokens that were active but named out-of-range indices     */
/* (those tokens write nothing). comp_out, if given, receives comp32 of each computed token.  */
int c128o_forward(int64_t num_tokens, const int32_t* token_to_req, const int64_t* positions,
                  const int64_t* slot_mapping, const int32_t* block_table, int64_t num_reqs,
                  int64_t bt_cols, int64_t bt_row_stride, const float* state, int64_t num_blocks,
                  int64_t st_s0, int64_t st_s1, const float* rms_w, float eps, const float* cos_sin,
                  int64_t max_pos, int64_t cs_stride, uint8_t* k_cache, int64_t num_kv_blocks,
                  int64_t kv_block_size, int64_t kc_block_stride, const int64_t* kv_slot_mapping,
                  float* comp_out, const int64_t* token_subset, int64_t n_subset) {
    int err = 0;
    int64_t n = token_subset ? n_subset : num_tokens;
    for (int64_t ii = 0; ii < n; ++ii) {
        int64_t t = token_subset ? token_subset[ii] : ii;
        if (t < 0 || t >= num_tokens) continue;
        int64_t slot = slot_mapping[t], p = positions[t], kvs = kv_slot_mapping[t];
        /* activity: slot >= 0, a window end ((p+1) % 128 == 0, p >= 0), and a kv slot */
        if (slot < 0 || p < 0 || (p + 1) % RATIO != 0 || kvs < 0) continue;
        int64_t r = token_to_req[t];
        int terr = 0;
        if (r < 0 || r >= num_reqs) terr |= ORC_BAD_REQ;
        if (p / SBLK >= bt_cols) terr |= ORC_BAD_BT_COL;
        int64_t cp = (p / RATIO) * RATIO;
        if (cp >= max_pos) terr |= ORC_BAD_COS_ROW;
        if (kvs >= num_kv_blocks * kv_block_size) terr |= ORC_BAD_KV_SLOT;
        const float* rows[RATIO];
        if (!(terr & (ORC_BAD_REQ | ORC_BAD_BT_COL))) {
            int64_t start = p - (RATIO - 1);
            for (int i = 0; i < RATIO; ++i) {
                int64_t q = start + i;
                int64_t b = block_table[r * bt_row_stride + q / SBLK];
                if (b < 0 || b >= num_blocks) { terr |= ORC_BAD_BLOCK; break; }
                rows[i] = state + b * st_s0 + (q % SBLK) * st_s1;
            }
        }
        if (terr) { err |= terr; continue; }
        float comp32[HEAD];
        c128o_compress_window(rows, comp32);
        if (comp_out) memcpy(comp_out + t * HEAD, comp32, sizeof comp32);
        int64_t blk = kvs / kv_block_size, off = kvs % kv_block_size;
        uint8_t* base = k_cache + blk * kc_block_stride;
        c128o_epilogue(comp32, rms_w, eps, cos_sin + cp * cs_stride,
                       base + off * TOKEN_STRIDE,
                       base + kv_block_size * TOKEN_STRIDE + off * SCALE_DIM);
    }
    return err;
}

/* ---------------------------------------------------------------------------------------- */
/* Array forms of the two encoders, for exhaustive checks.                                     */
void c128o_bf16_n(const float* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = c128o_bf16(x[i]);
}
void c128o_e4m3_n(const float* x, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = c128o_e4m3(x[i]);
}


/* ========================================================================================== */
/* The other configurations of the fused kernels on the API page:                             */
/*   format 0  _fused_kv_compress_norm_rope_insert_sparse_attn  (head 512: nope FP8 + rope bf16) */
/*   format 1  _fused_kv_compress_norm_rope_insert_indexer_attn (head 128: RoPE, then one FP8    */
/*             block with an fp32 power-of-two scale)                                           */
/*   format 2  _fused_kv_compress_norm_rope_insert_indexer_mxfp4_attn (head 128: RoPE, bf16     */
/*             round, MXFP4 E2M1 pairs with one UE8M0 byte per 32 values)                       */
/* with any compress ratio, with or without overlap ("Gather state cache entries": 2*ratio rows */
/* when overlapping; the newer `ratio` rows read kv and score at +head; rows at negative        */
/* positions are left out of the softmax). A state row is kv[state_width] then score[state_width]. */
typedef struct c128o_cfg {
    int32_t head;         /* 512 (format 0) or 128 (formats 1, 2) */
    int32_t rope;         /* 64 */
    int32_t ratio;        /* compress ratio (window end: (p+1) % ratio == 0) */
    int32_t overlap;      /* 0 or 1 */
    int32_t state_width;  /* kv columns of a state row; as many score columns follow */
    int32_t format;       /* 0, 1, 2 as above */
} c128o_cfg;

#define IDX_HEAD 128
#define IDX_TOKEN_FP8 128    /* indexer FP8: 128 e4m3 bytes per token, then one fp32 scale */
#define IDX_TOKEN_FP4 64     /* indexer MXFP4: 64 bytes of E2M1 pairs, then 4 UE8M0 bytes */
#define IDX_SCALE_DIM 4

/* E2M1 (OCP MXFP4 element): sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6. Nearest by exhaustive search, ties to the even code, values beyond
 * 6 saturate, the sign bit of x is kept. The API page calls a helper _fp32x2_to_fp4x2 on the
 * scaled pairs of _fused_kv_compress_norm_rope_insert_indexer_mxfp4_attn but does not print its
 * body, so the rounding is a reading: round to nearest with ties to the even code (the OCP
 * microscaling convention for conversions into E2M1) and saturation at 6, the largest
 * magnitude, because the block scale is chosen so that |x| * 2^-e <= 6 up to rounding. */
uint8_t c128o_e2m1(float x) {
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double a = fabs((double)x);
    int best = 0;
    double bestd = a;
    for (int c = 1; c < 8; ++c) {
        double d = fabs(mag[c] - a);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) { best = c; bestd = d; }
    }
    return (uint8_t)(best | ((f2u(x) >> 31) ? 0x8 : 0));
}

/* Softmax-weighted sum of one window for `head` columns: rows[i] == NULL marks a masked row;
 * kv of row i at rows[i][koff[i] + c], its score at rows[i][soff[i] + c]. binary64, one rounding. */
static void compress_window_ex(int nrows, const float* const* rows, const int* koff, const int* soff, int head,
                               float* comp32) {
    for (int c = 0; c < head; ++c) {
        double m = -INFINITY;
        for (int i = 0; i < nrows; ++i) {
            if (!rows[i]) continue;
            double s = rows[i][soff[i] + c];
            if (s > m) m = s;
        }
        double Z = 0.0, acc = 0.0;
        double w[256];
        for (int i = 0; i < nrows; ++i) {
            w[i] = rows[i] ? exp((double)rows[i][soff[i] + c] - m) : 0.0;
            Z += w[i];
        }
        for (int i = 0; i < nrows; ++i)
            if (rows[i]) acc += (w[i] / Z) * (double)rows[i][koff[i] + c];
        comp32[c] = (float)acc;
    }
}

/* RMSNorm over 128 columns then GPT-J RoPE of every pair, the 32 nope pairs with cos 1, sin 0
 * exactly as the page writes it (its masked loads give those values), the 32 rope pairs with
 * cos/sin of the window row. Output: the rotated fp32 pairs, even then odd. */
static void indexer_norm_rope(const float* comp32, const float* rms_w, float eps, const float* cs_row,
                              float* even, float* odd) {
    float var32 = c128o_mean_square_128(comp32);
    float rrms = c128o_rsqrt(var32 + eps);
    float normed[IDX_HEAD];
    for (int c = 0; c < IDX_HEAD; ++c) {
        float t = comp32[c] * rrms;
        normed[c] = t * rms_w[c];
    }
    const int nope_pairs = (IDX_HEAD - 64) / 2;
    for (int j = 0; j < IDX_HEAD / 2; ++j) {
        float ev = normed[2 * j], od = normed[2 * j + 1];
        float C = 1.0f, S = 0.0f;
        if (j >= nope_pairs) { C = cs_row[j - nope_pairs]; S = cs_row[32 + j - nope_pairs]; }
        float ec = ev * C, os = od * S, oc = od * C, es = ev * S;
        even[j] = ec - os;
        odd[j] = oc + es;
    }
}

/* format 1: bf16 round, one absmax over 128 (floor 1e-4), e = ceil(log2(absmax * RN32(1/448))),
 * 128 e4m3 codes of clamp(x * 2^-e, +-448), fp32 scale 2^e stored little-endian. */
void c128o_epilogue_indexer_fp8(const float* comp32, const float* rms_w, float eps, const float* cs_row,
                                uint8_t* token_bytes, uint8_t* scale_bytes) {
    float even[IDX_HEAD / 2], odd[IDX_HEAD / 2], x[IDX_HEAD];
    indexer_norm_rope(comp32, rms_w, eps, cs_row, even, odd);
    float amax = 0.0f;
    for (int j = 0; j < IDX_HEAD / 2; ++j) {
        x[2 * j] = bf16_value(even[j]);
        x[2 * j + 1] = bf16_value(odd[j]);
    }
    for (int c = 0; c < IDX_HEAD; ++c) if (fabsf(x[c]) > amax) amax = fabsf(x[c]);
    if (amax < (float)1e-4) amax = (float)1e-4;
    float raw = amax * (float)(1.0 / 448.0);
    int e = c128o_ceil_log2(raw);
    float inv_scale = (float)ldexp(1.0, -e);
    for (int c = 0; c < IDX_HEAD; ++c) {
        float y = x[c] * inv_scale;
        if (y > FP8_MAX) y = FP8_MAX;
        if (y < -FP8_MAX) y = -FP8_MAX;
        token_bytes[c] = c128o_e4m3(y);
    }
    float scale = (float)ldexp(1.0, e);
    uint32_t u = f2u(scale);
    for (int b = 0; b < 4; ++b) scale_bytes[b] = (uint8_t)(u >> (8 * b));
}

/* format 2: bf16 round of the rotated pairs; per 32 values (16 pairs) amax (floor 6*2^-126),
 * e = clamp(ceil(log2(amax * RN32(1/6))), -127, 127), E2M1 codes of x * 2^-e, byte j of the block =
 * even code in the low nibble, odd code in the high nibble; UE8M0 byte e + 127. */
void c128o_epilogue_indexer_mxfp4(const float* comp32, const float* rms_w, float eps, const float* cs_row,
                                  uint8_t* token_bytes, uint8_t* scale_bytes) {
    float even[IDX_HEAD / 2], odd[IDX_HEAD / 2];
    indexer_norm_rope(comp32, rms_w, eps, cs_row, even, odd);
    for (int j = 0; j < IDX_HEAD / 2; ++j) { even[j] = bf16_value(even[j]); odd[j] = bf16_value(odd[j]); }
    const float floor_amax = (float)(6.0 * ldexp(1.0, -126));
    const float inv6 = (float)(1.0 / 6.0);
    for (int b = 0; b < IDX_HEAD / 32; ++b) {
        float amax = 0.0f;
        for (int j = 16 * b; j < 16 * b + 16; ++j) {
            if (fabsf(even[j]) > amax) amax = fabsf(even[j]);
            if (fabsf(odd[j]) > amax) amax = fabsf(odd[j]);
        }
        if (amax < floor_amax) amax = floor_amax;
        int e = c128o_ceil_log2(amax * inv6);
        if (e < -127) e = -127;
        if (e > 127) e = 127;
        float inv_scale = (float)ldexp(1.0, -e);
        for (int j = 16 * b; j < 16 * b + 16; ++j)
            token_bytes[j] = (uint8_t)(c128o_e2m1(even[j] * inv_scale) | (c128o_e2m1(odd[j] * inv_scale) << 4));
        scale_bytes[b] = (uint8_t)(e + 127);
    }
}

/* The op for any configuration above (same index arguments as c128o_forward; state rows of
 * st_s1 >= 2 * state_width floats, blocks of `state_block` rows; comp_out is [T, head]). */
int c128o_forward_ex(const c128o_cfg* cfg, int64_t num_tokens, const int32_t* token_to_req,
                     const int64_t* positions, const int64_t* slot_mapping, const int32_t* block_table,
                     int64_t num_reqs, int64_t bt_cols, int64_t bt_row_stride, const float* state,
                     int64_t num_blocks, int64_t state_block, int64_t st_s0, int64_t st_s1,
                     const float* rms_w, float eps, const float* cos_sin, int64_t max_pos, int64_t cs_stride,
                     uint8_t* k_cache, int64_t num_kv_blocks, int64_t kv_block_size, int64_t kc_block_stride,
                     const int64_t* kv_slot_mapping, float* comp_out, const int64_t* token_subset,
                     int64_t n_subset) {
    const int head = cfg->head, ratio = cfg->ratio, nrows = (1 + (cfg->overlap ? 1 : 0)) * ratio;
    if (nrows > 256 || (cfg->format == 0 && head != HEAD) || (cfg->format != 0 && head != IDX_HEAD)) return -1;
    const int64_t tok_bytes = cfg->format == 0 ? TOKEN_STRIDE : cfg->format == 1 ? IDX_TOKEN_FP8 : IDX_TOKEN_FP4;
    const int64_t sc_bytes = cfg->format == 0 ? SCALE_DIM : IDX_SCALE_DIM;
    int err = 0;
    int64_t n = token_subset ? n_subset : num_tokens;
    for (int64_t ii = 0; ii < n; ++ii) {
        int64_t t = token_subset ? token_subset[ii] : ii;
        if (t < 0 || t >= num_tokens) continue;
        int64_t slot = slot_mapping[t], p = positions[t], kvs = kv_slot_mapping[t];
        if (slot < 0 || p < 0 || (p + 1) % ratio != 0 || kvs < 0) continue;
        int64_t r = token_to_req[t];
        int terr = 0;
        if (r < 0 || r >= num_reqs) terr |= ORC_BAD_REQ;
        if (p / state_block >= bt_cols) terr |= ORC_BAD_BT_COL;
        int64_t cp = (p / ratio) * ratio;
        if (cp >= max_pos) terr |= ORC_BAD_COS_ROW;
        if (kvs >= num_kv_blocks * kv_block_size) terr |= ORC_BAD_KV_SLOT;
        const float* rows[256];
        int koff[256], soff[256];
        if (!(terr & (ORC_BAD_REQ | ORC_BAD_BT_COL))) {
            int64_t start = p - nrows + 1;
            for (int i = 0; i < nrows; ++i) {
                int64_t q = start + i;
                int ho = i >= ratio ? head : 0;
                koff[i] = ho;
                soff[i] = cfg->state_width + ho;
                if (q < 0) { rows[i] = NULL; continue; }
                int64_t b = block_table[r * bt_row_stride + q / state_block];
                if (b < 0 || b >= num_blocks) { terr |= ORC_BAD_BLOCK; break; }
                rows[i] = state + b * st_s0 + (q % state_block) * st_s1;
            }
        }
        if (terr) { err |= terr; continue; }
        float comp32[HEAD];
        compress_window_ex(nrows, rows, koff, soff, head, comp32);
        if (comp_out) memcpy(comp_out + t * head, comp32, sizeof(float) * head);
        int64_t blk = kvs / kv_block_size, off = kvs % kv_block_size;
        uint8_t* base = k_cache + blk * kc_block_stride;
        uint8_t* tok = base + off * tok_bytes;
        uint8_t* sc = base + kv_block_size * tok_bytes + off * sc_bytes;
        const float* cs_row = cos_sin + cp * cs_stride;
        if (cfg->format == 0) c128o_epilogue(comp32, rms_w, eps, cs_row, tok, sc);
        else if (cfg->format == 1) c128o_epilogue_indexer_fp8(comp32, rms_w, eps, cs_row, tok, sc);
        else c128o_epilogue_indexer_mxfp4(comp32, rms_w, eps, cs_row, tok, sc);
    }
    return err;
}
