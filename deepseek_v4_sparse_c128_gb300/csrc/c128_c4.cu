// sm_103a kernels for windows of at most 8 rows (the C4 layout: compress ratio 4 with overlap):
// many small windows per SM at once instead of one window per CTA.
//
//   c4_indexer_kernel<FMT>  head 128: one warp per window; lane l owns columns 4l..4l+3 of all
//                           (up to 8) rows, 16-byte loads of kv and score, the softmax, the exact
//                           variance, RoPE and the FP8 / MXFP4 quantisation all in registers and
//                           warp shuffles.
//   c4_sparse_kernel        head 512: four warps per window; thread i owns columns 4i..4i+3; the
//                           variance meets in shared memory; the 7 nope blocks of 64 columns and the
//                           rope pairs are each handled by half a warp.
//
// Same arithmetic as the oracle's reading of _fused_kv_compress_norm_rope_insert_indexer_attn,
// ..._indexer_mxfp4_attn and ..._sparse_attn on the API page of
// vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache (gather with overlap: 2*ratio rows,
// the newer half at +head, rows at negative positions masked).
#include <cstddef>

#include "c128_device.cuh"

namespace c128 {
namespace {

constexpr int kMaxSmallRows = 8;
constexpr uint32_t kInv6BitsC4 = 0x3e2aaaabu;  // RN32(1/6)

__device__ __forceinline__ uint32_t pack_e2m1x2_c4(float lo, float hi) {
  uint16_t d;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tmov.b16 %0, {t, t};\n}" : "=h"(d) : "f"(hi), "f"(lo));
  return d & 0xffu;
}
__device__ __forceinline__ float pow2_neg_c4(int e) {  // 2^-e for e in [-127, 127]
  return e <= 126 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23) : __uint_as_float(0x00200000u);
}

// One window's softmax-weighted sum for 4 consecutive columns `col` of up to 8 rows.
// Returns false if a block id is out of range (uniform across the threads reading this window).
struct SmallWindow {
  int64_t t, pos, kvs, cp;
  int req;
  uint32_t err;
};

__device__ __forceinline__ SmallWindow read_window(const Params& p, int64_t t) {
  SmallWindow w;
  w.t = t;
  w.req = __ldg(p.ttr + t);
  w.pos = __ldg(p.pos + t);
  w.kvs = __ldg(p.kvslot + t);
  w.err = 0;
  if (w.req < 0 || w.req >= p.bt_rows) w.err |= C128_DEV_BAD_REQ;
  if (w.pos / p.sblk >= p.bt_cols) w.err |= C128_DEV_BAD_BT_COL;
  w.cp = (w.pos / p.ratio) * p.ratio;
  if (w.cp >= p.cs_rows) w.err |= C128_DEV_BAD_COS_ROW;
  if (w.kvs >= p.nkb * p.kv_bs) w.err |= C128_DEV_BAD_KV_SLOT;
  return w;
}

template <int HEAD>
__device__ __forceinline__ bool small_window_comp(const Params& p, const SmallWindow& w, int col, float4& comp) {
  const int n = (1 + p.overlap) * p.ratio;
  const int64_t start = w.pos - n + 1;
  float4 kv[kMaxSmallRows], sc[kMaxSmallRows];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kMaxSmallRows; ++i) {
    kv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    sc[i] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    const int64_t q = start + i;
    if (i < n && q >= 0) {
      const int b = __ldg(p.bt + static_cast<int64_t>(w.req) * p.bt_stride + q / p.sblk);
      if (b < 0 || b >= p.nb) {
        bad = true;
      } else {
        const float* row = p.state + static_cast<int64_t>(b) * p.s0 + (q % p.sblk) * p.s1 + (i >= p.ratio ? HEAD : 0) + col;
        kv[i] = __ldg(reinterpret_cast<const float4*>(row));
        sc[i] = __ldg(reinterpret_cast<const float4*>(row + p.sw));
      }
    }
  }
  if (bad) return false;
  float out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float mx = (&sc[0].x)[k];
#pragma unroll
    for (int i = 1; i < kMaxSmallRows; ++i) mx = fmaxf(mx, (&sc[i].x)[k]);
    const float bias = mx * kLog2e;  // the newest row is always valid, so mx is finite
    float l = 0.f, a = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxSmallRows; ++i) {
      const float e = ex2_approx(fmaf((&sc[i].x)[k], kLog2e, -bias));
      l += e;
      a = fmaf(e, (&kv[i].x)[k], a);
    }
    out[k] = __fdiv_rn(a, l);
  }
  comp = make_float4(out[0], out[1], out[2], out[3]);
  return true;
}

// Exact-variance pieces: 128-bit aligned squares of a thread's 4 values.
__device__ __forceinline__ uint32_t biased_exp(uint32_t u) { return u ? ((u >> 23) ? (u >> 23) : 1u) : 0u; }
__device__ __forceinline__ void add_square(uint32_t u, uint32_t emax, unsigned long long& lo, unsigned long long& hi,
                                           bool& fallback) {
  if (u == 0u) return;
  const uint32_t f = u >> 23;
  const uint32_t d = emax - biased_exp(u);
  if (d > 32u) {
    fallback = true;
    return;
  }
  const unsigned long long M = f ? ((u & 0x7fffffu) | 0x800000u) : (u & 0x7fffffu);
  const unsigned long long M2 = M * M;
  const int sh = 64 - 2 * static_cast<int>(d);
  const unsigned long long tlo = sh == 64 ? 0ull : (M2 << sh);
  const unsigned long long thi = sh == 0 ? 0ull : (M2 >> (64 - sh));
  const unsigned long long nlo = lo + tlo;
  hi += thi + (nlo < lo ? 1ull : 0ull);
  lo = nlo;
}
__device__ __forceinline__ uint32_t special_bits(uint32_t u) {
  return (u >> 23) == 255u ? ((u & 0x7fffffu) ? 2u : 1u) : 0u;
}
__device__ __forceinline__ void warp_sum128(unsigned long long& lo, unsigned long long& hi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long olo = __shfl_xor_sync(0xffffffffu, lo, o);
    const unsigned long long ohi = __shfl_xor_sync(0xffffffffu, hi, o);
    const unsigned long long nlo = lo + olo;
    hi += ohi + (nlo < lo ? 1ull : 0ull);
    lo = nlo;
  }
}

// ----------------------------------------------------------------- head 128: a warp per window
template <int FMT>
__global__ void __launch_bounds__(256) c4_indexer_kernel(Params p) {
  __shared__ __align__(16) float comp_s[8][128];  // per warp, for the rare exact-variance slow path
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = 4 * lane;
  grid_dependency_wait();
  const int32_t* list = reinterpret_cast<const int32_t*>(p.ws + 1);
  const int64_t A = min(static_cast<int64_t>(*reinterpret_cast<volatile unsigned*>(&p.ws->count)), p.T);
  const int64_t nw = static_cast<int64_t>(gridDim.x) * 8;
  constexpr int kTok = FMT == C128_FORMAT_INDEXER_FP8 ? 128 : 64;
  const float2 wa = *reinterpret_cast<const float2*>(p.rms_w + col);
  const float2 wb = *reinterpret_cast<const float2*>(p.rms_w + col + 2);
  for (int64_t a = static_cast<int64_t>(blockIdx.x) * 8 + warp; a < A; a += nw) {
    SmallWindow w = read_window(p, list[a]);
    float4 c;
    if (!w.err && !small_window_comp<128>(p, w, col, c)) w.err |= C128_DEV_BAD_BLOCK;
    if (w.err) {
      if (lane == 0) atomicOr(&p.ws->err, w.err);
      continue;
    }
    if (p.comp_out != nullptr) *reinterpret_cast<float4*>(p.comp_out + w.t * 128 + col) = c;
    // variance = RN32(exact(sum c^2) / 128)
    const uint32_t u[4] = {__float_as_uint(c.x) & 0x7fffffffu, __float_as_uint(c.y) & 0x7fffffffu,
                           __float_as_uint(c.z) & 0x7fffffffu, __float_as_uint(c.w) & 0x7fffffffu};
    const uint32_t emax = __reduce_max_sync(0xffffffffu, max(max(biased_exp(u[0]), biased_exp(u[1])),
                                                             max(biased_exp(u[2]), biased_exp(u[3]))));
    const uint32_t special = __reduce_or_sync(0xffffffffu, special_bits(u[0]) | special_bits(u[1]) |
                                                               special_bits(u[2]) | special_bits(u[3]));
    unsigned long long lo = 0ull, hi = 0ull;
    bool fb = false;
    if (special == 0u)
      for (int k = 0; k < 4; ++k) add_square(u[k], emax, lo, hi, fb);
    warp_sum128(lo, hi);
    fb = __any_sync(0xffffffffu, fb);
    float rrms = 0.f;
    if (fb) {
      *reinterpret_cast<float4*>(&comp_s[warp][col]) = c;
      __syncwarp();
    }
    if (lane == 0) {
      float var;
      if (special & 2u) var = __int_as_float(0x7fc00000);
      else if (special & 1u) var = INFINITY;
      else if (fb) var = mean_square_exact_slow(comp_s[warp], 128, 7);
      else var = round_u128_to_f32(lo, hi, 2 * static_cast<int>(emax) - 371, false);
      rrms = __frsqrt_rn(__fadd_rn(var, p.eps));
    }
    __syncwarp();
    rrms = __shfl_sync(0xffffffffu, rrms, 0);
    const float n[4] = {__fmul_rn(__fmul_rn(c.x, rrms), wa.x), __fmul_rn(__fmul_rn(c.y, rrms), wa.y),
                        __fmul_rn(__fmul_rn(c.z, rrms), wb.x), __fmul_rn(__fmul_rn(c.w, rrms), wb.y)};
    // RoPE of pairs j = 2*lane + k; pairs >= 32 (lanes 16..31) rotate, the others use cos 1, sin 0
    const float* cs_row = p.cs + w.cp * p.cs_stride;
    float x[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = 2 * lane + k;
      float C = 1.0f, S = 0.0f;
      if (j >= 32) {
        C = __ldg(cs_row + (j - 32));
        S = __ldg(cs_row + kRope / 2 + (j - 32));
      }
      const float ev = n[2 * k], od = n[2 * k + 1];
      const uint32_t b = pack_bf16x2(__fsub_rn(__fmul_rn(ev, C), __fmul_rn(od, S)),
                                     __fadd_rn(__fmul_rn(od, C), __fmul_rn(ev, S)));
      x[2 * k] = __uint_as_float(b << 16);
      x[2 * k + 1] = __uint_as_float(b & 0xffff0000u);
    }
    const int64_t kb = w.kvs / p.kv_bs, off = w.kvs % p.kv_bs;
    uint8_t* base = p.kc + kb * p.kc_stride0;
    uint8_t* tok = base + off * kTok;
    uint8_t* scale = base + p.kv_bs * kTok + off * 4;
    const uint32_t am_l = max(max(__float_as_uint(x[0]) & 0x7fffffffu, __float_as_uint(x[1]) & 0x7fffffffu),
                              max(__float_as_uint(x[2]) & 0x7fffffffu, __float_as_uint(x[3]) & 0x7fffffffu));
    if constexpr (FMT == C128_FORMAT_INDEXER_FP8) {
      const float amax = fmaxf(__uint_as_float(__reduce_max_sync(0xffffffffu, am_l)), __uint_as_float(kAbsmaxFloorBits));
      const uint32_t raw = __float_as_uint(__fmul_rn(amax, __uint_as_float(kInv448Bits)));
      const int e = static_cast<int>(raw >> 23) - 127 + ((raw & 0x7fffffu) ? 1 : 0);
      const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
      float y[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = fminf(fmaxf(__fmul_rn(x[k], inv), -448.f), 448.f);
      *reinterpret_cast<uint32_t*>(tok + col) =
          static_cast<uint32_t>(pack_e4m3x2(y[0], y[1])) | (static_cast<uint32_t>(pack_e4m3x2(y[2], y[3])) << 16);
      if (lane == 0) *reinterpret_cast<float*>(scale) = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
    } else {
      // MXFP4 block b = values 32b..32b+31 = lanes 8b..8b+7
      uint32_t am = am_l;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, o));
      const float amax = fmaxf(__uint_as_float(am), 6.0f * __uint_as_float(0x00800000u));
      const uint32_t ratio = __float_as_uint(__fmul_rn(amax, __uint_as_float(kInv6BitsC4)));
      const int e = min(max(static_cast<int>(ratio >> 23) - 127 + ((ratio & 0x7fffffu) ? 1 : 0), -127), 127);
      const float inv = pow2_neg_c4(e);
      const uint32_t b0 = pack_e2m1x2_c4(__fmul_rn(x[0], inv), __fmul_rn(x[1], inv));
      const uint32_t b1 = pack_e2m1x2_c4(__fmul_rn(x[2], inv), __fmul_rn(x[3], inv));
      *reinterpret_cast<uint16_t*>(tok + 2 * lane) = static_cast<uint16_t>(b0 | (b1 << 8));
      if ((lane & 7) == 0) scale[lane >> 3] = static_cast<uint8_t>(e + 127);
    }
  }
}

// ------------------------------------------------------------ head 512: four warps per window
constexpr int kQuadThreads = 128;
struct __align__(16) QuadSmem {  // 16-byte aligned: comp[] takes float4 stores in both quads
  unsigned long long lo[4], hi[4];
  uint32_t emax[4], special[4], fb[4];
  float comp[512];
  float rrms;
};
static_assert(offsetof(QuadSmem, comp) % 16 == 0 && sizeof(QuadSmem) % 16 == 0, "float4 access to QuadSmem::comp");
__device__ __forceinline__ void quad_bar(int quad) {
  asm volatile("bar.sync %0, %1;" ::"r"(3 + quad), "n"(kQuadThreads) : "memory");
}

__global__ void __launch_bounds__(256) c4_sparse_kernel(Params p) {
  __shared__ __align__(16) QuadSmem Q[2];
  const int quad = threadIdx.x >> 7, qt = threadIdx.x & 127;  // thread qt of the quad: columns 4qt..4qt+3
  const int qw = qt >> 5, lane = qt & 31;
  const int col = 4 * qt;
  QuadSmem& S = Q[quad];
  grid_dependency_wait();
  const int32_t* list = reinterpret_cast<const int32_t*>(p.ws + 1);
  const int64_t A = min(static_cast<int64_t>(*reinterpret_cast<volatile unsigned*>(&p.ws->count)), p.T);
  const int64_t nq = static_cast<int64_t>(gridDim.x) * 2;
  const float2 wa = *reinterpret_cast<const float2*>(p.rms_w + col);
  const float2 wb = *reinterpret_cast<const float2*>(p.rms_w + col + 2);
  for (int64_t a = static_cast<int64_t>(blockIdx.x) * 2 + quad; a < A; a += nq) {
    SmallWindow w = read_window(p, list[a]);
    float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
    bool bad = false;
    if (!w.err) bad = !small_window_comp<512>(p, w, col, c);
    // every thread read the same block ids; the vote keeps the decision uniform regardless
    quad_bar(quad);
    if (w.err || bad) {
      if (qt == 0) atomicOr(&p.ws->err, w.err | (bad ? static_cast<uint32_t>(C128_DEV_BAD_BLOCK) : 0u));
      continue;
    }
    if (p.comp_out != nullptr) *reinterpret_cast<float4*>(p.comp_out + w.t * 512 + col) = c;
    *reinterpret_cast<float4*>(&S.comp[col]) = c;
    const uint32_t u[4] = {__float_as_uint(c.x) & 0x7fffffffu, __float_as_uint(c.y) & 0x7fffffffu,
                           __float_as_uint(c.z) & 0x7fffffffu, __float_as_uint(c.w) & 0x7fffffffu};
    const uint32_t em_w = __reduce_max_sync(0xffffffffu, max(max(biased_exp(u[0]), biased_exp(u[1])),
                                                             max(biased_exp(u[2]), biased_exp(u[3]))));
    const uint32_t sp_w = __reduce_or_sync(0xffffffffu, special_bits(u[0]) | special_bits(u[1]) |
                                                            special_bits(u[2]) | special_bits(u[3]));
    if (lane == 0) {
      S.emax[qw] = em_w;
      S.special[qw] = sp_w;
    }
    quad_bar(quad);
    const uint32_t emax = max(max(S.emax[0], S.emax[1]), max(S.emax[2], S.emax[3]));
    const uint32_t special = S.special[0] | S.special[1] | S.special[2] | S.special[3];
    unsigned long long lo = 0ull, hi = 0ull;
    bool fb = false;
    if (special == 0u)
      for (int k = 0; k < 4; ++k) add_square(u[k], emax, lo, hi, fb);
    warp_sum128(lo, hi);
    fb = __any_sync(0xffffffffu, fb);
    if (lane == 0) {
      S.lo[qw] = lo;
      S.hi[qw] = hi;
      S.fb[qw] = fb;
    }
    quad_bar(quad);
    if (qt == 0) {
      unsigned long long vlo = 0ull, vhi = 0ull;
      for (int k = 0; k < 4; ++k) {
        const unsigned long long nlo = vlo + S.lo[k];
        vhi += S.hi[k] + (nlo < vlo ? 1ull : 0ull);
        vlo = nlo;
      }
      float var;
      if (special & 2u) var = __int_as_float(0x7fc00000);
      else if (special & 1u) var = INFINITY;
      else if (S.fb[0] | S.fb[1] | S.fb[2] | S.fb[3]) var = mean_square_exact_slow(S.comp, 512, 9);
      else var = round_u128_to_f32(vlo, vhi, 2 * static_cast<int>(emax) - 373, false);
      S.rrms = __frsqrt_rn(__fadd_rn(var, p.eps));
    }
    quad_bar(quad);
    const float rrms = S.rrms;
    const float n[4] = {__fmul_rn(__fmul_rn(c.x, rrms), wa.x), __fmul_rn(__fmul_rn(c.y, rrms), wa.y),
                        __fmul_rn(__fmul_rn(c.z, rrms), wb.x), __fmul_rn(__fmul_rn(c.w, rrms), wb.y)};
    const int64_t kb = w.kvs / p.kv_bs, off = w.kvs % p.kv_bs;
    uint8_t* base = p.kc + kb * p.kc_stride0;
    uint8_t* tok = base + off * kTokenStride;
    uint8_t* scale = base + p.kv_bs * kTokenStride + off * kScaleDim;
    const int blk = col / kQuantBlock;  // 0..7; half-warp h = lanes 16h..16h+15 of warp qw is block 2qw+h
    if (blk < kNope / kQuantBlock) {
      const uint32_t b01 = pack_bf16x2(n[0], n[1]), b23 = pack_bf16x2(n[2], n[3]);
      const float x[4] = {__uint_as_float(b01 << 16), __uint_as_float(b01 & 0xffff0000u), __uint_as_float(b23 << 16),
                          __uint_as_float(b23 & 0xffff0000u)};
      uint32_t am = max(max(__float_as_uint(x[0]) & 0x7fffffffu, __float_as_uint(x[1]) & 0x7fffffffu),
                        max(__float_as_uint(x[2]) & 0x7fffffffu, __float_as_uint(x[3]) & 0x7fffffffu));
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) am = max(am, __shfl_xor_sync(0x0000ffffu << (lane & 16), am, o));
      const float amax = fmaxf(__uint_as_float(am), __uint_as_float(kAbsmaxFloorBits));
      const uint32_t raw = __float_as_uint(__fmul_rn(amax, __uint_as_float(kInv448Bits)));
      const int e = static_cast<int>(raw >> 23) - 127 + ((raw & 0x7fffffu) ? 1 : 0);
      const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
      float y[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = fminf(fmaxf(__fmul_rn(x[k], inv), -448.f), 448.f);
      *reinterpret_cast<uint32_t*>(tok + col) =
          static_cast<uint32_t>(pack_e4m3x2(y[0], y[1])) | (static_cast<uint32_t>(pack_e4m3x2(y[2], y[3])) << 16);
      if ((col & (kQuantBlock - 1)) == 0) scale[blk] = static_cast<uint8_t>(min(max(e + 127, 0), 255));
    } else {
      // rope: pairs (448 + 2j, 449 + 2j), j = (col - 448) / 2 + k
      const float* cs_row = p.cs + w.cp * p.cs_stride;
      uint32_t out[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int j = (col - kNope) / 2 + k;
        const float C = __ldg(cs_row + j), Sn = __ldg(cs_row + kRope / 2 + j);
        const float ev = n[2 * k], od = n[2 * k + 1];
        out[k] = pack_bf16x2(__fsub_rn(__fmul_rn(ev, C), __fmul_rn(od, Sn)), __fadd_rn(__fmul_rn(od, C), __fmul_rn(ev, Sn)));
      }
      *reinterpret_cast<uint2*>(tok + kNope + 2 * (col - kNope)) = make_uint2(out[0], out[1]);
      if (col == kNope) scale[kNope / kQuantBlock] = 0;
    }
  }
}

}  // namespace

bool small_window_path(const Params& p) { return (1 + p.overlap) * p.ratio <= kMaxSmallRows; }

template <typename K>
int resident_ctas(K kernel, int sm_count) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
  return per_sm * sm_count;
}

cudaError_t launch_small(const Params& p, const LaunchCfg& cfg, cudaStream_t stream) {
  // one wave of resident CTAs (each loops over its share of the windows)
  static int grid_sparse = 0, grid_fp8 = 0, grid_fp4 = 0;
  if (grid_sparse == 0) {
    grid_sparse = resident_ctas(c4_sparse_kernel, cfg.sm_count);
    grid_fp8 = resident_ctas(c4_indexer_kernel<C128_FORMAT_INDEXER_FP8>, cfg.sm_count);
    grid_fp4 = resident_ctas(c4_indexer_kernel<C128_FORMAT_INDEXER_MXFP4>, cfg.sm_count);
  }
  const int grid = p.fmt == C128_FORMAT_SPARSE_FP8 ? grid_sparse : p.fmt == C128_FORMAT_INDEXER_FP8 ? grid_fp8 : grid_fp4;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(grid));
  lc.blockDim = dim3(256);
  lc.dynamicSmemBytes = 0;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = (cfg.pdl && cfg.ev_begin == nullptr) ? 1 : 0;
  if (p.fmt == C128_FORMAT_SPARSE_FP8) return cudaLaunchKernelEx(&lc, c4_sparse_kernel, p);
  if (p.fmt == C128_FORMAT_INDEXER_FP8) return cudaLaunchKernelEx(&lc, c4_indexer_kernel<C128_FORMAT_INDEXER_FP8>, p);
  return cudaLaunchKernelEx(&lc, c4_indexer_kernel<C128_FORMAT_INDEXER_MXFP4>, p);
}

}  // namespace c128
