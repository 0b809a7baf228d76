// sm_103a kernel for the other configurations of the compressor: C4-style overlapping windows
// (2 * ratio rows, the newer half read at +head, rows at negative positions masked) and the
// head-128 indexer caches (one FP8 block with an fp32 scale, or MXFP4). What is computed follows
// _fused_kv_compress_norm_rope_insert_sparse_attn, _fused_kv_compress_norm_rope_insert_indexer_attn
// and _fused_kv_compress_norm_rope_insert_indexer_mxfp4_attn on the API page of
// vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache.
//
// gather_kernel<HEAD, FMT> is persistent over the planning kernel's list (window a -> CTA a mod
// grid, all windows being the same size). Per window its 256 threads form HEAD/4 column groups
// (float4) times 256/(HEAD/4) row groups; each thread streams its rows' kv and score float4s with
// 16-byte loads and folds them into an online softmax; the row groups' partial states meet in
// shared memory and are merged in row-group order. The 512-wide format then runs the shared
// fused epilogue; the indexer formats run a 64-thread epilogue (RMSNorm, RoPE of the last 32
// pairs, bf16 round, then FP8 with one fp32 scale or MXFP4 with a UE8M0 byte per 32 values).
#include <cstddef>

#include "c128_device.cuh"

namespace c128 {
namespace {

template <int HEAD>
struct GatherGeo {
  static constexpr int kThreads = 256;
  static constexpr int kColGroups = HEAD / 4;
  static constexpr int kRowGroups = kThreads / kColGroups;  // 2 (head 512) or 8 (head 128)
  static constexpr int kChunk = 4;                          // rows folded per online update
};

constexpr int kIdxHead = 128;
constexpr int kIdxThreads = 64;      // indexer epilogue: thread j owns the pair (2j, 2j+1)
constexpr uint32_t kInv6Bits = 0x3e2aaaabu;  // RN32(1/6)

// Scratch of the 64-thread indexer epilogue.
struct IdxSmem {
  unsigned long long red_lo[2], red_hi[2];
  uint32_t red_emax[2], red_special[2], red_fallback[2], red_amax[2];
  float comp[kIdxHead];
  float rrms;
};

template <int HEAD>
struct GatherSmem {
  float pm[GatherGeo<HEAD>::kRowGroups][HEAD];  // partial running max (log2 units)
  float pl[GatherGeo<HEAD>::kRowGroups][HEAD];  // partial sum of weights
  float pa[GatherGeo<HEAD>::kRowGroups][HEAD];  // partial weighted sum of kv
  EpiSmem epi;
  IdxSmem idx;
};

static_assert(sizeof(float) * GatherGeo<512>::kRowGroups * 512 % 16 == 0 &&
                  sizeof(float) * GatherGeo<128>::kRowGroups * 128 % 16 == 0,
              "float4 access to the partial arrays");
static_assert(offsetof(IdxSmem, comp) % 8 == 0, "float2 access to IdxSmem::comp");

__device__ __forceinline__ void idx_bar() { asm volatile("bar.sync 2, %0;" ::"n"(kIdxThreads) : "memory"); }

// two fp32 -> packed E2M1 pair (round to nearest even, saturating); `lo` in bits 0..3
__device__ __forceinline__ uint32_t pack_e2m1x2(float lo, float hi) {
  uint16_t d;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tmov.b16 %0, {t, t};\n}"
      : "=h"(d)
      : "f"(hi), "f"(lo));
  return d & 0xffu;
}
// 2^-e as fp32 for e in [-127, 127] (2^-127 is the subnormal 0x00200000)
__device__ __forceinline__ float pow2_neg(int e) {
  return e <= 126 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23) : __uint_as_float(0x00200000u);
}

// Epilogue of one 128-wide window run by threads 0..63 (thread j: columns 2j, 2j+1 = pair j).
template <int FMT>
__device__ void indexer_epilogue(IdxSmem& E, int j, float cv0, float cv1, float2 w, float eps, const float* cs_row,
                                 uint8_t* tok, uint8_t* scale, float* comp_dst) {
  const int warp = j >> 5, lane = j & 31;
  if (comp_dst != nullptr) *reinterpret_cast<float2*>(comp_dst + 2 * j) = make_float2(cv0, cv1);
  *reinterpret_cast<float2*>(E.comp + 2 * j) = make_float2(cv0, cv1);
  // variance = RN32(exact(sum c^2) / 128), as in the 512-wide epilogue
  const uint32_t u0 = __float_as_uint(cv0) & 0x7fffffffu, u1 = __float_as_uint(cv1) & 0x7fffffffu;
  const uint32_t f0 = u0 >> 23, f1 = u1 >> 23;
  uint32_t special = (f0 == 255u ? ((u0 & 0x7fffffu) ? 2u : 1u) : 0u) | (f1 == 255u ? ((u1 & 0x7fffffu) ? 2u : 1u) : 0u);
  const uint32_t eb0 = u0 ? (f0 ? f0 : 1u) : 0u, eb1 = u1 ? (f1 ? f1 : 1u) : 0u;
  const uint32_t emax_w = __reduce_max_sync(0xffffffffu, max(eb0, eb1));
  special = __reduce_or_sync(0xffffffffu, special);
  if (lane == 0) {
    E.red_emax[warp] = emax_w;
    E.red_special[warp] = special;
  }
  idx_bar();
  const uint32_t emax = max(E.red_emax[0], E.red_emax[1]);
  special = E.red_special[0] | E.red_special[1];
  unsigned long long lo = 0ull, hi = 0ull;
  bool fallback = false;
  if (special == 0u) {
    const uint32_t us[2] = {u0, u1}, fs[2] = {f0, f1}, es[2] = {eb0, eb1};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (us[k] == 0u) continue;
      const uint32_t d = emax - es[k];
      if (d > 32u) {
        fallback = true;
        continue;
      }
      const unsigned long long M = fs[k] ? ((us[k] & 0x7fffffu) | 0x800000u) : (us[k] & 0x7fffffu);
      const unsigned long long M2 = M * M;
      const int sh = 64 - 2 * static_cast<int>(d);
      const unsigned long long tlo = sh == 64 ? 0ull : (M2 << sh);
      const unsigned long long thi = sh == 0 ? 0ull : (M2 >> (64 - sh));
      const unsigned long long nlo = lo + tlo;
      hi += thi + (nlo < lo ? 1ull : 0ull);
      lo = nlo;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long olo = __shfl_xor_sync(0xffffffffu, lo, o);
    const unsigned long long ohi = __shfl_xor_sync(0xffffffffu, hi, o);
    const unsigned long long nlo = lo + olo;
    hi += ohi + (nlo < lo ? 1ull : 0ull);
    lo = nlo;
  }
  const bool fb_w = __any_sync(0xffffffffu, fallback);
  if (lane == 0) {
    E.red_lo[warp] = lo;
    E.red_hi[warp] = hi;
    E.red_fallback[warp] = fb_w;
  }
  idx_bar();
  if (j == 0) {
    float var;
    const unsigned long long vlo = E.red_lo[0] + E.red_lo[1];
    const unsigned long long vhi = E.red_hi[0] + E.red_hi[1] + (vlo < E.red_lo[0] ? 1ull : 0ull);
    if (special & 2u) {
      var = __int_as_float(0x7fc00000);
    } else if (special & 1u) {
      var = INFINITY;
    } else if (E.red_fallback[0] | E.red_fallback[1]) {
      var = mean_square_exact_slow(E.comp, kIdxHead, 7);
    } else {
      var = round_u128_to_f32(vlo, vhi, 2 * static_cast<int>(emax) - 371, false);
    }
    E.rrms = __frsqrt_rn(__fadd_rn(var, eps));
  }
  idx_bar();
  const float rrms = E.rrms;
  const float n0 = __fmul_rn(__fmul_rn(cv0, rrms), w.x);
  const float n1 = __fmul_rn(__fmul_rn(cv1, rrms), w.y);
  // GPT-J RoPE of every pair; the 32 nope pairs with cos 1, sin 0 as the page computes them
  float C = 1.0f, S = 0.0f;
  if (j >= 32) {
    C = __ldg(cs_row + (j - 32));
    S = __ldg(cs_row + kRope / 2 + (j - 32));
  }
  const float ne = __fsub_rn(__fmul_rn(n0, C), __fmul_rn(n1, S));
  const float no = __fadd_rn(__fmul_rn(n1, C), __fmul_rn(n0, S));
  const uint32_t b = pack_bf16x2(ne, no);
  const float x0 = __uint_as_float(b << 16), x1 = __uint_as_float(b & 0xffff0000u);
  if constexpr (FMT == C128_FORMAT_INDEXER_FP8) {
    // one block: absmax over all 128 values (floor 1e-4), e = ceil(log2(absmax * RN32(1/448)))
    const uint32_t am_w =
        __reduce_max_sync(0xffffffffu, max(__float_as_uint(x0) & 0x7fffffffu, __float_as_uint(x1) & 0x7fffffffu));
    if (lane == 0) E.red_amax[warp] = am_w;
    idx_bar();
    const float amax = fmaxf(__uint_as_float(max(E.red_amax[0], E.red_amax[1])), __uint_as_float(kAbsmaxFloorBits));
    const uint32_t raw = __float_as_uint(__fmul_rn(amax, __uint_as_float(kInv448Bits)));
    const int e = static_cast<int>(raw >> 23) - 127 + ((raw & 0x7fffffu) ? 1 : 0);
    const float inv_scale = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    const float y0 = fminf(fmaxf(__fmul_rn(x0, inv_scale), -448.f), 448.f);
    const float y1 = fminf(fmaxf(__fmul_rn(x1, inv_scale), -448.f), 448.f);
    *reinterpret_cast<uint16_t*>(tok + 2 * j) = pack_e4m3x2(y0, y1);
    if (j == 0) *reinterpret_cast<float*>(scale) = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
  } else {
    // MXFP4: blocks of 16 pairs (32 values); amax (floor 6*2^-126), e = ceil(log2(amax*RN32(1/6)))
    uint32_t am = max(__float_as_uint(x0) & 0x7fffffffu, __float_as_uint(x1) & 0x7fffffffu);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, o));
    const float amax = fmaxf(__uint_as_float(am), 6.0f * __uint_as_float(0x00800000u));
    const uint32_t ratio = __float_as_uint(__fmul_rn(amax, __uint_as_float(kInv6Bits)));
    int e = static_cast<int>(ratio >> 23) - 127 + ((ratio & 0x7fffffu) ? 1 : 0);
    e = min(max(e, -127), 127);
    const float inv_scale = pow2_neg(e);
    tok[j] = static_cast<uint8_t>(pack_e2m1x2(__fmul_rn(x0, inv_scale), __fmul_rn(x1, inv_scale)));
    if ((j & 15) == 0) scale[j >> 4] = static_cast<uint8_t>(e + 127);
  }
}

template <int HEAD, int FMT>
__global__ void __launch_bounds__(256, 3) gather_kernel(Params p) {
  using G = GatherGeo<HEAD>;
  __shared__ __align__(16) GatherSmem<HEAD> S;
  const int tid = threadIdx.x;
  const int cg = tid % G::kColGroups, rg = tid / G::kColGroups;
  const int col = 4 * cg;
  // a programmatic dependent of the planning pass (which waits for the kernel before it): nothing
  // global is touched before it has completed
  grid_dependency_wait();
  __shared__ uint32_t chunk_prefix[kMaxPlanChunks + 1];
  __shared__ uint32_t active;
  if (tid < 32) {
    const uint32_t a = plan_prefix_warp(p, chunk_prefix, tid);
    if (tid == 0) active = a;
  }
  __syncthreads();
  const int64_t A = active;
  const int nrows = (1 + p.overlap) * p.ratio;
  constexpr int kTokBytes = FMT == C128_FORMAT_SPARSE_FP8 ? kTokenStride : (FMT == C128_FORMAT_INDEXER_FP8 ? 128 : 64);
  constexpr int kScaleBytes = FMT == C128_FORMAT_SPARSE_FP8 ? kScaleDim : 4;
  for (int64_t a = blockIdx.x; a < A; a += gridDim.x) {
    __syncthreads();  // the previous window's epilogue is done with the shared scratch
    const int64_t t = plan_token(p, chunk_prefix, static_cast<uint32_t>(a));
    const int req = __ldg(p.ttr + t);
    const int64_t pos = __ldg(p.pos + t), kvs = __ldg(p.kvslot + t);
    uint32_t err = 0;
    if (req < 0 || req >= p.bt_rows) err |= C128_DEV_BAD_REQ;
    if (pos / p.sblk >= p.bt_cols) err |= C128_DEV_BAD_BT_COL;
    const int64_t cp = (pos / p.ratio) * p.ratio;
    if (cp >= p.cs_rows) err |= C128_DEV_BAD_COS_ROW;
    if (kvs >= p.nkb * p.kv_bs) err |= C128_DEV_BAD_KV_SLOT;
    const int64_t start = pos - nrows + 1;
    // every thread checks the block ids of its rows; the CTA votes
    bool bad = false;
    if (!(err & (C128_DEV_BAD_REQ | C128_DEV_BAD_BT_COL))) {
      for (int i = rg; i < nrows; i += G::kRowGroups) {
        const int64_t q = start + i;
        if (q < 0) continue;
        const int b = __ldg(p.bt + static_cast<int64_t>(req) * p.bt_stride + q / p.sblk);
        bad |= b < 0 || b >= p.nb;
      }
    }
    if (__syncthreads_or(bad)) err |= C128_DEV_BAD_BLOCK;
    if (err) {
      if (tid == 0) atomicOr(&p.ws->err, err);
      continue;
    }
    // online softmax over this thread's rows (i = rg, rg + kRowGroups, ...), kChunk rows at a time
    float m[4], l[4], acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      m[k] = -INFINITY;
      l[k] = acc[k] = 0.f;
    }
    for (int i0 = rg; i0 < nrows; i0 += G::kRowGroups * G::kChunk) {
      float4 kv[G::kChunk], sc[G::kChunk];
#pragma unroll
      for (int r = 0; r < G::kChunk; ++r) {
        const int i = i0 + r * G::kRowGroups;
        const int64_t q = start + i;
        kv[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        sc[r] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (i < nrows && q >= 0) {
          const int b = __ldg(p.bt + static_cast<int64_t>(req) * p.bt_stride + q / p.sblk);
          const float* row = p.state + static_cast<int64_t>(b) * p.s0 + (q % p.sblk) * p.s1 +
                             (i >= p.ratio ? HEAD : 0) + col;
          kv[r] = __ldg(reinterpret_cast<const float4*>(row));
          sc[r] = __ldg(reinterpret_cast<const float4*>(row + p.sw));
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float mx = (&sc[0].x)[k];
#pragma unroll
        for (int r = 1; r < G::kChunk; ++r) mx = fmaxf(mx, (&sc[r].x)[k]);
        const float nm = fmaxf(m[k], mx * kLog2e);
        const float bias = nm == -INFINITY ? 0.f : nm;
        const float rs = ex2_approx(m[k] - bias);
        float ps = 0.f, pk = 0.f;
#pragma unroll
        for (int r = 0; r < G::kChunk; ++r) {
          const float e = ex2_approx(fmaf((&sc[r].x)[k], kLog2e, -bias));
          ps += e;
          pk = fmaf(e, (&kv[r].x)[k], pk);
        }
        m[k] = nm;
        l[k] = fmaf(l[k], rs, ps);
        acc[k] = fmaf(acc[k], rs, pk);
      }
    }
    *reinterpret_cast<float4*>(&S.pm[rg][col]) = make_float4(m[0], m[1], m[2], m[3]);
    *reinterpret_cast<float4*>(&S.pl[rg][col]) = make_float4(l[0], l[1], l[2], l[3]);
    *reinterpret_cast<float4*>(&S.pa[rg][col]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    __syncthreads();

    // merge the row groups in order; thread j finishes columns 2j, 2j+1
    constexpr int kFinishers = HEAD / 2;
    if (tid < kFinishers) {
      float cv[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int c = 2 * tid + k;
        float M = -INFINITY;
#pragma unroll
        for (int g = 0; g < G::kRowGroups; ++g) M = fmaxf(M, S.pm[g][c]);
        const float B = M == -INFINITY ? 0.f : M;
        float L = 0.f, Acc = 0.f;
#pragma unroll
        for (int g = 0; g < G::kRowGroups; ++g) {
          const float s = ex2_approx(S.pm[g][c] - B);
          L = fmaf(S.pl[g][c], s, L);
          Acc = fmaf(S.pa[g][c], s, Acc);
        }
        cv[k] = __fdiv_rn(Acc, L);
      }
      const float2 w = *reinterpret_cast<const float2*>(p.rms_w + 2 * tid);
      const int64_t kb = kvs / p.kv_bs, off = kvs % p.kv_bs;
      uint8_t* base = p.kc + kb * p.kc_stride0;
      uint8_t* tok = base + off * kTokBytes;
      uint8_t* scale = base + p.kv_bs * kTokBytes + off * kScaleBytes;
      float* comp_dst = p.comp_out ? p.comp_out + t * HEAD : nullptr;
      const float* cs_row = p.cs + cp * p.cs_stride;
      if constexpr (FMT == C128_FORMAT_SPARSE_FP8) {
        const int cw = tid >> 5, lane = tid & 31;
        float cosv = 0.f, sinv = 0.f;
        if (cw == kConsumerWarps - 1) {
          cosv = __ldg(cs_row + lane);
          sinv = __ldg(cs_row + kRope / 2 + lane);
        }
        epilogue(S.epi, tid, cv[0], cv[1], w, p.eps, cosv, sinv, tok, scale, comp_dst, false);
      } else {
        indexer_epilogue<FMT>(S.idx, tid, cv[0], cv[1], w, p.eps, cs_row, tok, scale, comp_dst);
      }
    }
  }
}

template <int HEAD, int FMT>
cudaError_t launch_gather_t(const Params& p, const LaunchCfg& cfg, cudaStream_t stream) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(3 * cfg.sm_count));
  lc.blockDim = dim3(GatherGeo<HEAD>::kThreads);
  lc.dynamicSmemBytes = 0;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = (cfg.pdl && cfg.ev_begin == nullptr) ? 1 : 0;
  return cudaLaunchKernelEx(&lc, gather_kernel<HEAD, FMT>, p);
}

}  // namespace

cudaError_t launch_gather(const Params& p, const LaunchCfg& cfg, cudaStream_t stream) {
  if (p.fmt == C128_FORMAT_SPARSE_FP8) return launch_gather_t<512, C128_FORMAT_SPARSE_FP8>(p, cfg, stream);
  if (p.fmt == C128_FORMAT_INDEXER_FP8) return launch_gather_t<128, C128_FORMAT_INDEXER_FP8>(p, cfg, stream);
  return launch_gather_t<128, C128_FORMAT_INDEXER_MXFP4>(p, cfg, stream);
}

}  // namespace c128
