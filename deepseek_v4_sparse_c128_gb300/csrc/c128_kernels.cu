// sm_103a kernels of the DeepSeek-V4 C128 KV compressor.
//
//   plan_kernel      compacts the indices of active tokens (slot >= 0, position at a window end,
//                    kv slot >= 0) into the workspace list; one pass over the per-token metadata.
//   compress_kernel  persistent, one CTA per SM. Warp 0 claims windows from the list and resolves
//                    their 16 state blocks through the block table; warp 1 streams each block
//                    (8 rows x 4 KiB = 32 KiB) into a 6-stage shared-memory ring with
//                    cp.async.bulk (TMA bulk copies completing on mbarriers); warps 2..9 run an
//                    online per-column softmax and weighted sum over the 128 rows and then the
//                    fused epilogue: exact RMS variance, RMSNorm, bf16 round, per-64-column
//                    absmax / UE8M0 exponent / e4m3 codes, GPT-J RoPE to bf16, paged store.
//
// What is computed follows _fused_kv_compress_norm_rope_insert_sparse_attn on the API page of
// vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache. The pages' own Blackwell design
// (vLLM PR #44230, "Why This Is Faster": 8 warps x 16 rows per 64-column head tile with a
// cross-warp reduce, then a separate store kernel) is replaced here by whole-window CTAs, so no
// cross-CTA or cross-warp softmax combine and no fp32 scratch round trip are needed.
//
// Every wait is bounded (kWaitTimeoutNs); on expiry the kernel records C128_DEV_TIMEOUT, drains
// its own copies in flight and returns.
#include "c128_internal.h"
#include "c128compress.h"

#include <math.h>

namespace c128 {
namespace {

// ------------------------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase with the given parity; give up after kWaitTimeoutNs, or as soon as
// *abort_flag is set when one is given.
__device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}
// L2 policy of the state stream: evict-first by default (every state byte is read once).
#ifndef C128_L2_POLICY
#define C128_L2_POLICY 1
#endif
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
#if C128_L2_POLICY == 1
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
#else
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
#endif
  return pol;
}
// TMA bulk copy global -> shared; completion is counted in bytes on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// two fp32 -> packed bf16x2 (round to nearest even); `lo` lands in bits 0..15
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// two fp32 -> packed e4m3x2 (round to nearest even, saturating); `lo` lands in bits 0..7
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}
constexpr int kConsumerThreads = 32 * kConsumerWarps;
__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}
// Barrier over the consumer warps that also returns the OR of `pred` over them (uniform).
__device__ __forceinline__ bool consumer_bar_or(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(pred)), "n"(kConsumerThreads)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ------------------------------------------------------------------------------ plan kernel
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(Params p) {
  launch_dependents();
  __shared__ uint32_t warp_base[kPlanThreads / 32];
  __shared__ uint32_t cta_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kPlanTokensPerCta;
  uint32_t flags = 0;
#pragma unroll
  for (int i = 0; i < kPlanTokensPerThread; ++i) {
    const int64_t t = base + i * kPlanThreads + tid;
    if (t < p.T) {
      const int64_t s = __ldg(p.slot + t), pos = __ldg(p.pos + t), kv = __ldg(p.kvslot + t);
      const bool active = (s >= 0) & (pos >= 0) & ((pos & (kRatio - 1)) == kRatio - 1) & (kv >= 0);
      flags |= static_cast<uint32_t>(active) << i;
    }
  }
  const uint32_t n = __popc(flags);
  uint32_t incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_base[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    uint32_t tot = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) {
      const uint32_t v = warp_base[w];
      warp_base[w] = tot;
      tot += v;
    }
    cta_base = tot ? atomicAdd(&p.ws->count, tot) : 0u;
  }
  __syncthreads();
  uint32_t out = cta_base + warp_base[warp] + incl - n;
  int32_t* list = reinterpret_cast<int32_t*>(p.ws + 1);
#pragma unroll
  for (int i = 0; i < kPlanTokensPerThread; ++i)
    if ((flags >> i) & 1u) list[out++] = static_cast<int32_t>(base + i * kPlanThreads + tid);
}

// --------------------------------------------------------------------------- compress kernel
struct __align__(16) WinDesc {
  const float* src[kWindowBlocks];  // row 0 of each of the window's 16 state blocks
  uint8_t* kv_dst;                  // 576 token bytes of the k_cache slot
  uint8_t* scale_dst;               // 8 scale bytes of the slot
  const float* cs_row;              // cos_sin_cache row of the window start
  float* comp_dst;                  // optional fp32 export
  int32_t kind;                     // 0: window, 1: no more windows
  int32_t pad[3];
};

// Consumer-only scratch of the fused epilogue (one window at a time).
struct EpiSmem {
  unsigned long long red_lo[kConsumerWarps];
  unsigned long long red_hi[kConsumerWarps];
  uint32_t red_emax[kConsumerWarps];
  uint32_t red_special[kConsumerWarps];
  uint32_t red_fallback[kConsumerWarps];
  float comp[kHead];
  float rrms;
};

// Shared memory of the persistent (list-mode) kernel.
struct Smem {
  float stage[kStages][kStateBlock * kRow];
  WinDesc desc[kDescSlots];
  uint64_t full[kStages];        // stage landed (1 arrival + 32 KiB of transactions)
  uint64_t empty[kStages];       // stage consumed (one arrival per consumer warp)
  uint64_t dfull[kDescSlots];    // window descriptor written (scheduler)
  uint64_t dempty[kDescSlots];   // descriptor released (copy warp + consumer warps)
  EpiSmem epi;
  int abort_flag;
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kInv448Bits = 0x3b124925u;   // RN32(1/448)
constexpr uint32_t kAbsmaxFloorBits = 0x38d1b717u;  // RN32(1e-4)

__device__ __forceinline__ double pow2_double(int e) {  // e in [-1022, 1023]
  return __longlong_as_double(static_cast<long long>(e + 1023) << 52);
}

// Round V * 2^k to fp32 (nearest even, subnormals kept), where V = hi:lo is a 128-bit integer and
// `sticky_in` says the true value is a little above V * 2^k (bits below V's LSB were non-zero).
__device__ float round_u128_to_f32(unsigned long long lo, unsigned long long hi, int k, bool sticky_in) {
  if ((lo | hi) == 0ull) return 0.0f;  // sticky_in never comes with V == 0
  const int msb = hi ? 127 - __clzll(static_cast<long long>(hi)) : 63 - __clzll(static_cast<long long>(lo));
  int lsb = msb - 23;
  if (lsb < -149 - k) lsb = -149 - k;
  unsigned long long q;
  if (lsb <= 0) {
    q = lo;  // msb <= 23, exact (sticky_in bits are below half an ulp of the smallest subnormal? no:
             // only reached when the value needs no rounding at all, i.e. sticky_in is false)
    lsb = 0;
  } else {
    if (lsb > msb + 1) return 0.0f;  // below half the smallest subnormal
    q = (lsb >= 64) ? (hi >> (lsb - 64)) : ((lo >> lsb) | (lsb ? (hi << (64 - lsb)) : 0ull));
    const int rb = lsb - 1;
    const unsigned rbit = rb >= 64 ? static_cast<unsigned>((hi >> (rb - 64)) & 1ull)
                                   : static_cast<unsigned>((lo >> rb) & 1ull);
    bool sticky = sticky_in;
    if (rb > 0) {
      if (rb >= 64) {
        sticky |= (lo != 0ull) || ((hi & ((rb == 64) ? 0ull : ((1ull << (rb - 64)) - 1ull))) != 0ull);
      } else {
        sticky |= (lo & ((1ull << rb) - 1ull)) != 0ull;
      }
    }
    if (rbit && (sticky || (q & 1ull))) ++q;
  }
  return __double2float_rn(static_cast<double>(q) * pow2_double(lsb + k));
}

// Exact RN32(sum c^2 / 512) for any finite inputs, one thread: a 640-bit accumulator of 32-bit
// limbs (|c| = M * 2^(eb-150), c^2 = M^2 * 2^(2eb-300); LSB of the accumulator is 2^-298).
__device__ __noinline__ float mean_square_exact_slow(const float* c) {
  uint32_t acc[20];
#pragma unroll
  for (int j = 0; j < 20; ++j) acc[j] = 0u;
  for (int i = 0; i < kHead; ++i) {
    const uint32_t u = __float_as_uint(c[i]) & 0x7fffffffu;
    if (u == 0u) continue;
    const uint32_t ef = u >> 23;
    const uint32_t eb = ef ? ef : 1u;
    const unsigned long long M = ef ? ((u & 0x7fffffu) | 0x800000u) : (u & 0x7fffffu);
    const unsigned long long sq = M * M;  // < 2^48
    const int shift = 2 * static_cast<int>(eb) - 2;
    const int limb = shift >> 5, bit = shift & 31;
    // sq << bit spans at most 80 bits = 3 limbs
    uint32_t part[3];
    part[0] = static_cast<uint32_t>(sq << bit);
    part[1] = static_cast<uint32_t>((sq << bit) >> 32);
    part[2] = bit ? static_cast<uint32_t>(sq >> (64 - bit)) : 0u;
    unsigned long long carry = 0ull;
    for (int j = limb; j < 20; ++j) {
      const int k = j - limb;
      if (k >= 3 && carry == 0ull) break;
      const unsigned long long s = static_cast<unsigned long long>(acc[j]) + (k < 3 ? part[k] : 0u) + carry;
      acc[j] = static_cast<uint32_t>(s);
      carry = s >> 32;
    }
  }
  int top = -1;
  for (int j = 19; j >= 0; --j)
    if (acc[j]) {
      top = j;
      break;
    }
  if (top < 0) return 0.0f;
  // value = acc * 2^-298 / 512 = acc * 2^-307. Take a 128-bit window whose top limb is `top`.
  const int w0 = top >= 3 ? top - 3 : 0;  // limb index of the window's LSB
  unsigned long long lo = 0ull, hi = 0ull;
  lo = static_cast<unsigned long long>(acc[w0]) | (w0 + 1 <= top ? static_cast<unsigned long long>(acc[w0 + 1]) << 32 : 0ull);
  if (w0 + 2 <= top) hi = static_cast<unsigned long long>(acc[w0 + 2]);
  if (w0 + 3 <= top) hi |= static_cast<unsigned long long>(acc[w0 + 3]) << 32;
  bool sticky = false;
  for (int j = 0; j < w0; ++j) sticky |= acc[j] != 0u;
  return round_u128_to_f32(lo, hi, 32 * w0 - 307, sticky);
}

__device__ void scheduler_warp(const Params& p, Smem& S, int lane) {
  grid_dependency_wait();  // the list and the counters come from plan_kernel
  const int32_t* list = reinterpret_cast<const int32_t*>(p.ws + 1);
  const volatile int* abort_flag = &S.abort_flag;
  const uint32_t A = static_cast<uint32_t>(min(static_cast<int64_t>(*reinterpret_cast<volatile unsigned*>(&p.ws->count)), p.T));
  uint32_t widx = 0;
  for (;;) {
    if (*abort_flag) return;
    uint32_t a = 0;
    if (lane == 0) a = atomicAdd(&p.ws->next, 1u);
    a = __shfl_sync(0xffffffffu, a, 0);
    const bool end = a >= A;
    long long t = 0, pos = 0, kvs = 0;
    int req = 0;
    uint32_t err = 0;
    if (!end) {
      if (lane == 0) {
        t = list[a];
        req = __ldg(p.ttr + t);
        pos = __ldg(p.pos + t);
        kvs = __ldg(p.kvslot + t);
        if (req < 0 || req >= p.bt_rows) err |= C128_DEV_BAD_REQ;
        if (pos / kStateBlock >= p.bt_cols) err |= C128_DEV_BAD_BT_COL;
        if (pos - (kRatio - 1) >= p.cs_rows) err |= C128_DEV_BAD_COS_ROW;  // (p/128)*128 == p-127
        if (kvs >= p.nkb * p.kv_bs) err |= C128_DEV_BAD_KV_SLOT;
      }
      t = __shfl_sync(0xffffffffu, t, 0);
      req = __shfl_sync(0xffffffffu, req, 0);
      pos = __shfl_sync(0xffffffffu, pos, 0);
      kvs = __shfl_sync(0xffffffffu, kvs, 0);
      err = __shfl_sync(0xffffffffu, err, 0);
    }
    int blk = 0;
    if (!end && !(err & (C128_DEV_BAD_REQ | C128_DEV_BAD_BT_COL))) {
      if (lane < kWindowBlocks)
        blk = __ldg(p.bt + static_cast<int64_t>(req) * p.bt_stride + (pos - (kRatio - 1)) / kStateBlock + lane);
      const bool bad = lane < kWindowBlocks && (blk < 0 || blk >= p.nb);
      if (__any_sync(0xffffffffu, bad)) err |= C128_DEV_BAD_BLOCK;
    }
    if (!end && err) {
      if (lane == 0) atomicOr(&p.ws->err, err);
      continue;
    }
    const int ds = widx % kDescSlots;
    if (widx >= kDescSlots) {
      bool ok = mbar_wait(&S.dempty[ds], ((widx / kDescSlots) - 1u) & 1u, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) {
          S.abort_flag = 1;
          atomicOr(&p.ws->err, static_cast<unsigned>(C128_DEV_TIMEOUT));
        }
        return;
      }
    }
    WinDesc& d = S.desc[ds];
    if (!end) {
      if (lane < kWindowBlocks) d.src[lane] = p.state + static_cast<int64_t>(blk) * p.s0;
      if (lane == 0) {
        const long long kb = kvs / p.kv_bs, off = kvs % p.kv_bs;
        uint8_t* base = p.kc + kb * p.kc_stride0;
        d.kv_dst = base + off * kTokenStride;
        d.scale_dst = base + p.kv_bs * kTokenStride + off * kScaleDim;
        d.cs_row = p.cs + (pos - (kRatio - 1)) * p.cs_stride;
        d.comp_dst = p.comp_out ? p.comp_out + t * kHead : nullptr;
      }
    }
    if (lane == 0) d.kind = end ? 1 : 0;
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      mbar_arrive(&S.dfull[ds]);
    }
    ++widx;
    if (end) return;
  }
}

__device__ void copy_thread(const Params& p, Smem& S) {
  const volatile int* abort_flag = &S.abort_flag;
  const uint64_t policy = l2_evict_first_policy();
  const bool block_contiguous = p.s1 == kRow;
  uint32_t it = 0, widx = 0;
  bool failed = false;
  for (;;) {
    const int ds = widx % kDescSlots;
    if (!mbar_wait(&S.dfull[ds], (widx / kDescSlots) & 1u, abort_flag)) {
      failed = true;
      break;
    }
    const WinDesc& d = S.desc[ds];
    if (d.kind != 0) break;
    for (int j = 0; j < kWindowBlocks; ++j) {
      const int s = it % kStages;
      const uint32_t round = it / kStages;
      if (round > 0 && !mbar_wait(&S.empty[s], (round - 1u) & 1u, abort_flag)) {
        failed = true;
        break;
      }
      mbar_arrive_expect_tx(&S.full[s], kStageBytes);
      const float* src = d.src[j];
      if (block_contiguous) {
        bulk_copy_g2s(S.stage[s], src, kStageBytes, &S.full[s], policy);
      } else {
        for (int r = 0; r < kStateBlock; ++r)
          bulk_copy_g2s(S.stage[s] + r * kRow, src + r * p.s1, kRow * 4, &S.full[s], policy);
      }
      ++it;
    }
    if (failed) break;
    mbar_arrive(&S.dempty[ds]);
    ++widx;
  }
  if (failed) {
    S.abort_flag = 1;
    atomicOr(&p.ws->err, static_cast<unsigned>(C128_DEV_TIMEOUT));
    // let every copy this thread issued land before the CTA may exit
    for (uint32_t i = it > static_cast<uint32_t>(kStages) ? it - kStages : 0u; i < it; ++i)
      mbar_wait(&S.full[i % kStages], (i / kStages) & 1u, nullptr);
  }
}

// Online softmax state of a thread's two columns; the running max is kept in log2 units.
struct Online {
  float m0, m1, l0, l1, a0, a1;
};
__device__ __forceinline__ void online_init(Online& o) {
  o.m0 = o.m1 = -INFINITY;
  o.l0 = o.l1 = o.a0 = o.a1 = 0.f;
}
// Fold the 8 rows of one staged state block into the state of columns c0, c0 + 1.
__device__ __forceinline__ void online_stage(const float* st, int c0, Online& o) {
  float2 kv[kStateBlock], sc[kStateBlock];
#pragma unroll
  for (int r = 0; r < kStateBlock; ++r) {
    kv[r] = *reinterpret_cast<const float2*>(st + r * kRow + c0);
    sc[r] = *reinterpret_cast<const float2*>(st + r * kRow + kHead + c0);
  }
  float mx0 = sc[0].x, mx1 = sc[0].y;
#pragma unroll
  for (int r = 1; r < kStateBlock; ++r) {
    mx0 = fmaxf(mx0, sc[r].x);
    mx1 = fmaxf(mx1, sc[r].y);
  }
  const float n0 = fmaxf(o.m0, mx0 * kLog2e), n1 = fmaxf(o.m1, mx1 * kLog2e);
  // a column whose scores so far are all -inf keeps weight 0 instead of producing NaN
  const float b0 = n0 == -INFINITY ? 0.f : n0, b1 = n1 == -INFINITY ? 0.f : n1;
  const float r0 = ex2_approx(o.m0 - b0), r1 = ex2_approx(o.m1 - b1);
  o.m0 = n0;
  o.m1 = n1;
  float ps0 = 0.f, ps1 = 0.f, pk0 = 0.f, pk1 = 0.f;
#pragma unroll
  for (int r = 0; r < kStateBlock; ++r) {
    const float e0 = ex2_approx(fmaf(sc[r].x, kLog2e, -b0));
    const float e1 = ex2_approx(fmaf(sc[r].y, kLog2e, -b1));
    ps0 += e0;
    ps1 += e1;
    pk0 = fmaf(e0, kv[r].x, pk0);
    pk1 = fmaf(e1, kv[r].y, pk1);
  }
  o.l0 = fmaf(o.l0, r0, ps0);
  o.l1 = fmaf(o.l1, r1, ps1);
  o.a0 = fmaf(o.a0, r0, pk0);
  o.a1 = fmaf(o.a1, r1, pk1);
}

// Fused epilogue of one window, run by all 256 consumer threads (thread ci owns columns 2ci,
// 2ci+1; warp w owns quant block w, warp 7 the rope pairs). `failed` is this thread's view of the
// window's data; if any consumer failed, nothing is stored and false is returned (uniformly).
__device__ bool epilogue(EpiSmem& E, int ci, float cv0, float cv1, float2 w, float eps, float cosv, float sinv,
                         uint8_t* kv_dst, uint8_t* scale_dst, float* comp_dst, bool failed) {
  const int cw = ci >> 5, lane = ci & 31;
  const int c0 = 2 * ci;
  if (!failed && comp_dst != nullptr) *reinterpret_cast<float2*>(comp_dst + c0) = make_float2(cv0, cv1);
  *reinterpret_cast<float2*>(E.comp + c0) = make_float2(cv0, cv1);

  // variance = RN32(exact(sum c^2) / 512): align every square to the largest exponent and add them
  // as 128-bit integers (exact while all non-zero |c| are within 2^32 of the largest)
  const uint32_t u0 = __float_as_uint(cv0) & 0x7fffffffu, u1 = __float_as_uint(cv1) & 0x7fffffffu;
  const uint32_t f0 = u0 >> 23, f1 = u1 >> 23;
  uint32_t special = (f0 == 255u ? ((u0 & 0x7fffffu) ? 2u : 1u) : 0u) | (f1 == 255u ? ((u1 & 0x7fffffu) ? 2u : 1u) : 0u);
  const uint32_t eb0 = u0 ? (f0 ? f0 : 1u) : 0u, eb1 = u1 ? (f1 ? f1 : 1u) : 0u;
  const uint32_t emax_w = __reduce_max_sync(0xffffffffu, max(eb0, eb1));
  special = __reduce_or_sync(0xffffffffu, special);
  if (lane == 0) {
    E.red_emax[cw] = emax_w;
    E.red_special[cw] = special;
  }
  if (consumer_bar_or(failed)) return false;
  uint32_t emax = 0u;
  special = 0u;
#pragma unroll
  for (int k = 0; k < kConsumerWarps; ++k) {
    emax = max(emax, E.red_emax[k]);
    special |= E.red_special[k];
  }
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
    E.red_lo[cw] = lo;
    E.red_hi[cw] = hi;
    E.red_fallback[cw] = fb_w;
  }
  consumer_bar();
  if (ci == 0) {
    float var;
    bool fb = false;
    unsigned long long vlo = 0ull, vhi = 0ull;
#pragma unroll
    for (int k = 0; k < kConsumerWarps; ++k) {
      fb |= E.red_fallback[k] != 0u;
      const unsigned long long nlo = vlo + E.red_lo[k];
      vhi += E.red_hi[k] + (nlo < vlo ? 1ull : 0ull);
      vlo = nlo;
    }
    if (special & 2u) {
      var = __int_as_float(0x7fc00000);
    } else if (special & 1u) {
      var = INFINITY;
    } else if (fb) {
      var = mean_square_exact_slow(E.comp);
    } else {
      var = round_u128_to_f32(vlo, vhi, 2 * static_cast<int>(emax) - 373, false);
    }
    // rrms: the correctly rounded fp32 reciprocal square root of RN32(var + eps)
    E.rrms = __frsqrt_rn(__fadd_rn(var, eps));
  }
  consumer_bar();
  const float rrms = E.rrms;
  const float n0 = __fmul_rn(__fmul_rn(cv0, rrms), w.x);
  const float n1 = __fmul_rn(__fmul_rn(cv1, rrms), w.y);

  if (cw < kConsumerWarps - 1) {
    // nope block cw: bf16 round, absmax, UE8M0 exponent, e4m3 codes
    const uint32_t b = pack_bf16x2(n0, n1);
    const float x0 = __uint_as_float(b << 16), x1 = __uint_as_float(b & 0xffff0000u);
    const uint32_t amax_bits =
        __reduce_max_sync(0xffffffffu, max(__float_as_uint(x0) & 0x7fffffffu, __float_as_uint(x1) & 0x7fffffffu));
    const float amax = fmaxf(__uint_as_float(amax_bits), __uint_as_float(kAbsmaxFloorBits));
    const uint32_t raw = __float_as_uint(__fmul_rn(amax, __uint_as_float(kInv448Bits)));
    const int e = static_cast<int>(raw >> 23) - 127 + ((raw & 0x7fffffu) ? 1 : 0);  // ceil(log2(raw))
    const float inv_scale = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    const float y0 = fminf(fmaxf(__fmul_rn(x0, inv_scale), -448.f), 448.f);
    const float y1 = fminf(fmaxf(__fmul_rn(x1, inv_scale), -448.f), 448.f);
    *reinterpret_cast<uint16_t*>(kv_dst + cw * kQuantBlock + 2 * lane) = pack_e4m3x2(y0, y1);
    if (lane == 0) scale_dst[cw] = static_cast<uint8_t>(min(max(e + 127, 0), 255));
  } else {
    // rope pair j = lane: (448 + 2j, 449 + 2j)
    const float ne = __fsub_rn(__fmul_rn(n0, cosv), __fmul_rn(n1, sinv));
    const float no = __fadd_rn(__fmul_rn(n1, cosv), __fmul_rn(n0, sinv));
    *reinterpret_cast<uint32_t*>(kv_dst + kNope + 4 * lane) = pack_bf16x2(ne, no);
    if (lane == 0) scale_dst[kNope / kQuantBlock] = 0;
  }
  return true;
}

__device__ void consumer_warps(const Params& p, Smem& S, int ci) {
  const int cw = ci >> 5, lane = ci & 31;
  const int c0 = 2 * ci;  // this thread's columns: c0, c0 + 1
  const volatile int* abort_flag = &S.abort_flag;
  const float2 w = *reinterpret_cast<const float2*>(p.rms_w + c0);
  uint32_t it = 0, widx = 0;
  for (;;) {
    const int ds = widx % kDescSlots;
    const bool got = mbar_wait(&S.dfull[ds], (widx / kDescSlots) & 1u, abort_flag);
    int kind = 1;
    uint8_t* kv_dst = nullptr;
    uint8_t* scale_dst = nullptr;
    const float* cs_row = nullptr;
    float* comp_dst = nullptr;
    if (got) {
      const WinDesc& d = S.desc[ds];
      kind = d.kind;
      kv_dst = d.kv_dst;
      scale_dst = d.scale_dst;
      cs_row = d.cs_row;
      comp_dst = d.comp_dst;
    } else {
      S.abort_flag = 1;
      atomicOr(&p.ws->err, static_cast<unsigned>(C128_DEV_TIMEOUT));
    }
    if (consumer_bar_or(!got || kind != 0 || *abort_flag)) return;

    float cosv = 0.f, sinv = 0.f;
    if (cw == kConsumerWarps - 1) {  // the rope warp: pair j = lane
      cosv = __ldg(cs_row + lane);
      sinv = __ldg(cs_row + kRope / 2 + lane);
    }
    Online o;
    online_init(o);
    bool failed = false;
    for (int j = 0; j < kWindowBlocks; ++j) {
      const int s = it % kStages;
      bool ok = !failed && mbar_wait(&S.full[s], (it / kStages) & 1u, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        online_stage(S.stage[s], c0, o);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[s]);
      } else {
        failed = true;
      }
      ++it;
    }
    if (failed) {
      S.abort_flag = 1;
      atomicOr(&p.ws->err, static_cast<unsigned>(C128_DEV_TIMEOUT));
    }
    const float cv0 = __fdiv_rn(o.a0, o.l0), cv1 = __fdiv_rn(o.a1, o.l1);
    if (!epilogue(S.epi, ci, cv0, cv1, w, p.eps, cosv, sinv, kv_dst, scale_dst, comp_dst, failed)) return;
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.dempty[ds]);
    ++widx;
  }
}

__global__ void __launch_bounds__(kThreads, 1) compress_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);
    }
    for (int d = 0; d < kDescSlots; ++d) {
      mbar_init(&S.dfull[d], 1);
      mbar_init(&S.dempty[d], kConsumerWarps + 1);
    }
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == 0) {
    scheduler_warp(p, S, lane);
  } else if (warp == 1) {
    if (lane == 0) copy_thread(p, S);
  } else {
    consumer_warps(p, S, tid - 64);
  }
}

// --------------------------------------------------------------------------- direct kernel
// Few tokens (T x S <= #SM): no planning pass. Cluster c (S CTAs) takes token c; CTA rank r
// streams blocks [r*16/S, (r+1)*16/S) of the window through its own ring, its consumers fold
// them into partial softmax states, rank 0 merges the S partials from distributed shared memory
// (in rank order) and runs the same epilogue. Every CTA of a cluster reads the same token and all
// 16 block ids, so every early exit is uniform across the cluster.
template <int S>
struct DirectCfg {
  static constexpr int kBlocks = kWindowBlocks / S;                 // stages per CTA
  static constexpr int kRing = kBlocks < kStages ? kBlocks : kStages;
};

template <int S>
struct DirectSmem {
  float stage[DirectCfg<S>::kRing][kStateBlock * kRow];
  uint64_t full[DirectCfg<S>::kRing];
  uint64_t empty[DirectCfg<S>::kRing];
  float2 part_m[kHead / 2];   // partial softmax state of this CTA's rows, per column pair
  float2 part_l[kHead / 2];
  float2 part_a[kHead / 2];
  int part_failed;
  EpiSmem epi;
  int abort_flag;
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// address of `p` (this CTA's shared memory) in the shared memory of cluster CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

template <int S>
__global__ void __launch_bounds__(kThreads, 1) direct_kernel(Params p) {
  using Cfg = DirectCfg<S>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  DirectSmem<S>& D = *reinterpret_cast<DirectSmem<S>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
  const int64_t t = static_cast<int64_t>(blockIdx.x) / S;
  if (tid == 0) {
    for (int s = 0; s < Cfg::kRing; ++s) {
      mbar_init(&D.full[s], 1);
      mbar_init(&D.empty[s], kConsumerWarps);
    }
    D.abort_flag = 0;
    D.part_failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const volatile int* abort_flag = &D.abort_flag;

  // the token and its window (every thread; broadcast loads)
  const int64_t slot = __ldg(p.slot + t), pos = __ldg(p.pos + t), kvs = __ldg(p.kvslot + t);
  if (!((slot >= 0) & (pos >= 0) & ((pos & (kRatio - 1)) == kRatio - 1) & (kvs >= 0))) return;
  const int req = __ldg(p.ttr + t);
  uint32_t err = 0;
  if (req < 0 || req >= p.bt_rows) err |= C128_DEV_BAD_REQ;
  if (pos / kStateBlock >= p.bt_cols) err |= C128_DEV_BAD_BT_COL;
  if (pos - (kRatio - 1) >= p.cs_rows) err |= C128_DEV_BAD_COS_ROW;
  if (kvs >= p.nkb * p.kv_bs) err |= C128_DEV_BAD_KV_SLOT;
  int blk = 0;  // lane j of every warp holds block id j of the window
  if (!(err & (C128_DEV_BAD_REQ | C128_DEV_BAD_BT_COL))) {
    if (lane < kWindowBlocks)
      blk = __ldg(p.bt + static_cast<int64_t>(req) * p.bt_stride + (pos - (kRatio - 1)) / kStateBlock + lane);
    if (__any_sync(0xffffffffu, lane < kWindowBlocks && (blk < 0 || blk >= p.nb))) err |= C128_DEV_BAD_BLOCK;
  }
  if (err) {
    if (rank == 0 && tid == 0) atomicOr(&p.ws->err, err);
    return;
  }

  const int ci = tid - 64;
  const int c0 = 2 * (ci < 0 ? 0 : ci);
  Online o;
  online_init(o);
  bool failed = false;
  if (warp == 0) {
    // copy thread: this CTA's blocks through the ring
    uint32_t issued = 0;
    const uint64_t policy = l2_evict_first_policy();
    for (int j = 0; j < Cfg::kBlocks; ++j) {
      const int b = __shfl_sync(0xffffffffu, blk, static_cast<int>(rank) * Cfg::kBlocks + j);
      if (lane == 0 && !failed) {
        const int s = j % Cfg::kRing;
        const uint32_t round = j / Cfg::kRing;
        if (round > 0 && !mbar_wait(&D.empty[s], (round - 1u) & 1u, abort_flag)) {
          failed = true;
        } else {
          mbar_arrive_expect_tx(&D.full[s], kStageBytes);
          const float* src = p.state + static_cast<int64_t>(b) * p.s0;
          if (p.s1 == kRow) {
            bulk_copy_g2s(D.stage[s], src, kStageBytes, &D.full[s], policy);
          } else {
            for (int r = 0; r < kStateBlock; ++r)
              bulk_copy_g2s(D.stage[s] + r * kRow, src + r * p.s1, kRow * 4, &D.full[s], policy);
          }
          ++issued;
        }
      }
    }
    if (lane == 0 && failed) {
      D.abort_flag = 1;
      atomicOr(&p.ws->err, static_cast<unsigned>(C128_DEV_TIMEOUT));
      for (uint32_t i = issued > static_cast<uint32_t>(Cfg::kRing) ? issued - Cfg::kRing : 0u; i < issued; ++i)
        mbar_wait(&D.full[i % Cfg::kRing], (i / Cfg::kRing) & 1u, nullptr);
    }
  } else if (ci >= 0) {
    for (int j = 0; j < Cfg::kBlocks; ++j) {
      const int s = j % Cfg::kRing;
      bool ok = !failed && mbar_wait(&D.full[s], (j / Cfg::kRing) & 1u, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        online_stage(D.stage[s], c0, o);
        __syncwarp();
        if (lane == 0) mbar_arrive(&D.empty[s]);
      } else {
        failed = true;
      }
    }
    if (failed) {
      D.abort_flag = 1;
      atomicOr(&p.ws->err, static_cast<unsigned>(C128_DEV_TIMEOUT));
    }
  }

  if constexpr (S > 1) {
    // publish this CTA's partial state, then rank 0 merges all partials in rank order
    if (ci >= 0) {
      D.part_m[ci] = make_float2(o.m0, o.m1);
      D.part_l[ci] = make_float2(o.l0, o.l1);
      D.part_a[ci] = make_float2(o.a0, o.a1);
      if (failed) D.part_failed = 1;
    }
    cluster_sync_all();
    if (rank == 0 && ci >= 0) {
      float2 m[S], l[S], a[S];
      m[0] = make_float2(o.m0, o.m1);
      l[0] = make_float2(o.l0, o.l1);
      a[0] = make_float2(o.a0, o.a1);
#pragma unroll
      for (int r = 1; r < S; ++r) {
        m[r] = ld_cluster_f2(map_to_rank(&D.part_m[ci], r));
        l[r] = ld_cluster_f2(map_to_rank(&D.part_l[ci], r));
        a[r] = ld_cluster_f2(map_to_rank(&D.part_a[ci], r));
        failed |= ld_cluster_s32(map_to_rank(&D.part_failed, r)) != 0;
      }
      float M0 = m[0].x, M1 = m[0].y;
#pragma unroll
      for (int r = 1; r < S; ++r) {
        M0 = fmaxf(M0, m[r].x);
        M1 = fmaxf(M1, m[r].y);
      }
      const float B0 = M0 == -INFINITY ? 0.f : M0, B1 = M1 == -INFINITY ? 0.f : M1;
      float L0 = 0.f, L1 = 0.f, A0 = 0.f, A1 = 0.f;
#pragma unroll
      for (int r = 0; r < S; ++r) {
        const float s0 = ex2_approx(m[r].x - B0), s1 = ex2_approx(m[r].y - B1);
        L0 = fmaf(l[r].x, s0, L0);
        L1 = fmaf(l[r].y, s1, L1);
        A0 = fmaf(a[r].x, s0, A0);
        A1 = fmaf(a[r].y, s1, A1);
      }
      o.l0 = L0;
      o.l1 = L1;
      o.a0 = A0;
      o.a1 = A1;
    }
    cluster_sync_all();  // the partials stay readable until rank 0 has them
  }
  if (rank != 0 || ci < 0) return;

  const int cw = ci >> 5;
  float cosv = 0.f, sinv = 0.f;
  const float* cs_row = p.cs + (pos - (kRatio - 1)) * p.cs_stride;
  if (cw == kConsumerWarps - 1) {
    cosv = __ldg(cs_row + lane);
    sinv = __ldg(cs_row + kRope / 2 + lane);
  }
  const float2 w = *reinterpret_cast<const float2*>(p.rms_w + c0);
  const long long kb = kvs / p.kv_bs, off = kvs % p.kv_bs;
  uint8_t* base = p.kc + kb * p.kc_stride0;
  const float cv0 = __fdiv_rn(o.a0, o.l0), cv1 = __fdiv_rn(o.a1, o.l1);
  epilogue(D.epi, ci, cv0, cv1, w, p.eps, cosv, sinv, base + off * kTokenStride,
           base + p.kv_bs * kTokenStride + off * kScaleDim, p.comp_out ? p.comp_out + t * kHead : nullptr, failed);
}

// Split factor for few tokens: the largest S in {8, 4, 2, 1} with T * S CTAs fitting one wave;
// 0 selects the planned, persistent path.
int direct_split(int64_t T, int sm_count) {
  if (T > sm_count) return 0;
  for (int s = 8; s > 1; s >>= 1)
    if (T * s <= sm_count) return s;
  return 1;
}

template <int S>
cudaError_t launch_direct(const Params& p, const LaunchCfg& cfg, cudaStream_t stream) {
  if (cfg.ev_begin != nullptr) {
    const cudaError_t e = cudaEventRecord(cfg.ev_begin, stream);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(p.T * S));
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = sizeof(DirectSmem<S>);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = S > 1 ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&lc, direct_kernel<S>, p);
  if (e != cudaSuccess) return e;
  if (cfg.ev_end != nullptr) e = cudaEventRecord(cfg.ev_end, stream);
  return e;
}

}  // namespace

int compress_smem_bytes() { return static_cast<int>(sizeof(Smem)); }

cudaError_t prepare_device(int /*device*/) {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(compress_kernel, a, static_cast<int>(sizeof(Smem)));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(direct_kernel<1>, a, static_cast<int>(sizeof(DirectSmem<1>)));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(direct_kernel<2>, a, static_cast<int>(sizeof(DirectSmem<2>)));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(direct_kernel<4>, a, static_cast<int>(sizeof(DirectSmem<4>)));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(direct_kernel<8>, a, static_cast<int>(sizeof(DirectSmem<8>)));
  return e;
}

cudaError_t launch(const Params& p, const LaunchCfg& cfg, cudaStream_t stream) {
  switch (direct_split(p.T, cfg.sm_count)) {
    case 8: return launch_direct<8>(p, cfg, stream);
    case 4: return launch_direct<4>(p, cfg, stream);
    case 2: return launch_direct<2>(p, cfg, stream);
    case 1: return launch_direct<1>(p, cfg, stream);
    default: break;
  }
  cudaError_t e = cudaMemsetAsync(p.ws, 0, 2 * sizeof(unsigned int), stream);  // count, next
  if (e != cudaSuccess) return e;
  const int plan_grid = static_cast<int>((p.T + kPlanTokensPerCta - 1) / kPlanTokensPerCta);
  plan_kernel<<<plan_grid, kPlanThreads, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (cfg.ev_begin != nullptr && (e = cudaEventRecord(cfg.ev_begin, stream)) != cudaSuccess) return e;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(cfg.grid));
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = sizeof(Smem);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = (cfg.pdl && cfg.ev_begin == nullptr) ? 1 : 0;
  e = cudaLaunchKernelEx(&lc, compress_kernel, p);
  if (e != cudaSuccess) return e;
  if (cfg.ev_end != nullptr) e = cudaEventRecord(cfg.ev_end, stream);
  return e;
}

}  // namespace c128
