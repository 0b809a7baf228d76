// Device code shared by the kernels of libc128compress: PTX wrappers (mbarrier, TMA bulk copy,
// conversions, named barriers, programmatic dependent launch), the exact variance, the online
// softmax step over one staged state block, and the fused epilogue of a 512-wide window.
// Included by each kernel translation unit (everything here has internal linkage).
#pragma once
#include <math.h>

#include "c128_internal.h"
#include "c128compress.h"

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
// The same wait, but each retry lets the hardware suspend the thread until the phase completes
// (at most kSuspendHintNs per try), so waiting warps take no issue slots from the warps that work.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, P;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
__device__ __noinline__ bool mbar_wait_suspend(uint64_t* bar, uint32_t parity, const volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity)) return true;
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

// ------------------------------------------------------------------ the planning pass's list
// Read by one warp after the kernel waited for the planning pass: the number of active windows,
// and with per-chunk lists the exclusive prefix of the chunk counts in prefix[0 .. nchunks]
// (shared memory, kMaxPlanChunks + 1 words). Only this warp may use `prefix` afterwards.
__device__ __noinline__ uint32_t plan_prefix_warp(const Params& p, uint32_t* prefix, int lane) {
  const int32_t* list = reinterpret_cast<const int32_t*>(p.ws + 1);
  if (!p.chunked)
    return static_cast<uint32_t>(min(static_cast<int64_t>(*reinterpret_cast<const volatile unsigned*>(&p.ws->count)), p.T));
  const int nchunks = static_cast<int>((p.T + kPlanTokensPerCta - 1) / kPlanTokensPerCta);
  // All counts are loaded before the first is used: one global round trip instead of one per
  // 32 chunks (a round trip from a busy SM costs microseconds, and this sits in front of the
  // kernel's first copy).
  constexpr int kPerLane = kMaxPlanChunks / 32;
  uint32_t n[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int c = 32 * i + lane;
    n[i] = c < nchunks ? static_cast<uint32_t>(list[p.T + c]) : 0u;
  }
  uint32_t A = 0;
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    if (32 * i >= nchunks) break;
    uint32_t incl = n[i];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (32 * i + lane < nchunks) prefix[32 * i + lane] = A + incl - n[i];
    A += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) prefix[nchunks] = A;
  __syncwarp();
  return A;
}
// The token of claim a (a below the number of active windows).
__device__ __forceinline__ int64_t plan_token(const Params& p, const uint32_t* prefix, uint32_t a) {
  const int32_t* list = reinterpret_cast<const int32_t*>(p.ws + 1);
  if (!p.chunked) return list[a];
  int lo = 0, hi = static_cast<int>((p.T + kPlanTokensPerCta - 1) / kPlanTokensPerCta) - 1;
  while (lo < hi) {  // the last chunk whose prefix is <= a
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= a) lo = mid; else hi = mid - 1;
  }
  return list[static_cast<int64_t>(lo) * kPlanTokensPerCta + (a - prefix[lo])];
}

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

// Exact RN32(sum c^2 / n) for any finite inputs, n = 2^log2n <= 512, one thread: a 640-bit
// accumulator of 32-bit limbs (|c| = M * 2^(eb-150), c^2 = M^2 * 2^(2eb-300); its LSB is 2^-298).
__device__ __noinline__ float mean_square_exact_slow(const float* c, int n, int log2n) {
  uint32_t acc[20];
#pragma unroll
  for (int j = 0; j < 20; ++j) acc[j] = 0u;
  for (int i = 0; i < n; ++i) {
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
  // value = acc * 2^-298 / 2^log2n. Take a 128-bit window whose top limb is `top`.
  const int w0 = top >= 3 ? top - 3 : 0;  // limb index of the window's LSB
  unsigned long long lo = 0ull, hi = 0ull;
  lo = static_cast<unsigned long long>(acc[w0]) | (w0 + 1 <= top ? static_cast<unsigned long long>(acc[w0 + 1]) << 32 : 0ull);
  if (w0 + 2 <= top) hi = static_cast<unsigned long long>(acc[w0 + 2]);
  if (w0 + 3 <= top) hi |= static_cast<unsigned long long>(acc[w0 + 3]) << 32;
  bool sticky = false;
  for (int j = 0; j < w0; ++j) sticky |= acc[j] != 0u;
  return round_u128_to_f32(lo, hi, 32 * w0 - 298 - log2n, sticky);
}

// Online softmax state of a thread's two columns; the running max is kept in log2 units.
struct Online {
  float m0, m1, l0, l1, a0, a1;
};
__device__ __forceinline__ void online_init(Online& o) {
  o.m0 = o.m1 = -INFINITY;
  o.l0 = o.l1 = o.a0 = o.a1 = 0.f;
}
// The 8 rows of one staged state block for columns c0, c0 + 1: kv and score pairs.
struct BlockRows {
  float2 kv[kStateBlock], sc[kStateBlock];
};
__device__ __forceinline__ void stage_rows(const float* st, int c0, BlockRows& br) {
#pragma unroll
  for (int r = 0; r < kStateBlock; ++r) {
    br.kv[r] = *reinterpret_cast<const float2*>(st + r * kRow + c0);
    br.sc[r] = *reinterpret_cast<const float2*>(st + r * kRow + kHead + c0);
  }
}
// Fold those rows into the state of columns c0, c0 + 1.
__device__ __forceinline__ void online_fold(const BlockRows& br, Online& o) {
  const float2* kv = br.kv;
  const float2* sc = br.sc;
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
      var = mean_square_exact_slow(E.comp, kHead, 9);
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

}  // namespace
}  // namespace c128
