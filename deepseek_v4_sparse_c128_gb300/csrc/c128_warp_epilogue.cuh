// Per-warp epilogue of a head-128 indexer window (lane l owns columns 4l..4l+3): the exact
// variance, RMSNorm, the RoPE of every pair (the 32 nope pairs with cos 1, sin 0, the 32 rope
// pairs with the window's cos/sin) and the FP8 or MXFP4 cache store, as the fused indexer kernels
// on the API page of vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache compute them.
// Shared by the kernel translation units that serve head 128 (internal linkage).
#pragma once
#include "c128_device.cuh"

namespace c128 {
namespace {

constexpr uint32_t kInv6BitsW = 0x3e2aaaabu;  // RN32(1/6)

__device__ __forceinline__ uint32_t pack_e2m1x2_w(float lo, float hi) {
  uint16_t d;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tmov.b16 %0, {t, t};\n}" : "=h"(d) : "f"(hi), "f"(lo));
  return d & 0xffu;
}
__device__ __forceinline__ float pow2_neg_w(int e) {  // 2^-e for e in [-127, 127]
  return e <= 126 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23) : __uint_as_float(0x00200000u);
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

// `c`: this lane's 4 compressed values; `cosv`/`sinv`: cos/sin of its pairs 2l, 2l + 1 (1 and 0
// for the nope pairs, lanes 0..15); `comp_s`: 128 floats of scratch for the exact-variance slow path.
template <int FMT>
__device__ __forceinline__ void indexer_warp_epilogue(float4 c, int lane, float2 wa, float2 wb, float eps, float2 cosv,
                                                      float2 sinv, uint8_t* tok, uint8_t* scale, float* comp_dst,
                                                      float* comp_s) {
  const int col = 4 * lane;
  if (comp_dst != nullptr) *reinterpret_cast<float4*>(comp_dst + col) = c;
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
    for (int j = 0; j < 4; ++j) add_square(u[j], emax, lo, hi, fb);
  warp_sum128(lo, hi);
  fb = __any_sync(0xffffffffu, fb);
  float rrms = 0.f;
  if (fb) {
    *reinterpret_cast<float4*>(comp_s + col) = c;
    __syncwarp();
  }
  if (lane == 0) {
    float var;
    if (special & 2u) var = __int_as_float(0x7fc00000);
    else if (special & 1u) var = INFINITY;
    else if (fb) var = mean_square_exact_slow(comp_s, 128, 7);
    else var = round_u128_to_f32(lo, hi, 2 * static_cast<int>(emax) - 371, false);
    rrms = __frsqrt_rn(__fadd_rn(var, eps));
  }
  __syncwarp();
  rrms = __shfl_sync(0xffffffffu, rrms, 0);
  const float nv[4] = {__fmul_rn(__fmul_rn(c.x, rrms), wa.x), __fmul_rn(__fmul_rn(c.y, rrms), wa.y),
                       __fmul_rn(__fmul_rn(c.z, rrms), wb.x), __fmul_rn(__fmul_rn(c.w, rrms), wb.y)};
  // RoPE of pairs j = 2*lane + k; pairs >= 32 (lanes 16..31) rotate, the others use cos 1, sin 0
  float x[4];
#pragma unroll
  for (int j2 = 0; j2 < 2; ++j2) {
    const float C = j2 ? cosv.y : cosv.x, Sn = j2 ? sinv.y : sinv.x;
    const float ev = nv[2 * j2], od = nv[2 * j2 + 1];
    const uint32_t b = pack_bf16x2(__fsub_rn(__fmul_rn(ev, C), __fmul_rn(od, Sn)),
                                   __fadd_rn(__fmul_rn(od, C), __fmul_rn(ev, Sn)));
    x[2 * j2] = __uint_as_float(b << 16);
    x[2 * j2 + 1] = __uint_as_float(b & 0xffff0000u);
  }
  const uint32_t am_l = max(max(__float_as_uint(x[0]) & 0x7fffffffu, __float_as_uint(x[1]) & 0x7fffffffu),
                            max(__float_as_uint(x[2]) & 0x7fffffffu, __float_as_uint(x[3]) & 0x7fffffffu));
  if constexpr (FMT == C128_FORMAT_INDEXER_FP8) {
    const float amax = fmaxf(__uint_as_float(__reduce_max_sync(0xffffffffu, am_l)), __uint_as_float(kAbsmaxFloorBits));
    const uint32_t raw = __float_as_uint(__fmul_rn(amax, __uint_as_float(kInv448Bits)));
    const int e = static_cast<int>(raw >> 23) - 127 + ((raw & 0x7fffffu) ? 1 : 0);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    float y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) y[j] = fminf(fmaxf(__fmul_rn(x[j], inv), -448.f), 448.f);
    *reinterpret_cast<uint32_t*>(tok + col) =
        static_cast<uint32_t>(pack_e4m3x2(y[0], y[1])) | (static_cast<uint32_t>(pack_e4m3x2(y[2], y[3])) << 16);
    if (lane == 0) *reinterpret_cast<float*>(scale) = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
  } else {
    // MXFP4 block b = values 32b..32b+31 = lanes 8b..8b+7
    uint32_t am = am_l;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, o));
    const float amax = fmaxf(__uint_as_float(am), 6.0f * __uint_as_float(0x00800000u));
    const uint32_t ratio = __float_as_uint(__fmul_rn(amax, __uint_as_float(kInv6BitsW)));
    const int e = min(max(static_cast<int>(ratio >> 23) - 127 + ((ratio & 0x7fffffu) ? 1 : 0), -127), 127);
    const float inv = pow2_neg_w(e);
    const uint32_t b0 = pack_e2m1x2_w(__fmul_rn(x[0], inv), __fmul_rn(x[1], inv));
    const uint32_t b1 = pack_e2m1x2_w(__fmul_rn(x[2], inv), __fmul_rn(x[3], inv));
    *reinterpret_cast<uint16_t*>(tok + 2 * lane) = static_cast<uint16_t>(b0 | (b1 << 8));
    if ((lane & 7) == 0) scale[lane >> 3] = static_cast<uint8_t>(e + 127);
  }
}

}  // namespace
}  // namespace c128
