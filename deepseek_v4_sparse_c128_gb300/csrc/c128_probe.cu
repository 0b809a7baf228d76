// c128_read_probe: a plain streaming read of one device buffer, the read-only bandwidth denominator
// beside the measured copy bandwidth. The compressor reads about 900 bytes for every byte it writes,
// so a copy (half reads, half writes) is not the rate its reads can reach; this kernel measures that
// rate on the same GPU, in the same process, right beside the compressor's own timing.
//
// Each thread keeps LOADS 16-byte loads in flight (ld.global.nc, no L1 allocation, L2 evict-first,
// the compressor's cache policy for state) over a grid-stride walk and folds the words it reads
// into an XOR; each warp XORs its result into one device word. The XOR makes every load
// observable, so nothing is skipped, and it lets a test check that every byte was read: the word
// equals the XOR of the buffer's 32-bit words.
#include <cuda_runtime.h>

#include <cstdint>

#include "c128compress.h"

namespace {

__device__ __forceinline__ uint4 ld_stream16(const uint4* p, uint64_t pol) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "l"(pol));
  return v;
}

template <int LOADS>
__global__ void __launch_bounds__(1024) read_probe_kernel(const uint4* __restrict__ src, int64_t n16,
                                                          uint32_t* __restrict__ xor_out) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + (LOADS - 1) * stride < n16; i += LOADS * stride) {
    uint4 v[LOADS];
#pragma unroll
    for (int u = 0; u < LOADS; ++u) v[u] = ld_stream16(src + i + u * stride, pol);
#pragma unroll
    for (int u = 0; u < LOADS; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ld_stream16(src + i, pol);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  acc = __reduce_xor_sync(0xffffffffu, acc);
  if ((threadIdx.x & 31) == 0 && acc != 0u) atomicXor(xor_out, acc);
}

template <int LOADS>
cudaError_t launch(const void* buf, int64_t n16, uint32_t* xor_out, int grid, int threads, cudaStream_t s) {
  read_probe_kernel<LOADS><<<grid, threads, 0, s>>>(static_cast<const uint4*>(buf), n16, xor_out);
  return cudaGetLastError();
}

}  // namespace

extern "C" int c128_read_probe(const void* buf, int64_t bytes, int32_t threads_per_cta, int32_t ctas_per_sm,
                               int32_t loads_in_flight, uint32_t* xor_out, c128_stream_t stream) {
  if (bytes < 0 || bytes % 16 != 0) return C128_ERR_ARG;
  if (threads_per_cta < 32 || threads_per_cta > 1024 || threads_per_cta % 32 != 0) return C128_ERR_ARG;
  if (ctas_per_sm < 1 || ctas_per_sm > 32 || static_cast<int64_t>(threads_per_cta) * ctas_per_sm > 2048)
    return C128_ERR_ARG;
  if (loads_in_flight != 1 && loads_in_flight != 2 && loads_in_flight != 4 && loads_in_flight != 8)
    return C128_ERR_ARG;
  if (bytes == 0) return C128_OK;
  if (buf == nullptr || xor_out == nullptr) return C128_ERR_NULL_PTR;
  if (reinterpret_cast<uintptr_t>(buf) % 16 != 0 || reinterpret_cast<uintptr_t>(xor_out) % 4 != 0)
    return C128_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return C128_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return C128_ERR_CUDA;
  // every CTA of the grid-stride walk must be resident at once, or the last ones read alone
  int resident = 0;
  cudaError_t e;
  switch (loads_in_flight) {
    case 1: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, read_probe_kernel<1>, threads_per_cta, 0); break;
    case 2: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, read_probe_kernel<2>, threads_per_cta, 0); break;
    case 4: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, read_probe_kernel<4>, threads_per_cta, 0); break;
    default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, read_probe_kernel<8>, threads_per_cta, 0); break;
  }
  if (e != cudaSuccess || resident < 1) return C128_ERR_CUDA;
  const int64_t n16 = bytes / 16;
  const int64_t want = static_cast<int64_t>(sms) * (ctas_per_sm < resident ? ctas_per_sm : resident);
  const int64_t needed = (n16 + threads_per_cta - 1) / threads_per_cta;  // CTAs with one load per thread
  const int grid = static_cast<int>(want < needed ? want : needed);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (loads_in_flight) {
    case 1: e = launch<1>(buf, n16, xor_out, grid, threads_per_cta, s); break;
    case 2: e = launch<2>(buf, n16, xor_out, grid, threads_per_cta, s); break;
    case 4: e = launch<4>(buf, n16, xor_out, grid, threads_per_cta, s); break;
    default: e = launch<8>(buf, n16, xor_out, grid, threads_per_cta, s); break;
  }
  return e == cudaSuccess ? C128_OK : C128_ERR_CUDA;
}
