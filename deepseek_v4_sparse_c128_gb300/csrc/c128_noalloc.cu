// c128_compress_norm_rope_store_noalloc: compress_norm_rope_store for callers that cannot
// allocate device memory. Its scratch (workspace header + active-token list) is the static device
// array below instead of a cudaMalloc'ed per-stream workspace; the kernels are the same.
#include <cuda_runtime.h>

#include <mutex>

#include "c128_internal.h"
#include "c128compress.h"

namespace {

constexpr int64_t kMaxTokens = C128_NOALLOC_MAX_TOKENS;
// header, then the token list and the per-chunk counts of the C128 planning pass
constexpr size_t kScratchBytes =
    sizeof(c128::WsHeader) + static_cast<size_t>(c128::plan_list_entries(kMaxTokens)) * sizeof(int32_t);

// Lives in every GPU that loads the library. In host code this name is only a stand-in for the
// symbol: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct DeviceSetup {
  bool ready = false;
  c128::WsHeader* ws = nullptr;
  int sm_count = 0;
};
std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];  // fixed table: the call path allocates nothing, host or device

// Once per device, with that device current: the scratch array's device address, the SM count
// and the compress kernel's shared-memory attribute.
int setup_device(int dev, DeviceSetup** out) {
  if (dev < 0 || dev >= kMaxDevices) return C128_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  DeviceSetup& d = g_setup[dev];
  if (!d.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess) return C128_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return C128_ERR_CUDA;
    if (c128::prepare_device(dev) != cudaSuccess) return C128_ERR_CUDA;
    d.ws = static_cast<c128::WsHeader*>(ptr);
    d.ready = true;
  }
  *out = &d;
  return C128_OK;
}

}  // namespace

extern "C" int c128_compress_norm_rope_store_noalloc(
    const c128_tensor_t* token_to_req_indices, const c128_tensor_t* positions, const c128_tensor_t* slot_mapping,
    const c128_tensor_t* block_table, const c128_tensor_t* state_cache, const c128_tensor_t* rms_w, float eps,
    const c128_tensor_t* cos_sin_cache, const c128_tensor_t* k_cache, const c128_tensor_t* kv_slot_mapping,
    int64_t kv_block_size, c128_stream_t stream) {
  c128::Params p{};
  const int rc = c128::validate_args(token_to_req_indices, positions, slot_mapping, block_table, state_cache,
                                     rms_w, eps, cos_sin_cache, k_cache, kv_slot_mapping, kv_block_size, nullptr,
                                     &p);
  if (rc != C128_OK) return rc;
  if (p.T > kMaxTokens) return C128_ERR_TOO_MANY_TOKENS;
  if (p.T == 0) return C128_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return C128_ERR_CUDA;
  DeviceSetup* d = nullptr;
  const int src = setup_device(dev, &d);
  if (src != C128_OK) return src;
  p.ws = d->ws;
  c128::LaunchCfg cfg{};
  cfg.sm_count = d->sm_count;
  cfg.grid = static_cast<int>(p.T < d->sm_count ? p.T : d->sm_count);
  cfg.pdl = true;
  // launch() resets what the kernels start from (the claim counter, and the counters or the
  // per-chunk counts of the planning pass) before or while it runs them
  return c128::launch(p, cfg, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? C128_OK : C128_ERR_CUDA;
}
