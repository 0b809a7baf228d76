// C-ABI of libc128compress: argument validation, per-(device, stream) workspaces, the kernel
// timer, and the launch of the planning and compress kernels. Declarations and their contract
// are in include/c128compress.h.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "c128_internal.h"
#include "c128compress.h"

namespace {

using c128::WsHeader;

constexpr int kVersion = 1;

struct Workspace {
  WsHeader* ptr = nullptr;
  int64_t capacity = 0;  // tokens the list holds
};

struct Timer {
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> events;
  size_t used = 0;
};

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int ctas_per_sm = 0;
};

std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
std::map<std::pair<int, cudaStream_t>, Timer> g_timers;
std::map<int, DeviceInfo> g_dev;

int cuda_fail(cudaError_t) { return C128_ERR_CUDA; }

// Must hold g_mu.
int device_info(int dev, DeviceInfo** out) {
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return C128_ERR_CUDA;
    if (c128::prepare_device(dev) != cudaSuccess) return C128_ERR_CUDA;
    d.ctas_per_sm = 1;
    d.ready = true;
  }
  *out = &d;
  return C128_OK;
}

// Must hold g_mu. Ensure the (dev, stream) workspace holds `tokens` list entries. Growth is
// stream-ordered and never waits on the host: the new buffer comes from the device's default
// memory pool (cudaMallocAsync on `stream`), the 256-byte header moves over with a device-to-device
// copy on `stream` (so the sticky error bits survive), and the old buffer goes back to the pool
// with cudaFreeAsync on `stream`, after every earlier call on the stream has used it. A stream
// that is being captured cannot grow its workspace: the call returns C128_ERR_CAPTURE.
int workspace_for(int dev, cudaStream_t stream, int64_t tokens, WsHeader** out) {
  Workspace& w = g_ws[{dev, stream}];
  if (w.ptr != nullptr && w.capacity >= tokens) {
    *out = w.ptr;
    return C128_OK;
  }
  cudaStreamCaptureStatus cap_status = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap_status) != cudaSuccess) {
    cudaGetLastError();
    return C128_ERR_CUDA;
  }
  if (cap_status != cudaStreamCaptureStatusNone) return C128_ERR_CAPTURE;
  int64_t cap = w.capacity > 0 ? w.capacity : 4096;
  while (cap < tokens) cap *= 2;
  void* p = nullptr;
  if (cudaMallocAsync(&p, sizeof(WsHeader) + static_cast<size_t>(cap) * sizeof(int32_t), stream) != cudaSuccess) {
    cudaGetLastError();
    return C128_ERR_NOMEM;
  }
  const cudaError_t e = w.ptr != nullptr
                            ? cudaMemcpyAsync(p, w.ptr, sizeof(WsHeader), cudaMemcpyDeviceToDevice, stream)
                            : cudaMemsetAsync(p, 0, sizeof(WsHeader), stream);
  if (e != cudaSuccess) {
    cudaFreeAsync(p, stream);
    return C128_ERR_CUDA;
  }
  if (w.ptr != nullptr && cudaFreeAsync(w.ptr, stream) != cudaSuccess) {
    cudaGetLastError();  // the old buffer stays allocated; the new one is in use from here on
  }
  w.ptr = static_cast<WsHeader*>(p);
  w.capacity = cap;
  *out = w.ptr;
  return C128_OK;
}

// ----------------------------------------------------------------------- descriptor checks
int check_desc(const c128_tensor_t* t, int dtype, int ndim) {
  if (t == nullptr) return C128_ERR_NULL_PTR;
  if (t->dtype != dtype) return C128_ERR_DTYPE;
  if (t->ndim != ndim) return C128_ERR_SHAPE;
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0) return C128_ERR_SHAPE;
  return C128_OK;
}
int64_t numel(const c128_tensor_t* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}
int check_data(const c128_tensor_t* t) {
  if (numel(t) > 0 && t->data == nullptr) return C128_ERR_NULL_PTR;
  return C128_OK;
}
int check_vector(const c128_tensor_t* t, int dtype, int64_t n) {
  int rc = check_desc(t, dtype, 1);
  if (rc) return rc;
  if (t->shape[0] != n) return C128_ERR_SHAPE;
  if (n > 1 && t->stride[0] != 1) return C128_ERR_STRIDE;
  return check_data(t);
}
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define C128_TRY(expr)         \
  do {                         \
    const int rc_ = (expr);    \
    if (rc_ != C128_OK) return rc_; \
  } while (0)

// Bytes of token data and of scales per k_cache slot, per cache format.
int64_t token_bytes(int fmt) { return fmt == C128_FORMAT_SPARSE_FP8 ? c128::kTokenStride : fmt == C128_FORMAT_INDEXER_FP8 ? 128 : 64; }
int64_t scale_bytes(int fmt) { return fmt == C128_FORMAT_SPARSE_FP8 ? c128::kScaleDim : 4; }

// Check a configuration of compress_norm_rope_store_ex (C128_ERR_UNSUPPORTED if the pages' kernels
// have no such case).
int check_config(const c128_config_t* c) {
  if (c == nullptr) return C128_ERR_NULL_PTR;
  if (c->rope_head_dim != c128::kRope) return C128_ERR_UNSUPPORTED;
  if (c->cache_format == C128_FORMAT_SPARSE_FP8) {
    if (c->head_dim != c128::kHead) return C128_ERR_UNSUPPORTED;
  } else if (c->cache_format == C128_FORMAT_INDEXER_FP8 || c->cache_format == C128_FORMAT_INDEXER_MXFP4) {
    if (c->head_dim != 128) return C128_ERR_UNSUPPORTED;
  } else {
    return C128_ERR_UNSUPPORTED;
  }
  if (c->overlap != 0 && c->overlap != 1) return C128_ERR_UNSUPPORTED;
  const int r = c->compress_ratio;
  if (r < 1 || (r & (r - 1)) != 0 || (1 + c->overlap) * r > 256) return C128_ERR_UNSUPPORTED;
  if (c->state_width < (1 + c->overlap) * c->head_dim || c->state_width % 4 != 0) return C128_ERR_UNSUPPORTED;
  return C128_OK;
}

int validate_call(const c128_tensor_t* ttr, const c128_tensor_t* pos, const c128_tensor_t* slot,
                  const c128_tensor_t* bt, const c128_tensor_t* state, const c128_tensor_t* rms_w, float eps,
                  const c128_tensor_t* cs, const c128_tensor_t* kc, const c128_tensor_t* kvslot,
                  int64_t kv_block_size, const c128_tensor_t* comp_out, c128::Params* out,
                  const c128_config_t* cfg) {
  // C128 unless a configuration is given
  const c128_config_t c128_cfg = {c128::kHead, c128::kRope, c128::kRatio, 0, c128::kHead, C128_FORMAT_SPARSE_FP8};
  if (cfg != nullptr) C128_TRY(check_config(cfg));
  const c128_config_t& C = cfg != nullptr ? *cfg : c128_cfg;
  const int64_t row_width = 2 * static_cast<int64_t>(C.state_width);
  // per-token vectors (the pages' token_to_req_indices, positions, slot_mapping, kv slot map)
  if (pos == nullptr) return C128_ERR_NULL_PTR;
  C128_TRY(check_desc(pos, C128_I64, 1));
  const int64_t T = pos->shape[0];
  C128_TRY(check_vector(pos, C128_I64, T));
  C128_TRY(check_vector(ttr, C128_I32, T));
  C128_TRY(check_vector(slot, C128_I64, T));
  C128_TRY(check_vector(kvslot, C128_I64, T));
  if (T > 0x7fffffffLL) return C128_ERR_ARG;
  // block table [R, MB] int32, rows may be padded
  C128_TRY(check_desc(bt, C128_I32, 2));
  if (bt->shape[1] > 1 && bt->stride[1] != 1) return C128_ERR_STRIDE;
  if (bt->shape[0] > 1 && bt->stride[0] < bt->shape[1]) return C128_ERR_STRIDE;
  C128_TRY(check_data(bt));
  // state cache [NB, block, 2*state_width] fp32 (C128 layout: state block 8, row = kv 512 | score 512)
  C128_TRY(check_desc(state, C128_F32, 3));
  if (cfg == nullptr && state->shape[1] != c128::kStateBlock) return C128_ERR_UNSUPPORTED;
  if (state->shape[1] < 1 || state->shape[2] != row_width) return C128_ERR_UNSUPPORTED;
  if (state->stride[2] != 1) return C128_ERR_STRIDE;
  if (state->stride[1] < row_width || state->stride[0] < 1) return C128_ERR_STRIDE;
  if (state->stride[1] % 4 != 0 || state->stride[0] % 4 != 0 || !aligned(state->data, 16)) return C128_ERR_ALIGN;
  C128_TRY(check_data(state));
  if (state->shape[0] > 0x7fffffffLL) return C128_ERR_ARG;
  // rms weight [head]
  C128_TRY(check_desc(rms_w, C128_F32, 1));
  if (rms_w->shape[0] != C.head_dim) return C128_ERR_UNSUPPORTED;
  if (rms_w->stride[0] != 1) return C128_ERR_STRIDE;
  C128_TRY(check_data(rms_w));
  if (!aligned(rms_w->data, 8)) return C128_ERR_ALIGN;
  // cos/sin cache [MP, 64] fp32
  C128_TRY(check_desc(cs, C128_F32, 2));
  if (cs->shape[1] != c128::kRope) return C128_ERR_UNSUPPORTED;
  if (cs->stride[1] != 1 || (cs->shape[0] > 1 && cs->stride[0] < c128::kRope)) return C128_ERR_STRIDE;
  C128_TRY(check_data(cs));
  // k_cache [NKB, bs, W] uint8, W >= slot bytes (584 for C128); block b is a flat byte range
  C128_TRY(check_desc(kc, C128_U8, 3));
  if (kv_block_size < 1 || kc->shape[1] != kv_block_size) return C128_ERR_ARG;
  if (kc->shape[2] < token_bytes(C.cache_format) + scale_bytes(C.cache_format)) return C128_ERR_SHAPE;
  if (kc->stride[2] != 1 || kc->stride[1] != kc->shape[2]) return C128_ERR_STRIDE;
  if (kc->shape[0] > 1 && kc->stride[0] < kc->shape[1] * kc->shape[2]) return C128_ERR_STRIDE;
  // the widest k_cache store: 8 bytes (bf16 rope quads, sparse), 4 (e4m3 quads and the fp32 scale,
  // indexer FP8), 2 (E2M1 byte pairs, MXFP4); block starts must keep that alignment
  const int kc_align = C.cache_format == C128_FORMAT_SPARSE_FP8 ? 8 : C.cache_format == C128_FORMAT_INDEXER_FP8 ? 4 : 2;
  if (kc->stride[0] % kc_align != 0 || !aligned(kc->data, 16)) return C128_ERR_ALIGN;
  C128_TRY(check_data(kc));
  // optional fp32 export [T, head]
  if (comp_out != nullptr) {
    C128_TRY(check_desc(comp_out, C128_F32, 2));
    if (comp_out->shape[0] != T || comp_out->shape[1] != C.head_dim) return C128_ERR_SHAPE;
    if (comp_out->stride[1] != 1 || (T > 1 && comp_out->stride[0] != C.head_dim)) return C128_ERR_STRIDE;
    C128_TRY(check_data(comp_out));
    if (!aligned(comp_out->data, 16)) return C128_ERR_ALIGN;
  }
  c128::Params& p = *out;
  p = c128::Params{};
  p.ttr = static_cast<const int32_t*>(ttr->data);
  p.pos = static_cast<const int64_t*>(pos->data);
  p.slot = static_cast<const int64_t*>(slot->data);
  p.kvslot = static_cast<const int64_t*>(kvslot->data);
  p.T = T;
  p.bt = static_cast<const int32_t*>(bt->data);
  p.bt_rows = bt->shape[0];
  p.bt_cols = bt->shape[1];
  p.bt_stride = bt->shape[0] > 1 ? bt->stride[0] : bt->shape[1];
  p.state = static_cast<const float*>(state->data);
  p.nb = state->shape[0];
  p.s0 = state->stride[0];
  p.s1 = state->stride[1];
  p.rms_w = static_cast<const float*>(rms_w->data);
  p.eps = eps;
  p.cs = static_cast<const float*>(cs->data);
  p.cs_rows = cs->shape[0];
  p.cs_stride = cs->shape[0] > 1 ? cs->stride[0] : c128::kRope;
  p.kc = static_cast<uint8_t*>(kc->data);
  p.nkb = kc->shape[0];
  p.kv_bs = kv_block_size;
  p.kc_stride0 = kc->shape[0] > 1 ? kc->stride[0] : kc->shape[1] * kc->shape[2];
  p.comp_out = comp_out != nullptr ? static_cast<float*>(comp_out->data) : nullptr;
  p.head = C.head_dim;
  p.ratio = C.compress_ratio;
  p.overlap = C.overlap;
  p.sw = C.state_width;
  p.fmt = C.cache_format;
  p.sblk = state->shape[1];
  return C128_OK;
}

int run(const c128_tensor_t* ttr, const c128_tensor_t* pos, const c128_tensor_t* slot,
        const c128_tensor_t* bt, const c128_tensor_t* state, const c128_tensor_t* rms_w, float eps,
        const c128_tensor_t* cs, const c128_tensor_t* kc, const c128_tensor_t* kvslot,
        int64_t kv_block_size, const c128_tensor_t* comp_out, cudaStream_t stream,
        const c128_config_t* config = nullptr, bool stall_test = false) {
  c128::Params p{};
  C128_TRY(validate_call(ttr, pos, slot, bt, state, rms_w, eps, cs, kc, kvslot, kv_block_size, comp_out, &p, config));
  p.stall_first_window = stall_test ? 1 : 0;
  const int64_t T = p.T;
  if (T == 0) return C128_OK;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return C128_ERR_CUDA;
  c128::LaunchCfg cfg{};
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo* di = nullptr;
    C128_TRY(device_info(dev, &di));
    C128_TRY(workspace_for(dev, stream, c128::plan_list_entries(T), &p.ws));
    cfg.sm_count = di->sm_count;
    // the C128 stall test needs the one-CTA-per-token or the compress kernel: more tokens than SMs
    if (stall_test && config == nullptr && T <= di->sm_count) return C128_ERR_ARG;
    const int64_t g = static_cast<int64_t>(di->sm_count) * di->ctas_per_sm;
    cfg.grid = static_cast<int>(T < g ? T : g);
    cfg.pdl = true;
    auto it = g_timers.find({dev, stream});
    if (it != g_timers.end() && it->second.on) {
      Timer& tm = it->second;
      if (tm.used == tm.events.size()) {
        cudaEvent_t a, b;
        if (cudaEventCreate(&a) != cudaSuccess) return C128_ERR_CUDA;
        if (cudaEventCreate(&b) != cudaSuccess) return C128_ERR_CUDA;
        tm.events.emplace_back(a, b);
      }
      cfg.ev_begin = tm.events[tm.used].first;
      cfg.ev_end = tm.events[tm.used].second;
      ++tm.used;
    }
  }
  const cudaError_t e = c128::launch(p, cfg, stream);
  return e == cudaSuccess ? C128_OK : cuda_fail(e);
}

}  // namespace

namespace c128 {
int validate_args(const c128_tensor_t* ttr, const c128_tensor_t* pos, const c128_tensor_t* slot,
                  const c128_tensor_t* bt, const c128_tensor_t* state, const c128_tensor_t* rms_w, float eps,
                  const c128_tensor_t* cs, const c128_tensor_t* kc, const c128_tensor_t* kvslot,
                  int64_t kv_block_size, const c128_tensor_t* comp_out, Params* out, const c128_config_t* cfg) {
  return validate_call(ttr, pos, slot, bt, state, rms_w, eps, cs, kc, kvslot, kv_block_size, comp_out, out, cfg);
}
}  // namespace c128

extern "C" {

int compress_norm_rope_store(const c128_tensor_t* token_to_req_indices, const c128_tensor_t* positions,
                             const c128_tensor_t* slot_mapping, const c128_tensor_t* block_table,
                             const c128_tensor_t* state_cache, const c128_tensor_t* rms_w, float eps,
                             const c128_tensor_t* cos_sin_cache, const c128_tensor_t* k_cache,
                             const c128_tensor_t* kv_slot_mapping, int64_t kv_block_size,
                             c128_stream_t stream) {
  return run(token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w, eps,
             cos_sin_cache, k_cache, kv_slot_mapping, kv_block_size, nullptr,
             reinterpret_cast<cudaStream_t>(stream));
}

int c128_debug_stall_first_window(const c128_tensor_t* token_to_req_indices, const c128_tensor_t* positions,
                                   const c128_tensor_t* slot_mapping, const c128_tensor_t* block_table,
                                   const c128_tensor_t* state_cache, const c128_tensor_t* rms_w, float eps,
                                   const c128_tensor_t* cos_sin_cache, const c128_tensor_t* k_cache,
                                   const c128_tensor_t* kv_slot_mapping, int64_t kv_block_size,
                                   c128_stream_t stream) {
  return run(token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w, eps,
             cos_sin_cache, k_cache, kv_slot_mapping, kv_block_size, nullptr,
             reinterpret_cast<cudaStream_t>(stream), nullptr, true);
}

int c128_debug_stall_first_window_ex(const c128_config_t* config, const c128_tensor_t* token_to_req_indices,
                                      const c128_tensor_t* positions, const c128_tensor_t* slot_mapping,
                                      const c128_tensor_t* block_table, const c128_tensor_t* state_cache,
                                      const c128_tensor_t* rms_w, float eps, const c128_tensor_t* cos_sin_cache,
                                      const c128_tensor_t* k_cache, const c128_tensor_t* kv_slot_mapping,
                                      int64_t kv_block_size, c128_stream_t stream) {
  if (config == nullptr) return C128_ERR_NULL_PTR;
  return run(token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w, eps,
             cos_sin_cache, k_cache, kv_slot_mapping, kv_block_size, nullptr,
             reinterpret_cast<cudaStream_t>(stream), config, true);
}

int c128_compress_norm_rope_store_debug(const c128_tensor_t* token_to_req_indices,
                                        const c128_tensor_t* positions, const c128_tensor_t* slot_mapping,
                                        const c128_tensor_t* block_table, const c128_tensor_t* state_cache,
                                        const c128_tensor_t* rms_w, float eps,
                                        const c128_tensor_t* cos_sin_cache, const c128_tensor_t* k_cache,
                                        const c128_tensor_t* kv_slot_mapping, int64_t kv_block_size,
                                        const c128_tensor_t* comp_out, c128_stream_t stream) {
  if (comp_out == nullptr) return C128_ERR_NULL_PTR;
  return run(token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w, eps,
             cos_sin_cache, k_cache, kv_slot_mapping, kv_block_size, comp_out,
             reinterpret_cast<cudaStream_t>(stream));
}

int compress_norm_rope_store_ex(const c128_config_t* config, const c128_tensor_t* token_to_req_indices,
                                const c128_tensor_t* positions, const c128_tensor_t* slot_mapping,
                                const c128_tensor_t* block_table, const c128_tensor_t* state_cache,
                                const c128_tensor_t* rms_w, float eps, const c128_tensor_t* cos_sin_cache,
                                const c128_tensor_t* k_cache, const c128_tensor_t* kv_slot_mapping,
                                int64_t kv_block_size, const c128_tensor_t* comp_out, c128_stream_t stream) {
  if (config == nullptr) return C128_ERR_NULL_PTR;
  return run(token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w, eps, cos_sin_cache,
             k_cache, kv_slot_mapping, kv_block_size, comp_out, reinterpret_cast<cudaStream_t>(stream), config);
}

const char* c128_status_string(int status) {
  switch (status) {
    case C128_OK: return "ok";
    case C128_ERR_NULL_PTR: return "null pointer";
    case C128_ERR_DTYPE: return "wrong dtype";
    case C128_ERR_SHAPE: return "wrong shape";
    case C128_ERR_STRIDE: return "unsupported stride";
    case C128_ERR_ALIGN: return "misaligned base or stride";
    case C128_ERR_UNSUPPORTED:
      return "unsupported configuration or layout (C128: state block 8, row 1024, head 512, rope 64)";
    case C128_ERR_ARG: return "bad argument (kv_block_size must equal k_cache.shape[1]; too many tokens)";
    case C128_ERR_CUDA: return "CUDA error";
    case C128_ERR_NOMEM: return "workspace allocation failed";
    case C128_ERR_CAPTURE:
      return "the stream's workspace would have to grow while the stream is being captured "
             "(call c128_reserve_workspace with the largest batch before capturing)";
    case C128_ERR_TOO_MANY_TOKENS:
      return "more tokens than the static workspace of c128_compress_norm_rope_store_noalloc holds "
             "(C128_NOALLOC_MAX_TOKENS)";
    default: return "unknown status";
  }
}

int c128_reserve_workspace(int64_t max_tokens, c128_stream_t stream) {
  if (max_tokens < 0 || max_tokens > 0x7fffffffLL) return C128_ERR_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return C128_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo* di = nullptr;
  C128_TRY(device_info(dev, &di));
  WsHeader* ws = nullptr;
  return workspace_for(dev, reinterpret_cast<cudaStream_t>(stream), c128::plan_list_entries(max_tokens > 0 ? max_tokens : 1),
                       &ws);
}

int c128_device_errors(c128_stream_t stream, uint32_t* bits, int clear) {
  if (bits == nullptr) return C128_ERR_NULL_PTR;
  *bits = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return C128_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_ws.find({dev, s});
  if (it == g_ws.end() || it->second.ptr == nullptr) return C128_OK;
  if (cudaStreamSynchronize(s) != cudaSuccess) return C128_ERR_CUDA;
  unsigned int err = 0;
  if (cudaMemcpy(&err, &it->second.ptr->err, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess)
    return C128_ERR_CUDA;
  *bits = err;
  if (clear && err) {
    const unsigned int zero = 0;
    if (cudaMemcpy(&it->second.ptr->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return C128_ERR_CUDA;
  }
  return C128_OK;
}

int c128_kernel_timer_begin(c128_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return C128_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  Timer& tm = g_timers[{dev, reinterpret_cast<cudaStream_t>(stream)}];
  tm.on = true;
  tm.used = 0;
  return C128_OK;
}

int c128_kernel_timer_end(c128_stream_t stream, double* total_ms, int64_t* launches) {
  if (total_ms == nullptr || launches == nullptr) return C128_ERR_NULL_PTR;
  *total_ms = 0.0;
  *launches = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return C128_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_timers.find({dev, s});
  if (it == g_timers.end()) return C128_OK;
  Timer& tm = it->second;
  tm.on = false;
  if (cudaStreamSynchronize(s) != cudaSuccess) return C128_ERR_CUDA;
  double sum = 0.0;
  for (size_t i = 0; i < tm.used; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, tm.events[i].first, tm.events[i].second) != cudaSuccess) return C128_ERR_CUDA;
    sum += ms;
  }
  *total_ms = sum;
  *launches = static_cast<int64_t>(tm.used);
  tm.used = 0;
  return C128_OK;
}

int c128_get_info(c128_info_t* info) {
  if (info == nullptr) return C128_ERR_NULL_PTR;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return C128_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo* di = nullptr;
  C128_TRY(device_info(dev, &di));
  info->sm_count = di->sm_count;
  info->threads = c128::kThreads;
  info->smem_bytes = c128::compress_smem_bytes();
  info->stages = c128::kStages;
  info->ctas_per_sm = di->ctas_per_sm;
  info->plan_tokens_per_cta = c128::kPlanTokensPerCta;
  info->wait_timeout_ms = static_cast<int32_t>(c128::kWaitTimeoutNs / 1000000ull);
  info->version = kVersion;
  return C128_OK;
}

int c128_release_stream(c128_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return C128_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap_status = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap_status) != cudaSuccess) {
    cudaGetLastError();
    return C128_ERR_CUDA;
  }
  if (cap_status != cudaStreamCaptureStatusNone) return C128_ERR_CAPTURE;  // a free would join the graph
  std::lock_guard<std::mutex> lk(g_mu);
  int rc = C128_OK;
  auto it = g_ws.find({dev, s});
  if (it != g_ws.end()) {
    if (it->second.ptr != nullptr && cudaFreeAsync(it->second.ptr, s) != cudaSuccess) {
      cudaGetLastError();
      rc = C128_ERR_CUDA;
    }
    g_ws.erase(it);
  }
  auto tt = g_timers.find({dev, s});
  if (tt != g_timers.end()) {
    for (auto& ev : tt->second.events) {  // destruction waits for pending records by itself
      cudaEventDestroy(ev.first);
      cudaEventDestroy(ev.second);
    }
    g_timers.erase(tt);
  }
  return rc;
}

int c128_release_all(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return C128_ERR_CUDA;
  int rc = C128_OK;
  for (auto& kv : g_ws) {
    if (kv.second.ptr == nullptr) continue;
    // the buffer came from the pool of device kv.first.first: free it there, after all work
    if (cudaSetDevice(kv.first.first) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        cudaFreeAsync(kv.second.ptr, 0) != cudaSuccess || cudaStreamSynchronize(0) != cudaSuccess) {
      cudaGetLastError();
      rc = C128_ERR_CUDA;
    }
  }
  g_ws.clear();
  if (!g_timers.empty() && cudaDeviceSynchronize() != cudaSuccess) rc = C128_ERR_CUDA;
  for (auto& kv : g_timers)
    for (auto& ev : kv.second.events) {
      cudaEventDestroy(ev.first);
      cudaEventDestroy(ev.second);
    }
  g_timers.clear();
  if (cudaSetDevice(cur) != cudaSuccess) rc = C128_ERR_CUDA;
  return rc;
}

}  // extern "C"
