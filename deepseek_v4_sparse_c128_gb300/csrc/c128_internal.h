// Internal declarations shared by the kernel translation unit and the C-ABI layer.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "c128compress.h"

namespace c128 {

// C128 layout (vLLM PR #44230, Summary; fused_compress_quant_cache API page, constexprs of
// _fused_kv_compress_norm_rope_insert_sparse_attn).
constexpr int kHead = 512;          // head size = state width
constexpr int kRow = 1024;          // fp32 values per state row: kv[512] | score[512]
constexpr int kStateBlock = 8;      // rows per state-cache block
constexpr int kRatio = 128;         // compress ratio = rows per window
constexpr int kWindowBlocks = kRatio / kStateBlock;  // 16
constexpr int kNope = 448;
constexpr int kRope = 64;
constexpr int kQuantBlock = 64;
constexpr int kTokenStride = 576;   // bytes: 448 e4m3 + 64 bf16
constexpr int kScaleDim = 8;        // 7 UE8M0 bytes + 1 zero pad
constexpr int kSlotBytes = kTokenStride + kScaleDim;  // 584

// Compress-kernel geometry.
#ifndef C128_STAGES
#define C128_STAGES 6
#endif
constexpr int kStages = C128_STAGES;               // smem ring depth, one state block per stage
constexpr int kStageBytes = kStateBlock * kRow * 4;  // 32 KiB
constexpr int kDescSlots = 2;                      // windows in flight per CTA
constexpr int kConsumerWarps = 8;                  // warp w owns columns [64w, 64w+64)
constexpr int kThreads = 64 + 32 * kConsumerWarps;  // scheduler warp, copy warp, consumers
constexpr int kPlanThreads = 256;
constexpr int kPlanTokensPerThread = 8;
constexpr int kPlanTokensPerCta = kPlanThreads * kPlanTokensPerThread;
// Up to this many tokens per SM the kernels run without the planning pass (C128: one CTA per
// token; the other configurations: token striding).
constexpr int kStridedTokensPerSm = 8;
// The planning pass writes, per chunk c of kPlanTokensPerCta tokens, its active tokens in token
// order at list[c * kPlanTokensPerCta ...] and their number at list[T + c]: nothing accumulates
// across CTAs or calls, so the pass needs no zeroed counters. The kernels that take windows from
// the list keep the prefix of the counts in shared memory, which bounds the chunks; above that a
// compact list behind a zeroing pass serves.
constexpr int kMaxPlanChunks = 512;  // token_num <= 512 x 2048 = 1 Mi
// List entries (int32) the workspace needs for a call of `T` tokens: the list and the counts.
constexpr int64_t plan_list_entries(int64_t T) { return T + (T + kPlanTokensPerCta - 1) / kPlanTokensPerCta; }
constexpr unsigned long long kWaitTimeoutNs = 1000ull * 1000ull * 1000ull;  // 1 s per wait

// Workspace layout: a 256-byte header then the list of active token indices.
struct WsHeader {
  unsigned int count;   // active windows of the compact list (zeroed per call; calls whose
                        // planning pass writes per-chunk counts do not use it)
  unsigned int next;    // the window kernels' shared claim counter (zeroed per call: by a
                        // memset, or by the per-chunk planning pass)
  unsigned int err;     // sticky C128_DEV_* bits
  unsigned int pad[61];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

struct Params {
  const int32_t* ttr;
  const int64_t* pos;
  const int64_t* slot;
  const int64_t* kvslot;
  int64_t T;
  const int32_t* bt;
  int64_t bt_rows, bt_cols, bt_stride;
  const float* state;
  int64_t nb, s0, s1;         // blocks, strides in elements
  const float* rms_w;
  float eps;
  const float* cs;
  int64_t cs_rows, cs_stride;
  uint8_t* kc;
  int64_t nkb, kv_bs, kc_stride0;  // blocks, block size, block stride in bytes
  float* comp_out;            // nullable [T, head]
  WsHeader* ws;               // header; the token list follows it
  // configuration (C128: head 512, ratio 128, no overlap, state width 512, format 0, block 8)
  int32_t head;               // 512 or 128
  int32_t ratio;              // compress ratio (a power of two)
  int32_t overlap;            // 1: windows of 2*ratio rows, the newer half read at +head
  int32_t sw;                 // state width: kv columns of a row, as many score columns follow
  int32_t fmt;                // cache format (C128_FORMAT_*)
  int64_t sblk;               // state-cache block size (rows per block)
  int32_t strided;            // small-window and indexer kernels: no planning pass, CTA c takes
                              // tokens c, c + grid, ...
  int32_t chunked;            // planned path: the list is per chunk (plan_chunks_kernel), else compact
  int32_t stall_first_window; // test only: one stage is armed but never filled (CTA 0's first in
                              // the compress, one-CTA-per-token and indexer kernels, the first
                              // listed window's in the small-window kernel)
};

// True for the configurations the specialised C128 kernels serve: the C128 layout, with 8-row
// state blocks or, through the configurable entry point, any multiple of 8 rows.
inline bool is_c128(const Params& p) {
  return p.head == kHead && p.ratio == kRatio && p.overlap == 0 && p.sw == kHead && p.fmt == 0 &&
         p.sblk >= kStateBlock && p.sblk % kStateBlock == 0;
}

struct LaunchCfg {
  int sm_count;
  int grid;
  bool pdl;
  cudaEvent_t ev_begin;  // recorded around the compress kernel when non-null
  cudaEvent_t ev_end;
};

// Check every argument of compress_norm_rope_store (C128_* code) and fill all of `out` but `ws`.
// `cfg` == nullptr means the C128 configuration (state block 8 required).
int validate_args(const c128_tensor_t* ttr, const c128_tensor_t* pos, const c128_tensor_t* slot,
                  const c128_tensor_t* bt, const c128_tensor_t* state, const c128_tensor_t* rms_w, float eps,
                  const c128_tensor_t* cs, const c128_tensor_t* kc, const c128_tensor_t* kvslot,
                  int64_t kv_block_size, const c128_tensor_t* comp_out, Params* out,
                  const c128_config_t* cfg = nullptr);

// Enqueue zeroing of the per-call counters, the planning kernel and the compress kernel.
cudaError_t launch(const Params& p, const LaunchCfg& cfg, cudaStream_t stream);
// The kernels for configurations other than C128 (after plan_kernel): windows of at most 8 rows
// (c128_c4.cu) and the rest (c128_gather.cu).
cudaError_t launch_gather(const Params& p, const LaunchCfg& cfg, cudaStream_t stream);
bool small_window_path(const Params& p);
cudaError_t launch_small(const Params& p, const LaunchCfg& cfg, cudaStream_t stream);
cudaError_t prepare_small();  // function attributes of the small-window kernels
// Head-128 windows of more than 8 rows (c128_indexer.cu); cudaErrorNotSupported (nothing
// launched) when the configuration or the state layout does not fit that kernel.
cudaError_t launch_indexer_windows(const Params& p, const LaunchCfg& cfg, cudaStream_t stream);
cudaError_t prepare_indexer_windows();
// Tensor map of the state cache for tiled loads of `box_rows` rows x (head kv + head score
// columns); false when the layout does not allow one (c128_c4.cu).
bool encode_state_map(const Params& p, int head, int box_rows, CUtensorMap* map);
int compress_smem_bytes();
cudaError_t prepare_device(int device);  // one-time function attributes

}  // namespace c128
