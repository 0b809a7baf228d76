// sm_103a kernel for windows of at most 8 rows (the C4 layout: compress ratio 4 with overlap):
// a persistent CTA per SM that streams many small windows through a ring of shared-memory stages.
//
//   warp 0      scheduler: claims 32 windows at a time; one lane per window resolves the token's
//               request, position, cache slot and state blocks, checks them, and writes the
//               resolved windows into a queue of two batches.
//   warp 1      copier: lane l takes the queued windows l, l + S, ... of each batch (S stages),
//               each on the stage it maps to; the warp polls its lanes' stages together, so a
//               lane issues as soon as its own stage is free. It writes the stage's descriptor and
//               issues the copies: one tiled TMA load (`cp.async.bulk.tensor.5d`) per group of
//               `ratio` consecutive rows (the older and the newer half of an overlapping window),
//               whose box takes the kv half-row and the score half-row of every row of the group;
//               where the state layout does not allow such a box (a group split across state
//               blocks), one `cp.async.bulk` per half-row instead. Completion is counted in bytes
//               on the stage's mbarrier.
//   warps 2..13 consumer groups: head 512 (sparse FP8 cache) three groups of four warps (thread i
//               owns columns 4i..4i+3), head 128 (indexer FP8 or MXFP4 cache) twelve one-warp
//               groups (lane l owns columns 4l..4l+3). Group g owns stages g, g + G, ...: it takes
//               windows g, g + G, ... in order, so each stage's barrier phases are produced and
//               consumed in order. A group releases its stage as soon as it has the compressed
//               vector (and has loaded the cos/sin it needs), before its epilogue.
//
// Same arithmetic as the oracle's reading of _fused_kv_compress_norm_rope_insert_indexer_attn,
// ..._indexer_mxfp4_attn and ..._sparse_attn on the API page of
// vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache (gather with overlap: 2*ratio rows,
// the newer half at +head, rows at negative positions masked).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "c128_device.cuh"
#include "c128_warp_epilogue.cuh"

namespace c128 {
namespace {

constexpr int kMaxSmallRows = 8;
constexpr int kBatch = 32;  // windows claimed at once
#ifndef C128_SMALL_GROUPS_512
#define C128_SMALL_GROUPS_512 6
#endif
#ifndef C128_SMALL_STAGES_512
#define C128_SMALL_STAGES_512 6
#endif
#ifndef C128_SMALL_GROUPS_128
#define C128_SMALL_GROUPS_128 12
#endif
#ifndef C128_SMALL_STAGES_128
#define C128_SMALL_STAGES_128 24
#endif
#ifndef C128_C4_POLL_NS
#define C128_C4_POLL_NS 64  // the copier's back-off when none of its lanes could issue
#endif
constexpr int kFlagTiled = 1;  // the state map serves the row copies

// ------------------------------------------------------------------------------ ring layout
// Per-quad scratch of the head-512 epilogue; 16-byte aligned because comp[] takes float4 stores.
struct __align__(16) QuadSmem {
  unsigned long long lo[4], hi[4];
  uint32_t emax[4], special[4], fb[4];
  float comp[512];
  float rrms;
};
static_assert(offsetof(QuadSmem, comp) % 16 == 0 && sizeof(QuadSmem) % 16 == 0, "float4 access to QuadSmem::comp");
struct __align__(16) WarpSmem128 {  // per-warp compressed vector for the rare exact-variance slow path
  float comp[128];
};

template <int HEAD>
struct SmallGeo {
  static constexpr int kGroupWarps = HEAD == 512 ? 4 : 1;
  static constexpr int kGroups = HEAD == 512 ? C128_SMALL_GROUPS_512 : C128_SMALL_GROUPS_128;
  static constexpr int kThreads = 32 * (2 + kGroups * kGroupWarps);  // scheduler, copier, consumer groups
  static constexpr int kRowFloats = 2 * HEAD;                         // kv half-row, then score half-row
  static constexpr int kStageFloats = kMaxSmallRows * kRowFloats;
  static constexpr int kStages = HEAD == 512 ? C128_SMALL_STAGES_512 : C128_SMALL_STAGES_128;  // about 200 KiB
  static_assert(kStages % kGroups == 0, "every stage belongs to one consumer group");
  using GroupSmem = typename std::conditional<HEAD == 512, QuadSmem, WarpSmem128>::type;
};

// One resolved window: queue entry (scheduler -> copier) and stage descriptor (copier -> group).
struct __align__(16) SmallDesc {
  const float* row[kMaxSmallRows];  // kv half-row of each present row, oldest first; its score at + state width
  uint8_t* tok;                     // token bytes of the cache slot
  uint8_t* scale;                   // scale bytes of the slot
  const float* cs_row;              // cos/sin row (p / ratio) * ratio
  float* comp_dst;                  // optional fp32 export
  int32_t nvalid;                   // rows present, 1..8; 0 marks the end of the work
  int32_t ngroups;                  // tiled path: groups of `ratio` rows present (1 or 2)
  int32_t g_blk[2];                 // tiled path: state block, first row in it and half of each group
  int32_t g_row[2];
  int32_t g_half[2];
  int32_t stall;                    // test only: leave this window's stage unfilled
  int32_t pad[2];
};

template <int HEAD>
struct SmallSmem {
  using G = SmallGeo<HEAD>;
  float stage[G::kStages][G::kStageFloats];
  SmallDesc desc[G::kStages];
  SmallDesc queue[2][kBatch];  // resolved windows of two claimed batches
  int32_t qcount[2];           // windows in the batch; -1: no more work
  uint64_t full[G::kStages];   // descriptor written and the window's bytes landed (1 arrival + bytes)
  uint64_t empty[G::kStages];  // the group is done with stage and descriptor (one arrival per group warp)
  uint64_t qfull[2];           // batch resolved (one arrival per scheduler lane)
  uint64_t qempty[2];          // batch taken (one arrival per copier lane)
  typename G::GroupSmem grp[G::kGroups];
  uint32_t chunk_prefix[kMaxPlanChunks + 1];  // planned path: active windows before each chunk
  int abort_flag;
};
static_assert(sizeof(SmallSmem<512>) <= 227 * 1024 && sizeof(SmallSmem<128>) <= 227 * 1024, "shared memory");
static_assert(sizeof(float) * SmallGeo<512>::kStageFloats % 128 == 0 &&
                  sizeof(float) * SmallGeo<128>::kStageFloats % 128 == 0,
              "stages stay 128-byte aligned");

template <int FMT>
struct SlotGeo {
  static constexpr int kTok = FMT == C128_FORMAT_SPARSE_FP8 ? kTokenStride : FMT == C128_FORMAT_INDEXER_FP8 ? 128 : 64;
  static constexpr int kScale = FMT == C128_FORMAT_SPARSE_FP8 ? kScaleDim : 4;
};

__device__ __forceinline__ bool group_bar_or(int id, int threads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ void group_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Tiled TMA load of one box of the state map (coordinates innermost first) into shared memory.
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

// Non-blocking test of a phase: true once the phase with this parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void set_timeout(const Params& p, int* abort_flag) {
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
  atomicOr(&p.ws->err, static_cast<unsigned>(C128_DEV_TIMEOUT));
}

// ------------------------------------------------------------------------------ scheduler warp
template <int HEAD, int FMT>
__device__ void small_scheduler(const Params& p, SmallSmem<HEAD>& S, int lane, bool tiled) {
  // list mode: windows from plan_kernel's list; token striding (few tokens, no planning pass):
  // this CTA tests tokens c, c + grid, ..., 32 candidates per step
  const bool strided = p.strided != 0;
  const volatile int* abort_flag = &S.abort_flag;
  // planned path (the kernel entry waited for the planning pass): the list's windows
  const uint32_t A = strided ? 0u : plan_prefix_warp(p, S.chunk_prefix, lane);
  const int n = (1 + p.overlap) * p.ratio;  // <= 8
  // claim size: 32 windows when there is plenty of work, else about one claim per CTA, so that a
  // small batch spreads over the SMs instead of a few CTAs taking 32 windows each
  const uint32_t per_cta = (A + gridDim.x - 1) / gridDim.x;
  uint32_t batch = per_cta >= static_cast<uint32_t>(kBatch) ? static_cast<uint32_t>(kBatch) : max(per_cta, 1u);
  int64_t next_t = blockIdx.x;
  bool stall_pending = strided && p.stall_first_window && blockIdx.x == 0;
  bool failed = false;
  for (uint32_t b = 0;; ++b) {
    const int qs = b & 1;
    if (b >= 2) {  // the queue slot of batch b - 2 is free once the copier took it
      const bool ok = mbar_wait_suspend(&S.qempty[qs], ((b >> 1) - 1u) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        failed = true;
        break;
      }
    }
    uint32_t base = 0;
    if (!strided && lane == 0) base = atomicAdd(&p.ws->next, batch);
    base = __shfl_sync(0xffffffffu, base, 0);
    // this claim takes windows base .. base + claim - 1; the next one is sized by what is left after
    // it (guided: a half share per CTA for head 128, a third with at least 2 windows for head 512,
    // at most kBatch), so the last claims of a call are small and the CTAs finish together. A
    // window's stage and group do not depend on the claim sizes.
    const uint32_t claim = batch;
    if (!strided) {
      constexpr uint32_t kDiv = HEAD == 512 ? 3u : 2u, kMin = HEAD == 512 ? 2u : 1u;
      const uint32_t left = A > base + claim ? A - (base + claim) : 0u;
      batch = min(static_cast<uint32_t>(kBatch), max(kMin, left / (kDiv * gridDim.x)));
    }
    if (strided ? next_t >= p.T : base >= A) {
      if (lane == 0) S.qcount[qs] = -1;
      mbar_arrive(&S.qfull[qs]);
      break;
    }
    // every lane resolves one window
    const uint32_t a = base + lane;
    bool live;
    int64_t t = 0, pos = 0, kvs = 0, cp = 0, start = 0, first = 0;
    if (strided) {
      t = next_t + static_cast<int64_t>(lane) * gridDim.x;
      next_t += 32ll * gridDim.x;
      live = false;
      if (t < p.T) {
        const int64_t sl = __ldg(p.slot + t), ps = __ldg(p.pos + t), kv = __ldg(p.kvslot + t);
        live = (sl >= 0) & (ps >= 0) & (((ps + 1) & (p.ratio - 1)) == 0) & (kv >= 0);
      }
    } else {
      live = a < A && static_cast<uint32_t>(lane) < claim;
      if (live) t = plan_token(p, S.chunk_prefix, a);
    }
    int req = 0, nvalid = 0, ngroups = 0;
    int blk0 = 0, row0 = 0, half0 = 0, blk1 = 0, row1 = 0, half1 = 0;
    uint32_t err = 0;
    if (live) {
      req = __ldg(p.ttr + t);
      pos = __ldg(p.pos + t);
      kvs = __ldg(p.kvslot + t);
      cp = pos & ~static_cast<int64_t>(p.ratio - 1);  // (p / ratio) * ratio; ratio is a power of two
      if (req < 0 || req >= p.bt_rows) err |= C128_DEV_BAD_REQ;
      if (pos / p.sblk >= p.bt_cols) err |= C128_DEV_BAD_BT_COL;
      if (cp >= p.cs_rows) err |= C128_DEV_BAD_COS_ROW;
      if (kvs >= p.nkb * p.kv_bs) err |= C128_DEV_BAD_KV_SLOT;
      start = pos - n + 1;
      first = start > 0 ? start : 0;  // rows before position 0 are masked
      nvalid = static_cast<int>(pos - first + 1);
    }
    const int32_t* bt_row = p.bt + static_cast<int64_t>(req) * p.bt_stride;
    const bool rows_ok = live && !(err & (C128_DEV_BAD_REQ | C128_DEV_BAD_BT_COL));
    if (rows_ok && tiled) {
      // groups of `ratio` rows start at multiples of ratio, so each is wholly present or masked,
      // and (state block a multiple of ratio) lies in one state block
      const int64_t q0 = start, q1 = start + p.ratio;
      if (q0 >= 0) {
        blk0 = __ldg(bt_row + q0 / p.sblk);
        row0 = static_cast<int>(q0 % p.sblk);
        half0 = 0;
        ngroups = 1;
      }
      if (p.overlap) {
        const int b1 = __ldg(bt_row + q1 / p.sblk);
        const int r1 = static_cast<int>(q1 % p.sblk);
        if (ngroups == 0) {
          blk0 = b1;
          row0 = r1;
          half0 = 1;
        } else {
          blk1 = b1;
          row1 = r1;
          half1 = 1;
        }
        ++ngroups;
      }
      if (blk0 < 0 || blk0 >= p.nb || (ngroups > 1 && (blk1 < 0 || blk1 >= p.nb))) err |= C128_DEV_BAD_BLOCK;
    }
    if (err) {
      atomicOr(&p.ws->err, err);
      live = false;
    }
    const uint32_t live_mask = __ballot_sync(0xffffffffu, live);
    const int rank = __popc(live_mask & ((1u << lane) - 1u));
    if (live) {
      SmallDesc& d = S.queue[qs][rank];
      const int64_t kb = kvs / p.kv_bs, off = kvs - kb * p.kv_bs;
      uint8_t* blk_base = p.kc + kb * p.kc_stride0;
      d.tok = blk_base + off * SlotGeo<FMT>::kTok;
      d.scale = blk_base + p.kv_bs * SlotGeo<FMT>::kTok + off * SlotGeo<FMT>::kScale;
      d.cs_row = p.cs + cp * p.cs_stride;
      d.comp_dst = p.comp_out ? p.comp_out + t * HEAD : nullptr;
      d.nvalid = nvalid;
      d.ngroups = ngroups;
      d.g_blk[0] = blk0;
      d.g_row[0] = row0;
      d.g_half[0] = half0;
      d.g_blk[1] = blk1;
      d.g_row[1] = row1;
      d.g_half[1] = half1;
      // test only: the first window of the list, or CTA 0's first window when striding
      d.stall = p.stall_first_window && (strided ? stall_pending && rank == 0 : a == 0);
      if (!tiled) {
        bool bad = false;
#pragma unroll
        for (int i = 0; i < kMaxSmallRows; ++i) {
          const float* r = nullptr;
          if (i < nvalid) {
            const int64_t q = first + i;
            const int b = __ldg(bt_row + q / p.sblk);
            if (b < 0 || b >= p.nb) {
              bad = true;
            } else {
              const int koff = (p.overlap && q - start >= p.ratio) ? HEAD : 0;
              r = p.state + static_cast<int64_t>(b) * p.s0 + (q % p.sblk) * p.s1 + koff;
            }
          }
          d.row[i] = r;
        }
        // a bad block id found here turns the window into one without rows to copy: the
        // copier then only signals the stage and the group skips it (nvalid < 0)
        if (bad) {
          atomicOr(&p.ws->err, static_cast<unsigned>(C128_DEV_BAD_BLOCK));
          d.nvalid = -1;
        }
      }
    }
    if (live_mask) stall_pending = false;
    if (lane == 0) S.qcount[qs] = __popc(live_mask);
    mbar_arrive(&S.qfull[qs]);
  }
  if (failed && lane == 0) set_timeout(p, &S.abort_flag);
}

// --------------------------------------------------------------------------------- copier warp
template <int HEAD>
__device__ void small_copier(const Params& p, SmallSmem<HEAD>& S, int lane, const CUtensorMap* map, bool tiled) {
  using G = SmallGeo<HEAD>;
  constexpr int kCw = HEAD < 256 ? HEAD : 256;
  static_assert(G::kStages <= 32 && G::kGroups <= G::kStages, "one copier lane per stage, one end marker per group");
  const volatile int* abort_flag = &S.abort_flag;
  const uint64_t policy = l2_evict_first_policy();
  const bool joined = p.sw == HEAD;  // the score half-row follows the kv half-row: one copy per row
  uint32_t k = 0;                    // windows given a stage so far
  bool failed = false;
  int pass_slot = -1;                // the stage of this lane's last window in the batch that failed,
  uint32_t pass_k = 0;               // if it issued copies, and that window
  for (uint32_t b = 0; !failed; ++b) {
    const int qs = b & 1;
    bool ok = mbar_wait_suspend(&S.qfull[qs], (b >> 1) & 1u, abort_flag);
    if (!__all_sync(0xffffffffu, ok)) {
      failed = true;
      break;
    }
    const int n = S.qcount[qs];
    if (n < 0) break;
    // Lane l < kStages takes the batch's windows j = l, l + kStages, ... (< n) in order; window j
    // is window k + j overall and goes to stage (k + j) % kStages, which last held window
    // k + j - kStages (same group) and is free once that group released it. The warp polls the
    // lanes' stages together and each lane issues its next window as soon as its own stage is free
    // (a blocking wait per lane would hold every lane until the last stage of the batch is free).
    int j = lane;
    bool pending = lane < G::kStages && j < n;
    ok = true;
    uint64_t t_progress = global_timer_ns();
    for (;;) {
      const uint32_t kk = k + static_cast<uint32_t>(j);
      const int sl = kk % G::kStages;
      const bool ready = pending && (kk < static_cast<uint32_t>(G::kStages) ||
                                     mbar_test_wait(&S.empty[sl], ((kk / G::kStages) - 1u) & 1u));
      if (ready) {
        const SmallDesc& e = S.queue[qs][j];
        SmallDesc& d = S.desc[sl];
        const int nvalid = e.nvalid;
        d.tok = e.tok;
        d.scale = e.scale;
        d.cs_row = e.cs_row;
        d.comp_dst = e.comp_dst;
        d.nvalid = nvalid;
        if (nvalid < 0) {
          mbar_arrive(&S.full[sl]);  // nothing to copy: the group skips the window
        } else {
          // the arrival releases the descriptor to the group that waits on this stage
          mbar_arrive_expect_tx(&S.full[sl], static_cast<uint32_t>(nvalid * G::kRowFloats * 4));
          pass_slot = sl;
          pass_k = kk;
          float* st = S.stage[sl];
          if (e.stall) {
            // test of the bounded waits: this stage never fills, so its group gives up after the
            // time limit and the kernel reports C128_DEV_TIMEOUT instead of hanging
          } else if (tiled) {
            // box {cw, head/cw, 2, ratio, 1}: per row the kv half-row, then the score half-row
            const int ng = e.ngroups;
            for (int g = 0; g < ng; ++g)
              tma_load_5d(st + g * p.ratio * G::kRowFloats, map, 0, e.g_half[g] * (HEAD / kCw), 0, e.g_row[g],
                          e.g_blk[g], &S.full[sl], policy);
          } else if (joined) {
            for (int i = 0; i < nvalid; ++i)
              bulk_copy_g2s(st + i * G::kRowFloats, e.row[i], G::kRowFloats * 4, &S.full[sl], policy);
          } else {
            for (int i = 0; i < nvalid; ++i) {
              bulk_copy_g2s(st + i * G::kRowFloats, e.row[i], HEAD * 4, &S.full[sl], policy);
              bulk_copy_g2s(st + i * G::kRowFloats + HEAD, e.row[i] + p.sw, HEAD * 4, &S.full[sl], policy);
            }
          }
        }
        j += G::kStages;
        pending = j < n;
      }
      if (__ballot_sync(0xffffffffu, pending) == 0u) break;
      const uint64_t now = global_timer_ns();
      if (__any_sync(0xffffffffu, ready)) {
        t_progress = now;
      } else {
        if (__any_sync(0xffffffffu, *abort_flag != 0) ||
            __shfl_sync(0xffffffffu, now - t_progress > kWaitTimeoutNs ? 1 : 0, 0)) {
          ok = !pending;
          break;
        }
#if C128_C4_POLL_NS > 0
        __nanosleep(C128_C4_POLL_NS);
#endif
      }
    }
    if (!__all_sync(0xffffffffu, ok)) {
      failed = true;
      break;
    }
    pass_slot = -1;
    k += static_cast<uint32_t>(n);
    mbar_arrive(&S.qempty[qs]);  // the batch's entries were copied into the stage descriptors
  }
  if (!failed) {
    // one end marker per consumer group: windows k .. k + kGroups - 1
    const uint32_t kk = k + lane;
    const int sl = kk % G::kStages;
    bool ok = true;
    if (lane < G::kGroups) {
      if (kk >= static_cast<uint32_t>(G::kStages))
        ok = mbar_wait_suspend(&S.empty[sl], ((kk / G::kStages) - 1u) & 1u, abort_flag);
      if (ok) {
        S.desc[sl].nvalid = 0;
        mbar_arrive(&S.full[sl]);
      }
    }
    failed = !__all_sync(0xffffffffu, ok);
  }
  if (failed) {
    if (lane == 0) set_timeout(p, &S.abort_flag);
    // let every copy this warp issued land before the CTA may exit: the windows of earlier batches
    // still in their stages, and this lane's last window of the batch that failed
    if (lane == 0)
      for (uint32_t j = k > static_cast<uint32_t>(G::kStages) ? k - G::kStages : 0u; j < k; ++j)
        mbar_wait(&S.full[j % G::kStages], (j / G::kStages) & 1u, nullptr);
    if (pass_slot >= 0) mbar_wait(&S.full[pass_slot], (pass_k / G::kStages) & 1u, nullptr);
    __syncwarp();
  }
}

// A window's present rows for 4 consecutive columns: score and kv quads, oldest row first.
struct WindowCols {
  float4 sc[kMaxSmallRows];
  float4 kv[kMaxSmallRows];
};

template <int HEAD>
__device__ __forceinline__ void stage_load(const float* st, int nvalid, int col, WindowCols& w) {
  constexpr int R = 2 * HEAD;
#pragma unroll
  for (int i = 0; i < kMaxSmallRows; ++i) {
    if (i < nvalid) {
      w.sc[i] = *reinterpret_cast<const float4*>(st + i * R + HEAD + col);
      w.kv[i] = *reinterpret_cast<const float4*>(st + i * R + col);
    }
  }
}

// Softmax-weighted sum over the window's present rows, column by column.
__device__ __forceinline__ float4 window_comp(const WindowCols& w, int nvalid) {
  float4 mx = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
  for (int i = 0; i < kMaxSmallRows; ++i) {
    if (i < nvalid) {
      mx.x = fmaxf(mx.x, w.sc[i].x);
      mx.y = fmaxf(mx.y, w.sc[i].y);
      mx.z = fmaxf(mx.z, w.sc[i].z);
      mx.w = fmaxf(mx.w, w.sc[i].w);
    }
  }
  const float4 bias = make_float4(mx.x * kLog2e, mx.y * kLog2e, mx.z * kLog2e, mx.w * kLog2e);
  float4 l = make_float4(0.f, 0.f, 0.f, 0.f), acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kMaxSmallRows; ++i) {
    if (i < nvalid) {
      const float4 kv = w.kv[i];
      const float ex = ex2_approx(fmaf(w.sc[i].x, kLog2e, -bias.x));
      const float ey = ex2_approx(fmaf(w.sc[i].y, kLog2e, -bias.y));
      const float ez = ex2_approx(fmaf(w.sc[i].z, kLog2e, -bias.z));
      const float ew = ex2_approx(fmaf(w.sc[i].w, kLog2e, -bias.w));
      l.x += ex;
      l.y += ey;
      l.z += ez;
      l.w += ew;
      acc.x = fmaf(ex, kv.x, acc.x);
      acc.y = fmaf(ey, kv.y, acc.y);
      acc.z = fmaf(ez, kv.z, acc.z);
      acc.w = fmaf(ew, kv.w, acc.w);
    }
  }
  return make_float4(__fdiv_rn(acc.x, l.x), __fdiv_rn(acc.y, l.y), __fdiv_rn(acc.z, l.z), __fdiv_rn(acc.w, l.w));
}

// Softmax-weighted sum of 4 consecutive columns `col` over the window's present rows, read from
// the stage as the arithmetic needs them.
template <int HEAD>
__device__ __forceinline__ float4 stage_comp(const float* st, int nvalid, int col) {
  constexpr int R = 2 * HEAD;
  float4 sc[kMaxSmallRows];
  float4 mx = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
  for (int i = 0; i < kMaxSmallRows; ++i) {
    if (i < nvalid) {
      sc[i] = *reinterpret_cast<const float4*>(st + i * R + HEAD + col);
      mx.x = fmaxf(mx.x, sc[i].x);
      mx.y = fmaxf(mx.y, sc[i].y);
      mx.z = fmaxf(mx.z, sc[i].z);
      mx.w = fmaxf(mx.w, sc[i].w);
    }
  }
  const float4 bias = make_float4(mx.x * kLog2e, mx.y * kLog2e, mx.z * kLog2e, mx.w * kLog2e);
  float4 l = make_float4(0.f, 0.f, 0.f, 0.f), acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kMaxSmallRows; ++i) {
    if (i < nvalid) {
      const float4 kv = *reinterpret_cast<const float4*>(st + i * R + col);
      const float ex = ex2_approx(fmaf(sc[i].x, kLog2e, -bias.x));
      const float ey = ex2_approx(fmaf(sc[i].y, kLog2e, -bias.y));
      const float ez = ex2_approx(fmaf(sc[i].z, kLog2e, -bias.z));
      const float ew = ex2_approx(fmaf(sc[i].w, kLog2e, -bias.w));
      l.x += ex;
      l.y += ey;
      l.z += ez;
      l.w += ew;
      acc.x = fmaf(ex, kv.x, acc.x);
      acc.y = fmaf(ey, kv.y, acc.y);
      acc.z = fmaf(ez, kv.z, acc.z);
      acc.w = fmaf(ew, kv.w, acc.w);
    }
  }
  return make_float4(__fdiv_rn(acc.x, l.x), __fdiv_rn(acc.y, l.y), __fdiv_rn(acc.z, l.z), __fdiv_rn(acc.w, l.w));
}

// ------------------------------------------------------------- head 512: a quad per window
__device__ void small_sparse_group(const Params& p, SmallSmem<512>& S, int g, int qt) {
  using G = SmallGeo<512>;
  const int qw = qt >> 5, lane = qt & 31;
  const int col = 4 * qt;
  const int bar_id = 1 + g;  // named barriers 1..kGroups
  QuadSmem& Q = S.grp[g];
  const volatile int* abort_flag = &S.abort_flag;
  const float2 wa = *reinterpret_cast<const float2*>(p.rms_w + col);
  const float2 wb = *reinterpret_cast<const float2*>(p.rms_w + col + 2);
  for (uint32_t k = g;; k += G::kGroups) {
    const int sl = k % G::kStages;
    const uint32_t par = (k / G::kStages) & 1u;
    const bool ok = mbar_wait_suspend(&S.full[sl], par, abort_flag);
    if (group_bar_or(bar_id, 128, !ok)) {
      if (qt == 0) set_timeout(p, &S.abort_flag);
      return;
    }
    const int nvalid = S.desc[sl].nvalid;
    if (nvalid == 0) return;
    if (nvalid < 0) {  // a bad block id: nothing was copied
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[sl]);
      continue;
    }
    const float4 c = stage_comp<512>(S.stage[sl], nvalid, col);
    const SmallDesc& d = S.desc[sl];
    uint8_t* tok = d.tok;
    uint8_t* scale = d.scale;
    float* comp_dst = d.comp_dst;
    // rope threads (columns 448..511): cos/sin of pairs j0, j0 + 1
    float2 cosv = make_float2(0.f, 0.f), sinv = make_float2(0.f, 0.f);
    if (col >= kNope) {
      const int j0 = (col - kNope) / 2;
      const float* cs = d.cs_row;
      cosv = make_float2(__ldg(cs + j0), __ldg(cs + j0 + 1));
      sinv = make_float2(__ldg(cs + kRope / 2 + j0), __ldg(cs + kRope / 2 + j0 + 1));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[sl]);  // stage and descriptor are free again

    if (comp_dst != nullptr) *reinterpret_cast<float4*>(comp_dst + col) = c;
    *reinterpret_cast<float4*>(&Q.comp[col]) = c;
    const uint32_t u[4] = {__float_as_uint(c.x) & 0x7fffffffu, __float_as_uint(c.y) & 0x7fffffffu,
                           __float_as_uint(c.z) & 0x7fffffffu, __float_as_uint(c.w) & 0x7fffffffu};
    const uint32_t em_w = __reduce_max_sync(0xffffffffu, max(max(biased_exp(u[0]), biased_exp(u[1])),
                                                             max(biased_exp(u[2]), biased_exp(u[3]))));
    const uint32_t sp_w = __reduce_or_sync(0xffffffffu, special_bits(u[0]) | special_bits(u[1]) |
                                                            special_bits(u[2]) | special_bits(u[3]));
    if (lane == 0) {
      Q.emax[qw] = em_w;
      Q.special[qw] = sp_w;
    }
    group_bar(bar_id, 128);
    const uint32_t emax = max(max(Q.emax[0], Q.emax[1]), max(Q.emax[2], Q.emax[3]));
    const uint32_t special = Q.special[0] | Q.special[1] | Q.special[2] | Q.special[3];
    unsigned long long lo = 0ull, hi = 0ull;
    bool fb = false;
    if (special == 0u)
      for (int j = 0; j < 4; ++j) add_square(u[j], emax, lo, hi, fb);
    warp_sum128(lo, hi);
    fb = __any_sync(0xffffffffu, fb);
    if (lane == 0) {
      Q.lo[qw] = lo;
      Q.hi[qw] = hi;
      Q.fb[qw] = fb;
    }
    group_bar(bar_id, 128);
    if (qt == 0) {
      unsigned long long vlo = 0ull, vhi = 0ull;
      for (int j = 0; j < 4; ++j) {
        const unsigned long long nlo = vlo + Q.lo[j];
        vhi += Q.hi[j] + (nlo < vlo ? 1ull : 0ull);
        vlo = nlo;
      }
      float var;
      if (special & 2u) var = __int_as_float(0x7fc00000);
      else if (special & 1u) var = INFINITY;
      else if (Q.fb[0] | Q.fb[1] | Q.fb[2] | Q.fb[3]) var = mean_square_exact_slow(Q.comp, 512, 9);
      else var = round_u128_to_f32(vlo, vhi, 2 * static_cast<int>(emax) - 373, false);
      Q.rrms = __frsqrt_rn(__fadd_rn(var, p.eps));
    }
    group_bar(bar_id, 128);
    const float rrms = Q.rrms;
    const float nv[4] = {__fmul_rn(__fmul_rn(c.x, rrms), wa.x), __fmul_rn(__fmul_rn(c.y, rrms), wa.y),
                         __fmul_rn(__fmul_rn(c.z, rrms), wb.x), __fmul_rn(__fmul_rn(c.w, rrms), wb.y)};
    const int blk = col / kQuantBlock;  // 0..7; half-warp h = lanes 16h..16h+15 of warp qw is block 2qw+h
    if (blk < kNope / kQuantBlock) {
      const uint32_t b01 = pack_bf16x2(nv[0], nv[1]), b23 = pack_bf16x2(nv[2], nv[3]);
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
      for (int j = 0; j < 4; ++j) y[j] = fminf(fmaxf(__fmul_rn(x[j], inv), -448.f), 448.f);
      *reinterpret_cast<uint32_t*>(tok + col) =
          static_cast<uint32_t>(pack_e4m3x2(y[0], y[1])) | (static_cast<uint32_t>(pack_e4m3x2(y[2], y[3])) << 16);
      if ((col & (kQuantBlock - 1)) == 0) scale[blk] = static_cast<uint8_t>(min(max(e + 127, 0), 255));
    } else {
      // rope: pairs (448 + 2j, 449 + 2j), j = (col - 448) / 2 + k
      uint32_t out[2];
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        const float C = j2 ? cosv.y : cosv.x, Sn = j2 ? sinv.y : sinv.x;
        const float ev = nv[2 * j2], od = nv[2 * j2 + 1];
        out[j2] = pack_bf16x2(__fsub_rn(__fmul_rn(ev, C), __fmul_rn(od, Sn)), __fadd_rn(__fmul_rn(od, C), __fmul_rn(ev, Sn)));
      }
      *reinterpret_cast<uint2*>(tok + kNope + 2 * (col - kNope)) = make_uint2(out[0], out[1]);
      if (col == kNope) scale[kNope / kQuantBlock] = 0;
    }
  }
}

// ----------------------------------------------------------------- head 128: a warp per window
template <int FMT>
__device__ void small_indexer_warp(const Params& p, SmallSmem<128>& S, int w, int lane) {
  using G = SmallGeo<128>;
  const int col = 4 * lane;
  float* comp_s = S.grp[w].comp;
  const volatile int* abort_flag = &S.abort_flag;
  const float2 wa = *reinterpret_cast<const float2*>(p.rms_w + col);
  const float2 wb = *reinterpret_cast<const float2*>(p.rms_w + col + 2);
  for (uint32_t k = w;; k += G::kGroups) {
    const int sl = k % G::kStages;
    const uint32_t par = (k / G::kStages) & 1u;
    const bool ok = mbar_wait_suspend(&S.full[sl], par, abort_flag);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) set_timeout(p, &S.abort_flag);
      return;
    }
    const int nvalid = S.desc[sl].nvalid;
    if (nvalid == 0) return;
    if (nvalid < 0) {  // a bad block id: nothing was copied
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[sl]);
      continue;
    }
    const SmallDesc& d = S.desc[sl];
    uint8_t* tok = d.tok;
    uint8_t* scale = d.scale;
    float* comp_dst = d.comp_dst;
    // pairs j = 2*lane, 2*lane + 1; pairs >= 32 (lanes 16..31) rotate, the others use cos 1, sin 0.
    // The cos/sin loads go out first and land while the window is folded.
    float2 cosv = make_float2(1.f, 1.f), sinv = make_float2(0.f, 0.f);
    if (lane >= 16) {
      const int j0 = 2 * lane - 32;
      const float* cs = d.cs_row;
      cosv = make_float2(__ldg(cs + j0), __ldg(cs + j0 + 1));
      sinv = make_float2(__ldg(cs + kRope / 2 + j0), __ldg(cs + kRope / 2 + j0 + 1));
    }
    // the window's rows go to registers and the stage is released before the arithmetic, so the
    // copier can refill it while this warp folds the window and runs the epilogue
    WindowCols wc;
    stage_load<128>(S.stage[sl], nvalid, col, wc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[sl]);
    const float4 c = window_comp(wc, nvalid);

    indexer_warp_epilogue<FMT>(c, lane, wa, wb, p.eps, cosv, sinv, tok, scale, comp_dst, comp_s);
  }
}

// ------------------------------------------------------------------------------------ kernel
template <int HEAD, int FMT>
__global__ void __launch_bounds__(SmallGeo<HEAD>::kThreads, 1)
    small_window_kernel(Params p, const __grid_constant__ CUtensorMap state_map, int flags) {
  using G = SmallGeo<HEAD>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SmallSmem<HEAD>& S = *reinterpret_cast<SmallSmem<HEAD>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // A programmatic dependent of the kernel before it on the stream (with token striding the
  // previous call's kernel or whatever precedes the call, on the planned path the planning pass,
  // which itself waits for the kernel before it): nothing global is touched before that kernel has
  // completed (the barriers, in shared memory, are set up while it runs). The next launch may
  // start as soon as every CTA of this one runs.
  launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], G::kGroupWarps);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&S.qfull[q], 32);
      mbar_init(&S.qempty[q], 32);
    }
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  grid_dependency_wait();
  // tiled loads need 128-byte aligned destinations (every stage offset is a multiple of 1 KiB)
  const bool use_tiled = (flags & kFlagTiled) != 0 && (smem_addr(smem_raw) & 127u) == 0u;
  if (warp == 0) {
    small_scheduler<HEAD, FMT>(p, S, lane, use_tiled);
  } else if (warp == 1) {
    small_copier<HEAD>(p, S, lane, &state_map, use_tiled);
  } else if constexpr (HEAD == 512) {
    const int ct = tid - 64;
    small_sparse_group(p, S, ct >> 7, ct & 127);
  } else {
    small_indexer_warp<FMT>(p, S, warp - 2, lane);
  }
}

template <int HEAD, int FMT>
cudaError_t launch_small_kernel(const Params& p, const LaunchCfg& cfg, cudaStream_t stream) {
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  const int flags = encode_state_map(p, HEAD, p.ratio, &map) ? kFlagTiled : 0;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(cfg.sm_count));  // one persistent CTA per SM
  lc.blockDim = dim3(SmallGeo<HEAD>::kThreads);
  lc.dynamicSmemBytes = sizeof(SmallSmem<HEAD>);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = (cfg.pdl && cfg.ev_begin == nullptr) ? 1 : 0;
  return cudaLaunchKernelEx(&lc, small_window_kernel<HEAD, FMT>, p, map, flags);
}

}  // namespace

// The state cache as a 5-D tensor for tiled loads of `box_rows` consecutive rows of one state
// block, innermost first: cw columns (cw = min(head, 256)), chunks of cw columns within the kv
// (or score) part of a row, kv / score part, row within a state block, state block. The box takes
// head columns of kv and of score for each of its rows. False when the layout does not fit such a
// map (the caller then uses per-row bulk copies or another kernel).
namespace {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}
}  // namespace

bool encode_state_map(const Params& p, int head, int box_rows, CUtensorMap* map) {
  const int cw = head < 256 ? head : 256;
  if (box_rows < 1 || box_rows > 256 || p.sblk % box_rows != 0 || p.sw < (1 + p.overlap) * head) return false;
  if (p.nb > (1ll << 31) || p.sblk > (1ll << 31)) return false;
  const uint64_t s1 = static_cast<uint64_t>(p.s1) * 4, s0 = static_cast<uint64_t>(p.s0) * 4;
  if (s1 >= (1ull << 40) || s0 >= (1ull << 40) || s1 < static_cast<uint64_t>(2 * p.sw) * 4) return false;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(cw), static_cast<cuuint64_t>(p.sw / cw), 2,
                              static_cast<cuuint64_t>(p.sblk), static_cast<cuuint64_t>(p.nb)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(cw) * 4, static_cast<cuuint64_t>(p.sw) * 4, s1, s0};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(cw), static_cast<cuuint32_t>(head / cw), 2,
                             static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, const_cast<float*>(p.state), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool small_window_path(const Params& p) { return (1 + p.overlap) * p.ratio <= kMaxSmallRows; }

cudaError_t prepare_small() {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(small_window_kernel<512, C128_FORMAT_SPARSE_FP8>, a,
                                       static_cast<int>(sizeof(SmallSmem<512>)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(small_window_kernel<128, C128_FORMAT_INDEXER_FP8>, a,
                             static_cast<int>(sizeof(SmallSmem<128>)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(small_window_kernel<128, C128_FORMAT_INDEXER_MXFP4>, a,
                             static_cast<int>(sizeof(SmallSmem<128>)));
  return e;
}

cudaError_t launch_small(const Params& p, const LaunchCfg& cfg, cudaStream_t stream) {
  if (p.fmt == C128_FORMAT_SPARSE_FP8) return launch_small_kernel<512, C128_FORMAT_SPARSE_FP8>(p, cfg, stream);
  if (p.fmt == C128_FORMAT_INDEXER_FP8) return launch_small_kernel<128, C128_FORMAT_INDEXER_FP8>(p, cfg, stream);
  return launch_small_kernel<128, C128_FORMAT_INDEXER_MXFP4>(p, cfg, stream);
}

}  // namespace c128
