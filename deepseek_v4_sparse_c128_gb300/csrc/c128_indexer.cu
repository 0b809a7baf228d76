// sm_103a kernel for head-128 windows of more than 8 rows (the indexer compressor at compress
// ratio 128, and any ratio >= 8 whose windows exceed 8 rows): a persistent CTA per SM streams one
// window at a time through a ring of 32 KiB shared-memory stages.
//
//   warp 0       scheduler: claims the next window, resolves the token's request, position and
//                cache slot and, one lane per chunk of 8 rows, the chunk's state block, checks
//                them and writes a window descriptor (two in flight).
//   warp 1       copier (lane 0): per stage, up to 4 tiled TMA loads (`cp.async.bulk.tensor.5d`)
//                of 8 rows each; the box takes the kv half-row and the score half-row of every
//                row (the older or the newer half of an overlapping window). Completion is
//                counted in bytes on the stage's mbarrier.
//   warps 2..9   consumers: row group g (two warps, thread i owns columns 2i, 2i+1) folds chunk g
//                of every stage into an online softmax; after the window's last stage they write
//                the four row groups' partial states (double-buffered) and go on with the next
//                window.
//   warp 10      epilogue: merges the partial states in row-group order and runs the indexer
//                epilogue (RMSNorm, RoPE, FP8 or MXFP4 cache store), so no consumer waits for it.
//
// Same arithmetic as the oracle's reading of _fused_kv_compress_norm_rope_insert_indexer_attn and
// ..._indexer_mxfp4_attn on the API page of vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache.
#include <cuda.h>

#include <cstddef>

#include "c128_device.cuh"
#include "c128_warp_epilogue.cuh"

namespace c128 {
namespace {

constexpr int kIxHead = 128;
constexpr int kIxChunk = 8;                                            // rows per tiled load
constexpr int kIxStageChunks = 4;                                      // 32 rows per stage
constexpr int kIxStages = 6;
constexpr int kIxMaxChunks = 32;                                       // windows of up to 256 rows
constexpr int kIxRowFloats = 2 * kIxHead;                              // kv half-row | score half-row
constexpr int kIxChunkFloats = kIxChunk * kIxRowFloats;                // 8 KiB
constexpr int kIxStageFloats = kIxStageChunks * kIxChunkFloats;        // 32 KiB
constexpr int kIxConsumerWarps = 8;
constexpr int kIxConsumerThreads = 32 * kIxConsumerWarps;
constexpr int kIxThreads = 32 * (3 + kIxConsumerWarps);                // + the epilogue warp
constexpr int kIxRowGroups = kIxStageChunks;                           // row group g takes chunk g of a stage
#ifndef C128_IX_DESC_SLOTS
#define C128_IX_DESC_SLOTS 2
#endif
constexpr int kIxDescSlots = C128_IX_DESC_SLOTS;
static_assert(kIxRowGroups * kIxHead / 2 == kIxConsumerThreads, "two columns per consumer thread");

struct __align__(16) IxDesc {
  int32_t blk[kIxMaxChunks];   // state block of each present chunk, oldest first
  int32_t row[kIxMaxChunks];   // the chunk's first row within its block
  int32_t half[kIxMaxChunks];  // 0: older half of an overlapping window (or no overlap), 1: newer half
  uint8_t* tok;                // token bytes of the cache slot
  uint8_t* scale;              // scale bytes of the slot
  const float* cs_row;         // cos/sin row (p / ratio) * ratio
  float* comp_dst;             // optional fp32 export
  int32_t nchunks;             // chunks present; 0 marks the end of the work
  int32_t pad[3];
};

struct IxSmem {
  float stage[kIxStages][kIxStageFloats];
  IxDesc desc[kIxDescSlots];
  uint64_t full[kIxStages];       // stage landed (1 arrival + its bytes)
  uint64_t empty[kIxStages];      // stage consumed (one arrival per consumer warp)
  uint64_t dfull[kIxDescSlots];   // descriptor written (scheduler)
  uint64_t dempty[kIxDescSlots];  // descriptor released (copier + consumer warps)
  // row-group partial states (log2-unit max, sum, weighted sum), double-buffered by window parity
  alignas(16) float part_m[2][kIxRowGroups][kIxHead];
  alignas(16) float part_l[2][kIxRowGroups][kIxHead];
  alignas(16) float part_a[2][kIxRowGroups][kIxHead];
  alignas(16) float comp_s[kIxHead];  // exact-variance slow path of the epilogue warp (float4 stores)
  struct PartMeta {
    uint8_t* tok;
    uint8_t* scale;
    const float* cs_row;
    float* comp_dst;
    int32_t end;  // no more windows
    int32_t pad[3];
  } meta[2];
  uint64_t pfull[2];   // a window's partials written (one arrival per consumer warp)
  uint64_t pempty[2];  // the epilogue warp is done with them (one arrival)
  uint32_t chunk_prefix[kMaxPlanChunks + 1];  // planned path: active windows before each chunk
  int abort_flag;
};
static_assert(sizeof(IxSmem) <= 227 * 1024, "shared memory");
static_assert(sizeof(float) * kIxStageFloats % 128 == 0 && sizeof(float) * kIxChunkFloats % 128 == 0,
              "tiled-load destinations stay 128-byte aligned");

__device__ __forceinline__ void ix_set_timeout(const Params& p, int* abort_flag) {
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
  atomicOr(&p.ws->err, static_cast<unsigned>(C128_DEV_TIMEOUT));
}

__device__ __forceinline__ void ix_tma_load(void* dst, const CUtensorMap* map, int half, int row, int blk,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(half), "r"(0), "r"(row), "r"(blk), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

// ------------------------------------------------------------------------------ scheduler warp
template <int FMT, bool STRIDED>
__device__ void ix_scheduler(const Params& p, IxSmem& S, int lane) {
  constexpr int kTok = FMT == C128_FORMAT_INDEXER_FP8 ? 128 : 64;
  // list mode: windows from plan_kernel's list; token striding (few tokens, no planning pass):
  // this CTA tests tokens c, c + grid, ..., 32 candidates per step. The mode is a template
  // parameter: with a run-time branch on it here, list-mode calls ran about 8 % slower.
  constexpr bool strided = STRIDED;
  const volatile int* abort_flag = &S.abort_flag;
  // planned path (the kernel entry waited for the planning pass): the list's windows
  const uint32_t A = strided ? 0u : plan_prefix_warp(p, S.chunk_prefix, lane);
  int64_t next_t = blockIdx.x;
  const int n = (1 + p.overlap) * p.ratio;  // 16..256 rows, a multiple of 8
  uint32_t widx = 0;
  bool first_claim = true;
  for (;;) {
    if (*abort_flag) return;
    bool end;
    long long t = 0, pos = 0, kvs = 0;
    if (strided) {
      long long found = -1;
      while (found < 0 && next_t < p.T) {
        const int64_t c = next_t + static_cast<int64_t>(lane) * gridDim.x;
        bool act = false;
        if (c < p.T) {
          const int64_t sl = __ldg(p.slot + c), ps = __ldg(p.pos + c), kv = __ldg(p.kvslot + c);
          act = (sl >= 0) & (ps >= 0) & (((ps + 1) & (p.ratio - 1)) == 0) & (kv >= 0);
        }
        const uint32_t m = __ballot_sync(0xffffffffu, act);
        if (m) {
          found = next_t + static_cast<int64_t>(__ffs(m) - 1) * gridDim.x;
          next_t = found + gridDim.x;
        } else {
          next_t += 32ll * gridDim.x;
        }
      }
      end = found < 0;
      t = found;
    } else {
      // the first window of CTA c is window c; later ones come from the shared counter
      uint32_t a = 0;
      if (lane == 0) a = first_claim ? blockIdx.x : gridDim.x + atomicAdd(&p.ws->next, 1u);
      a = __shfl_sync(0xffffffffu, a, 0);
      first_claim = false;
      end = a >= A;
      if (!end && lane == 0) t = plan_token(p, S.chunk_prefix, a);
    }
    int req = 0;
    uint32_t err = 0;
    if (!end) {
      if (lane == 0) {
        req = __ldg(p.ttr + t);
        pos = __ldg(p.pos + t);
        kvs = __ldg(p.kvslot + t);
        if (req < 0 || req >= p.bt_rows) err |= C128_DEV_BAD_REQ;
        if (pos / p.sblk >= p.bt_cols) err |= C128_DEV_BAD_BT_COL;
        if ((pos & ~static_cast<long long>(p.ratio - 1)) >= p.cs_rows) err |= C128_DEV_BAD_COS_ROW;
        if (kvs >= p.nkb * p.kv_bs) err |= C128_DEV_BAD_KV_SLOT;
      }
      t = __shfl_sync(0xffffffffu, t, 0);
      req = __shfl_sync(0xffffffffu, req, 0);
      pos = __shfl_sync(0xffffffffu, pos, 0);
      kvs = __shfl_sync(0xffffffffu, kvs, 0);
      err = __shfl_sync(0xffffffffu, err, 0);
    }
    // window rows start .. pos; start and 0 are multiples of 8, so masked rows fill whole chunks
    const long long start = pos - n + 1, first = start > 0 ? start : 0;
    const int nch = end ? 0 : static_cast<int>((pos - first + 1) / kIxChunk);
    int blk = 0, row = 0, half = 0;
    if (!end && !(err & (C128_DEV_BAD_REQ | C128_DEV_BAD_BT_COL))) {
      bool bad = false;
      if (lane < nch) {
        const long long q0 = first + static_cast<long long>(kIxChunk) * lane;
        blk = __ldg(p.bt + static_cast<int64_t>(req) * p.bt_stride + q0 / p.sblk);
        row = static_cast<int>(q0 % p.sblk);
        half = (p.overlap && q0 - start >= p.ratio) ? 1 : 0;
        bad = blk < 0 || blk >= p.nb;
      }
      if (__any_sync(0xffffffffu, bad)) err |= C128_DEV_BAD_BLOCK;
    }
    if (!end && err) {
      if (lane == 0) atomicOr(&p.ws->err, err);
      continue;
    }
    const int ds = widx % kIxDescSlots;
    if (widx >= kIxDescSlots) {
      bool ok = mbar_wait_suspend(&S.dempty[ds], ((widx / kIxDescSlots) - 1u) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) ix_set_timeout(p, &S.abort_flag);
        return;
      }
    }
    IxDesc& d = S.desc[ds];
    if (lane < nch) {
      d.blk[lane] = blk;
      d.row[lane] = row;
      d.half[lane] = half;
    }
    if (lane == 0) {
      if (!end) {
        const long long kb = kvs / p.kv_bs, off = kvs - kb * p.kv_bs;
        uint8_t* base = p.kc + kb * p.kc_stride0;
        d.tok = base + off * kTok;
        d.scale = base + p.kv_bs * kTok + off * 4;
        d.cs_row = p.cs + (pos & ~static_cast<long long>(p.ratio - 1)) * p.cs_stride;
        d.comp_dst = p.comp_out ? p.comp_out + t * kIxHead : nullptr;
      }
      d.nchunks = nch;
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      mbar_arrive(&S.dfull[ds]);
    }
    ++widx;
    if (end) return;
  }
}

// --------------------------------------------------------------------------------- copier thread
__device__ void ix_copier(const Params& p, IxSmem& S, const CUtensorMap* map) {
  const volatile int* abort_flag = &S.abort_flag;
  const uint64_t policy = l2_evict_first_policy();
  // rows of kv[128] | score[128] one after the other: an 8-row chunk is one contiguous 8 KiB range
  const bool linear = p.sw == kIxHead && p.s1 == kIxRowFloats;
  uint32_t it = 0, widx = 0;
  bool failed = false;
  for (;;) {
    const int ds = widx % kIxDescSlots;
    if (!mbar_wait_suspend(&S.dfull[ds], (widx / kIxDescSlots) & 1u, abort_flag)) {
      failed = true;
      break;
    }
    const IxDesc& d = S.desc[ds];
    const int nch = d.nchunks;
    if (nch == 0) break;
    for (int c0 = 0; c0 < nch; c0 += kIxStageChunks) {
      const int s = it % kIxStages;
      const uint32_t round = it / kIxStages;
      if (round > 0 && !mbar_wait_suspend(&S.empty[s], (round - 1u) & 1u, abort_flag)) {
        failed = true;
        break;
      }
      const int cnt = min(kIxStageChunks, nch - c0);
      mbar_arrive_expect_tx(&S.full[s], static_cast<uint32_t>(cnt * kIxChunkFloats * 4));
      // test of the bounded waits: CTA 0's first stage never fills
      const int issue = p.stall_first_window && blockIdx.x == 0 && it == 0 ? 0 : cnt;
      for (int j = 0; j < issue; ++j) {
        if (linear)
          bulk_copy_g2s(S.stage[s] + j * kIxChunkFloats,
                        p.state + static_cast<int64_t>(d.blk[c0 + j]) * p.s0 + static_cast<int64_t>(d.row[c0 + j]) * p.s1,
                        kIxChunkFloats * 4, &S.full[s], policy);
        else
          ix_tma_load(S.stage[s] + j * kIxChunkFloats, map, d.half[c0 + j], d.row[c0 + j], d.blk[c0 + j], &S.full[s],
                      policy);
      }
      ++it;
    }
    if (failed) break;
    mbar_arrive(&S.dempty[ds]);
    ++widx;
  }
  if (failed) {
    ix_set_timeout(p, &S.abort_flag);
    // let every copy this thread issued land before the CTA may exit
    for (uint32_t i = it > static_cast<uint32_t>(kIxStages) ? it - kIxStages : 0u; i < it; ++i)
      mbar_wait(&S.full[i % kIxStages], (i / kIxStages) & 1u, nullptr);
  }
}

// ------------------------------------------------------------------------------ consumer warps
// The 8 rows of one staged chunk for columns c0, c0 + 1: kv and score pairs.
struct ChunkRows {
  float2 kv[kIxChunk], sc[kIxChunk];
};
__device__ __forceinline__ void ix_load_chunk(const float* st, int c0, ChunkRows& cr) {
#pragma unroll
  for (int r = 0; r < kIxChunk; ++r) {
    cr.kv[r] = *reinterpret_cast<const float2*>(st + r * kIxRowFloats + c0);
    cr.sc[r] = *reinterpret_cast<const float2*>(st + r * kIxRowFloats + kIxHead + c0);
  }
}
// Fold those rows into the online state of columns c0, c0 + 1.
__device__ __forceinline__ void ix_fold_chunk(const ChunkRows& cr, Online& o) {
  const float2* kv = cr.kv;
  const float2* sc = cr.sc;
  float mx0 = sc[0].x, mx1 = sc[0].y;
#pragma unroll
  for (int r = 1; r < kIxChunk; ++r) {
    mx0 = fmaxf(mx0, sc[r].x);
    mx1 = fmaxf(mx1, sc[r].y);
  }
  const float n0 = fmaxf(o.m0, mx0 * kLog2e), n1 = fmaxf(o.m1, mx1 * kLog2e);
  const float b0 = n0 == -INFINITY ? 0.f : n0, b1 = n1 == -INFINITY ? 0.f : n1;
  const float r0 = ex2_approx(o.m0 - b0), r1 = ex2_approx(o.m1 - b1);
  o.m0 = n0;
  o.m1 = n1;
  float ps0 = 0.f, ps1 = 0.f, pk0 = 0.f, pk1 = 0.f;
#pragma unroll
  for (int r = 0; r < kIxChunk; ++r) {
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

template <int FMT>
__device__ void ix_consumers(const Params& p, IxSmem& S, int ci) {
  const int lane = ci & 31;
  const int rg = ci / (kIxHead / 2);     // row group: chunk rg of every stage
  const int c0 = 2 * (ci % (kIxHead / 2));
  const volatile int* abort_flag = &S.abort_flag;
  uint32_t it = 0, widx = 0;
  for (;;) {
    const int ds = widx % kIxDescSlots;
    const bool got = mbar_wait_suspend(&S.dfull[ds], (widx / kIxDescSlots) & 1u, abort_flag);
    int nch = 0;
    uint8_t* tok = nullptr;
    uint8_t* scale = nullptr;
    const float* cs_row = nullptr;
    float* comp_dst = nullptr;
    if (got) {
      const IxDesc& d = S.desc[ds];
      nch = d.nchunks;
      tok = d.tok;
      scale = d.scale;
      cs_row = d.cs_row;
      comp_dst = d.comp_dst;
    } else {
      ix_set_timeout(p, &S.abort_flag);
    }
    if (consumer_bar_or(!got || nch == 0 || *abort_flag)) {
      // a clean end (every consumer saw the end marker, nothing aborted): tell the epilogue warp,
      // through the next partials buffer, that no window follows
      if (!consumer_bar_or(!got || *abort_flag)) {
        const int pb = widx & 1;
        const bool free_ok = __all_sync(
            0xffffffffu, widx < 2 || mbar_wait_suspend(&S.pempty[pb], ((widx >> 1) - 1u) & 1u, abort_flag));
        if (free_ok) {
          if (ci == 0) S.meta[pb].end = 1;
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.pfull[pb]);
        } else if (lane == 0) {
          ix_set_timeout(p, &S.abort_flag);
        }
      }
      return;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.dempty[ds]);  // the fields above are in registers

    Online o;
    online_init(o);
    bool failed = false;
    for (int cs0 = 0; cs0 < nch; cs0 += kIxStageChunks) {
      const int s = it % kIxStages;
      bool ok = !failed && mbar_wait_suspend(&S.full[s], (it / kIxStages) & 1u, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        // the rows go to registers and the stage is released before the arithmetic, so the copier
        // can refill it while the warp folds the chunk
        const bool mine = cs0 + rg < nch;
        ChunkRows cr;
        if (mine) ix_load_chunk(S.stage[s] + rg * kIxChunkFloats, c0, cr);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[s]);
        if (mine) ix_fold_chunk(cr, o);
      } else {
        failed = true;
      }
      ++it;
    }
    if (failed) ix_set_timeout(p, &S.abort_flag);
    // hand the partial states to the epilogue warp (buffer widx & 1, free once it took window widx - 2)
    const int pb = widx & 1;
    bool free_ok = widx < 2 || mbar_wait_suspend(&S.pempty[pb], ((widx >> 1) - 1u) & 1u, abort_flag);
    if (consumer_bar_or(failed || !free_ok)) {
      if (!free_ok) ix_set_timeout(p, &S.abort_flag);
      return;
    }
    *reinterpret_cast<float2*>(&S.part_m[pb][rg][c0]) = make_float2(o.m0, o.m1);
    *reinterpret_cast<float2*>(&S.part_l[pb][rg][c0]) = make_float2(o.l0, o.l1);
    *reinterpret_cast<float2*>(&S.part_a[pb][rg][c0]) = make_float2(o.a0, o.a1);
    if (ci == 0) S.meta[pb] = IxSmem::PartMeta{tok, scale, cs_row, comp_dst, 0, {0, 0, 0}};
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.pfull[pb]);
    ++widx;
  }
}

// ------------------------------------------------------------------------------- epilogue warp
template <int FMT>
__device__ void ix_epilogue_warp(const Params& p, IxSmem& S, int lane) {
  const volatile int* abort_flag = &S.abort_flag;
  const float2 wa = *reinterpret_cast<const float2*>(p.rms_w + 4 * lane);  // lane l owns columns 4l..4l+3
  const float2 wb = *reinterpret_cast<const float2*>(p.rms_w + 4 * lane + 2);
  for (uint32_t widx = 0;; ++widx) {
    const int pb = widx & 1;
    const bool ok = mbar_wait_suspend(&S.pfull[pb], (widx >> 1) & 1u, abort_flag);
    if (!__all_sync(0xffffffffu, ok)) return;  // the consumers stopped (a timeout already reported)
    const IxSmem::PartMeta m = S.meta[pb];
    if (m.end) return;
    float2 cosv = make_float2(1.f, 1.f), sinv = make_float2(0.f, 0.f);
    if (lane >= 16) {  // pairs 2l, 2l + 1 >= 32 rotate
      const int j0 = 2 * lane - 32;
      cosv = make_float2(__ldg(m.cs_row + j0), __ldg(m.cs_row + j0 + 1));
      sinv = make_float2(__ldg(m.cs_row + kRope / 2 + j0), __ldg(m.cs_row + kRope / 2 + j0 + 1));
    }
    // merge the row groups in order, columns 4l..4l+3
    float out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = 4 * lane + j;
      float M = S.part_m[pb][0][col];
#pragma unroll
      for (int g = 1; g < kIxRowGroups; ++g) M = fmaxf(M, S.part_m[pb][g][col]);
      const float B = M == -INFINITY ? 0.f : M;
      float L = 0.f, Acc = 0.f;
#pragma unroll
      for (int g = 0; g < kIxRowGroups; ++g) {
        const float sc = ex2_approx(S.part_m[pb][g][col] - B);
        L = fmaf(S.part_l[pb][g][col], sc, L);
        Acc = fmaf(S.part_a[pb][g][col], sc, Acc);
      }
      out[j] = __fdiv_rn(Acc, L);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.pempty[pb]);  // the partials are in registers
    indexer_warp_epilogue<FMT>(make_float4(out[0], out[1], out[2], out[3]), lane, wa, wb, p.eps, cosv, sinv, m.tok,
                               m.scale, m.comp_dst, S.comp_s);
  }
}

template <int FMT>
__global__ void __launch_bounds__(kIxThreads, 1)
    indexer_window_kernel(Params p, const __grid_constant__ CUtensorMap state_map) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  IxSmem& S = *reinterpret_cast<IxSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // A programmatic dependent of the kernel before it on the stream (with token striding the
  // previous call's kernel or whatever precedes the call, on the planned path the planning pass,
  // which itself waits for the kernel before it): nothing global is touched before that kernel has
  // completed (the barriers, in shared memory, are set up while it runs). The next launch may
  // start as soon as every CTA of this one runs.
  launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kIxStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kIxConsumerWarps);
    }
    for (int d = 0; d < kIxDescSlots; ++d) {
      mbar_init(&S.dfull[d], 1);
      mbar_init(&S.dempty[d], kIxConsumerWarps + 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.pfull[b], kIxConsumerWarps);
      mbar_init(&S.pempty[b], 1);
    }
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  grid_dependency_wait();
  if (warp == 0) {
    if (p.strided)
      ix_scheduler<FMT, true>(p, S, lane);
    else
      ix_scheduler<FMT, false>(p, S, lane);
  } else if (warp == 1) {
    if (lane == 0) ix_copier(p, S, &state_map);
  } else {
    if (warp < 2 + kIxConsumerWarps)
      ix_consumers<FMT>(p, S, tid - 64);
    else
      ix_epilogue_warp<FMT>(p, S, lane);
  }
}

}  // namespace

cudaError_t prepare_indexer_windows() {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(indexer_window_kernel<C128_FORMAT_INDEXER_FP8>, a, static_cast<int>(sizeof(IxSmem)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(indexer_window_kernel<C128_FORMAT_INDEXER_MXFP4>, a, static_cast<int>(sizeof(IxSmem)));
  return e;
}

cudaError_t launch_indexer_windows(const Params& p, const LaunchCfg& cfg, cudaStream_t stream) {
  const int n = (1 + p.overlap) * p.ratio;
  if (p.head != kIxHead || p.fmt == C128_FORMAT_SPARSE_FP8 || n <= 8 || n > kIxChunk * kIxMaxChunks ||
      p.ratio % kIxChunk != 0)
    return cudaErrorNotSupported;
  CUtensorMap map;
  if (!encode_state_map(p, kIxHead, kIxChunk, &map)) return cudaErrorNotSupported;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(cfg.sm_count));  // one persistent CTA per SM
  lc.blockDim = dim3(kIxThreads);
  lc.dynamicSmemBytes = sizeof(IxSmem);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = (cfg.pdl && cfg.ev_begin == nullptr) ? 1 : 0;
  if (p.fmt == C128_FORMAT_INDEXER_FP8)
    return cudaLaunchKernelEx(&lc, indexer_window_kernel<C128_FORMAT_INDEXER_FP8>, p, map);
  return cudaLaunchKernelEx(&lc, indexer_window_kernel<C128_FORMAT_INDEXER_MXFP4>, p, map);
}

}  // namespace c128
