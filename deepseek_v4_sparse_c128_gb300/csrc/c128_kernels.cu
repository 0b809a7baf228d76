// sm_103a kernels of the DeepSeek-V4 C128 KV compressor.
//
//   plan_chunks_kernel  the planning pass: per chunk of 2048 tokens, the indices of its active
//                    tokens (slot >= 0, position at a window end, kv slot >= 0) in token order and
//                    their number; plan_kernel compacts them into one list instead (above 1 Mi
//                    tokens).
//   direct_kernel    one token per cluster of S CTAs, no planning pass: S in {8, 4, 2, 1} while
//                    token_num x S fits the SMs in one wave (the window split over the cluster,
//                    merged over distributed shared memory), then up to 8 tokens per SM one CTA
//                    per token with a 3-stage ring, two CTAs per SM.
//   compress_kernel  above that: persistent, one CTA per SM. Warp 0 claims windows from the list and resolves
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
#include "c128_device.cuh"

namespace c128 {
namespace {
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
      const bool active = (s >= 0) & (pos >= 0) & (((pos + 1) & (p.ratio - 1)) == 0) & (kv >= 0);
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

// C128 planning pass: CTA c takes tokens [c * 2048, (c + 1) * 2048), writes its active tokens in
// token order at list[c * 2048 ...] and their number at list[T + c], and CTA 0 zeroes the claim
// counter. Every word it writes is overwritten by each call, so no zeroing pass precedes it, and
// the list order does not depend on which CTA finishes first. It is launched as a programmatic
// dependent of the kernel before it (the previous call's compress kernel still reads the list and
// the claim counter until it completes): it waits for that kernel before any global access.
// THREADS threads per CTA (256 or 512), kPlanTokensPerCta / THREADS tokens each.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) plan_chunks_kernel(Params p) {
  constexpr int kTok = kPlanTokensPerCta / THREADS;
  static_assert(kTok * THREADS == kPlanTokensPerCta && kTok <= 32, "whole chunks, one flag bit per token");
  launch_dependents();
  grid_dependency_wait();
  __shared__ uint32_t warp_base[THREADS / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kPlanTokensPerCta;
  if (blockIdx.x == 0 && tid == 0) p.ws->next = 0u;
  // thread tid takes tokens base + kTok tid .. + kTok - 1, so that the list comes out in token order
  uint32_t flags = 0;
#pragma unroll
  for (int i = 0; i < kTok; ++i) {
    const int64_t t = base + static_cast<int64_t>(tid) * kTok + i;
    if (t < p.T) {
      const int64_t s = __ldg(p.slot + t), pos = __ldg(p.pos + t), kv = __ldg(p.kvslot + t);
      const bool active = (s >= 0) & (pos >= 0) & (((pos + 1) & (p.ratio - 1)) == 0) & (kv >= 0);
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
  uint32_t out = incl - n, total = 0;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) {
    const uint32_t c = warp_base[w];
    if (w < warp) out += c;
    total += c;
  }
  int32_t* list = reinterpret_cast<int32_t*>(p.ws + 1);
#pragma unroll
  for (int i = 0; i < kTok; ++i)
    if ((flags >> i) & 1u) list[base + out++] = static_cast<int32_t>(base + static_cast<int64_t>(tid) * kTok + i);
  if (tid == 0) list[p.T + blockIdx.x] = static_cast<int32_t>(total);
}

// --------------------------------------------------------------------------- compress kernel
// State blocks other than 8 rows (any multiple of 8, through the configurable entry point): the
// window's 128 rows are 16 chunks of 8 rows, chunk j starting at row q0 = start + 8j of the
// request, which is row q0 % sblk of block block_table[req][q0 / sblk]. start is a multiple of 128
// and sblk of 8, so a chunk never spans two blocks. Returns the block id (for the range check)
// and the chunk's element offset. The 8-row kernels (the C128 layout, where a chunk is a block)
// are separate template instances that carry none of these 64-bit divisions.
__device__ __forceinline__ int chunk_block(const Params& p, int req, long long start, int j, int64_t* off) {
  const long long q0 = start + static_cast<long long>(kStateBlock) * j;
  const long long col = q0 / p.sblk, row = q0 - col * p.sblk;
  const int blk = __ldg(p.bt + static_cast<int64_t>(req) * p.bt_stride + col);
  *off = static_cast<int64_t>(blk) * p.s0 + row * p.s1;
  return blk;
}

struct __align__(16) WinDesc {
  const float* src[kWindowBlocks];  // first row of each of the window's 16 chunks of 8 rows
  uint8_t* kv_dst;                  // 576 token bytes of the k_cache slot
  uint8_t* scale_dst;               // 8 scale bytes of the slot
  const float* cs_row;              // cos_sin_cache row of the window start
  float* comp_dst;                  // optional fp32 export
  int32_t kind;                     // 0: window, 1: no more windows
  int32_t pad[3];
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
  uint32_t chunk_prefix[kMaxPlanChunks + 1];  // planned path: active windows before each chunk
  int abort_flag;
};

template <bool ANY>
__device__ void scheduler_warp(const Params& p, Smem& S, int lane) {
  const volatile int* abort_flag = &S.abort_flag;
  // the planning pass's list (the kernel entry waited for that pass)
  const uint32_t A = plan_prefix_warp(p, S.chunk_prefix, lane);
  uint32_t widx = 0;
  for (bool first_claim = true;; first_claim = false) {
    if (*abort_flag) return;
    long long t = 0, pos = 0, kvs = 0;
    int req = 0;
    uint32_t err = 0;
    // the first claim is static (CTA b takes window b), which takes a global round trip off the
    // way to the first copy; the rest come from the shared counter
    uint32_t a = 0;
    if (lane == 0) a = first_claim ? blockIdx.x : gridDim.x + atomicAdd(&p.ws->next, 1u);
    a = __shfl_sync(0xffffffffu, a, 0);
    const bool end = a >= A;
    if (!end && lane == 0) t = plan_token(p, S.chunk_prefix, a);
    if (!end) {
      if (lane == 0) {
        req = __ldg(p.ttr + t);
        pos = __ldg(p.pos + t);
        kvs = __ldg(p.kvslot + t);
        if (req < 0 || req >= p.bt_rows) err |= C128_DEV_BAD_REQ;
        if ((ANY ? pos / p.sblk : pos / kStateBlock) >= p.bt_cols) err |= C128_DEV_BAD_BT_COL;
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
    int64_t choff = 0;
    if (!end && !(err & (C128_DEV_BAD_REQ | C128_DEV_BAD_BT_COL))) {
      if constexpr (ANY) {
        if (lane < kWindowBlocks) blk = chunk_block(p, req, pos - (kRatio - 1), lane, &choff);
      } else {
        if (lane < kWindowBlocks)
          blk = __ldg(p.bt + static_cast<int64_t>(req) * p.bt_stride + (pos - (kRatio - 1)) / kStateBlock + lane);
      }
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
      if (lane < kWindowBlocks) d.src[lane] = p.state + (ANY ? choff : static_cast<int64_t>(blk) * p.s0);
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
      if (p.stall_first_window && blockIdx.x == 0 && it == 0) {
        // test of the bounded waits: this stage never fills, so its consumers give up after the
        // time limit and the kernel reports C128_DEV_TIMEOUT instead of hanging
      } else if (block_contiguous) {
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
        // the rows go to registers and the stage is released before the arithmetic
        BlockRows br;
        stage_rows(S.stage[s], c0, br);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[s]);
        online_fold(br, o);
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

template <bool ANY>
__global__ void __launch_bounds__(kThreads, 1) compress_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Launched as a programmatic dependent of the planning pass, which itself waits for the kernel
  // before it: nothing global is touched before that pass has completed (the barriers, in shared
  // memory, are set up while it runs). The next launch may start as soon as every CTA of this one
  // runs.
  launch_dependents();
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
  grid_dependency_wait();
  if (warp == 0) {
    scheduler_warp<ANY>(p, S, lane);
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
// R: ring depth; 0 = as deep as the CTA's blocks allow up to kStages (one CTA per SM). A shallower
// ring lets several CTAs share an SM, so that one CTA's start overlaps another's stream.
template <int S, int R = 0>
struct DirectCfg {
  static constexpr int kBlocks = kWindowBlocks / S;                 // stages per CTA
  static constexpr int kDeep = kBlocks < kStages ? kBlocks : kStages;
  static constexpr int kRing = R > 0 && R < kDeep ? R : kDeep;
};

constexpr int kMidRing = 3;  // ring of the one-CTA-per-token kernel (more tokens than SMs)
static_assert(2 * (kMidRing * kStageBytes + 12 * 1024) <= 227 * 1024, "two such CTAs per SM");

template <int S, int R = 0>
struct DirectSmem {
  float stage[DirectCfg<S, R>::kRing][kStateBlock * kRow];
  uint64_t full[DirectCfg<S, R>::kRing];
  uint64_t empty[DirectCfg<S, R>::kRing];
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

template <int S, bool ANY, int R = 0>
__global__ void __launch_bounds__(kThreads, R > 0 ? 2 : 1) direct_kernel(Params p) {
  using Cfg = DirectCfg<S, R>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  DirectSmem<S, R>& D = *reinterpret_cast<DirectSmem<S, R>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
  const int64_t t = static_cast<int64_t>(blockIdx.x) / S;
  // Launched as a programmatic dependent of the kernel before it on the stream: the next call may
  // start as soon as every CTA of this one runs, and this one reads nothing before the kernel
  // before it has completed (its writes, possibly these inputs, are then visible).
  launch_dependents();
  grid_dependency_wait();
  // the token (every thread; broadcast loads), issued before the barrier set-up so that their
  // latency overlaps it
  const int64_t slot = __ldg(p.slot + t), pos = __ldg(p.pos + t), kvs = __ldg(p.kvslot + t);
  const int req = __ldg(p.ttr + t);
  // an inactive token's CTAs leave at once (uniformly: every CTA of a cluster reads the same token)
  if (!((slot >= 0) & (pos >= 0) & ((pos & (kRatio - 1)) == kRatio - 1) & (kvs >= 0))) return;
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

  // the token's window
  uint32_t err = 0;
  if (req < 0 || req >= p.bt_rows) err |= C128_DEV_BAD_REQ;
  if ((ANY ? pos / p.sblk : pos / kStateBlock) >= p.bt_cols) err |= C128_DEV_BAD_BT_COL;
  if (pos - (kRatio - 1) >= p.cs_rows) err |= C128_DEV_BAD_COS_ROW;
  if (kvs >= p.nkb * p.kv_bs) err |= C128_DEV_BAD_KV_SLOT;
  int blk = 0;  // lane j of every warp holds the block id of chunk j
  if (!(err & (C128_DEV_BAD_REQ | C128_DEV_BAD_BT_COL))) {
    if constexpr (ANY) {
      int64_t unused;
      if (lane < kWindowBlocks) blk = chunk_block(p, req, pos - (kRatio - 1), lane, &unused);
    } else {
      if (lane < kWindowBlocks)
        blk = __ldg(p.bt + static_cast<int64_t>(req) * p.bt_stride + (pos - (kRatio - 1)) / kStateBlock + lane);
    }
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
      // the block id travels by shuffle (32 bits), lane 0 adds the chunk's row within the block
      const int b = __shfl_sync(0xffffffffu, blk, static_cast<int>(rank) * Cfg::kBlocks + j);
      if (lane == 0 && !failed) {
        const int s = j % Cfg::kRing;
        const uint32_t round = j / Cfg::kRing;
        if (round > 0 && !mbar_wait(&D.empty[s], (round - 1u) & 1u, abort_flag)) {
          failed = true;
        } else {
          mbar_arrive_expect_tx(&D.full[s], kStageBytes);
          int64_t o = static_cast<int64_t>(b) * p.s0;
          if constexpr (ANY)
            o += ((pos - (kRatio - 1) + static_cast<long long>(kStateBlock) * (static_cast<int>(rank) * Cfg::kBlocks + j)) %
                  p.sblk) * p.s1;
          const float* src = p.state + o;
          if (p.stall_first_window && blockIdx.x == 0 && j == 0) {
            // test of the bounded waits: this stage never fills, so the consumers give up after
            // the time limit and the kernel reports C128_DEV_TIMEOUT instead of hanging
          } else if (p.s1 == kRow) {
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
        // the rows go to registers and the stage is released before the arithmetic
        BlockRows br;
        stage_rows(D.stage[s], c0, br);
        __syncwarp();
        if (lane == 0) mbar_arrive(&D.empty[s]);
        online_fold(br, o);
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

template <int S, bool ANY, int R = 0>
cudaError_t launch_direct(const Params& p, const LaunchCfg& cfg, cudaStream_t stream) {
  if (cfg.ev_begin != nullptr) {
    const cudaError_t e = cudaEventRecord(cfg.ev_begin, stream);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(p.T * S));
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = sizeof(DirectSmem<S, R>);
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (cfg.pdl && cfg.ev_begin == nullptr) {  // events between the kernels would serialise them anyway
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (S > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = S;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  lc.attrs = attr;
  lc.numAttrs = n;
  cudaError_t e = cudaLaunchKernelEx(&lc, direct_kernel<S, ANY, R>, p);
  if (e != cudaSuccess) return e;
  if (cfg.ev_end != nullptr) e = cudaEventRecord(cfg.ev_end, stream);
  return e;
}

}  // namespace

int compress_smem_bytes() { return static_cast<int>(sizeof(Smem)); }

namespace {
template <bool ANY>
cudaError_t set_direct_smem(cudaFuncAttribute a) {
  cudaError_t e = cudaFuncSetAttribute(direct_kernel<1, ANY>, a, static_cast<int>(sizeof(DirectSmem<1>)));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(direct_kernel<2, ANY>, a, static_cast<int>(sizeof(DirectSmem<2>)));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(direct_kernel<4, ANY>, a, static_cast<int>(sizeof(DirectSmem<4>)));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(direct_kernel<8, ANY>, a, static_cast<int>(sizeof(DirectSmem<8>)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(direct_kernel<1, ANY, kMidRing>, a, static_cast<int>(sizeof(DirectSmem<1, kMidRing>)));
  if (e == cudaSuccess)  // all of the SM's shared memory, for two of these CTAs
    e = cudaFuncSetAttribute(direct_kernel<1, ANY, kMidRing>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return e;
}
}  // namespace

cudaError_t prepare_device(int /*device*/) {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(compress_kernel<false>, a, static_cast<int>(sizeof(Smem)));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(compress_kernel<true>, a, static_cast<int>(sizeof(Smem)));
  if (e == cudaSuccess) e = set_direct_smem<false>(a);
  if (e == cudaSuccess) e = set_direct_smem<true>(a);
  if (e == cudaSuccess) e = prepare_small();
  if (e == cudaSuccess) e = prepare_indexer_windows();
  return e;
}

namespace {
// Enqueue the planning pass and return, in *q, the parameters of the kernel that takes windows from
// its list: per-chunk lists (no zeroing pass) up to kMaxPlanChunks chunks, else the compact list
// behind a zeroing of its counters. With `early`, the pass is a programmatic dependent of the
// kernel before it (it launches while that kernel finishes and waits for it before any global
// access). Not behind the head-512 small-window kernel: there every call took about 20 us longer
// than its kernel (the 832-thread CTAs and the early pass did not overlap; measured, not
// explained), against 1 us without the early launch. `wide`: 512 threads of 4 tokens per chunk
// instead of 256 of 8 (1.0-1.8 us less per planned call, but 2.7 us more behind the head-128
// small-window kernel, whose CTAs the early 512-thread CTAs then sit beside).
cudaError_t launch_plan(const Params& p, const LaunchCfg& cfg, cudaStream_t stream, Params* q, bool early,
                        bool wide) {
  const int plan_grid = static_cast<int>((p.T + kPlanTokensPerCta - 1) / kPlanTokensPerCta);
  *q = p;
  q->chunked = plan_grid <= kMaxPlanChunks;
  if (q->chunked) {
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3(static_cast<unsigned>(plan_grid));
    pc.blockDim = dim3(wide ? 512 : 256);
    pc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    pc.attrs = attr;
    pc.numAttrs = cfg.pdl && early ? 1 : 0;
    return wide ? cudaLaunchKernelEx(&pc, plan_chunks_kernel<512>, *q) : cudaLaunchKernelEx(&pc, plan_chunks_kernel<256>, *q);
  }
  cudaError_t e = cudaMemsetAsync(p.ws, 0, 2 * sizeof(unsigned int), stream);  // count, next
  if (e != cudaSuccess) return e;
  plan_kernel<<<plan_grid, kPlanThreads, 0, stream>>>(*q);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch(const Params& p, const LaunchCfg& cfg, cudaStream_t stream) {
  if (!is_c128(p)) {
    cudaError_t e;
    if (p.T <= static_cast<int64_t>(kStridedTokensPerSm) * cfg.sm_count) {
      // few tokens per SM: the ring kernels stride over the tokens themselves (no planning pass,
      // no counters); configurations the gather kernel serves still take the planned path
      Params q = p;
      q.strided = 1;
      if (cfg.ev_begin != nullptr && (e = cudaEventRecord(cfg.ev_begin, stream)) != cudaSuccess) return e;
      e = small_window_path(q) ? launch_small(q, cfg, stream) : launch_indexer_windows(q, cfg, stream);
      if (e != cudaErrorNotSupported) {
        if (e != cudaSuccess) return e;
        if (cfg.ev_end != nullptr) e = cudaEventRecord(cfg.ev_end, stream);
        return e;
      }
    }
    Params q;
    const bool small = small_window_path(p);
    if ((e = launch_plan(p, cfg, stream, &q, !(small && p.head == kHead), !(small && p.head != kHead))) != cudaSuccess)
      return e;
    if (cfg.ev_begin != nullptr && (e = cudaEventRecord(cfg.ev_begin, stream)) != cudaSuccess) return e;
    if (small_window_path(q)) {
      e = launch_small(q, cfg, stream);
    } else {
      e = launch_indexer_windows(q, cfg, stream);
      if (e == cudaErrorNotSupported) e = launch_gather(q, cfg, stream);
    }
    if (e != cudaSuccess) return e;
    if (cfg.ev_end != nullptr) e = cudaEventRecord(cfg.ev_end, stream);
    return e;
  }
  const bool any_block = p.sblk != kStateBlock;  // the C128 layout has 8-row state blocks
  switch (direct_split(p.T, cfg.sm_count)) {
    case 8: return any_block ? launch_direct<8, true>(p, cfg, stream) : launch_direct<8, false>(p, cfg, stream);
    case 4: return any_block ? launch_direct<4, true>(p, cfg, stream) : launch_direct<4, false>(p, cfg, stream);
    case 2: return any_block ? launch_direct<2, true>(p, cfg, stream) : launch_direct<2, false>(p, cfg, stream);
    case 1: return any_block ? launch_direct<1, true>(p, cfg, stream) : launch_direct<1, false>(p, cfg, stream);
    default: break;
  }
  cudaError_t e;
  // up to 8 tokens per SM: one CTA per token with a 3-stage ring, two CTAs per SM, so that the
  // hardware deals the windows out and one CTA's start and epilogue overlap another's stream
  if (p.T <= static_cast<int64_t>(kStridedTokensPerSm) * cfg.sm_count)
    return any_block ? launch_direct<1, true, kMidRing>(p, cfg, stream) : launch_direct<1, false, kMidRing>(p, cfg, stream);
  Params q;
  e = launch_plan(p, cfg, stream, &q, true, true);
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
  e = any_block ? cudaLaunchKernelEx(&lc, compress_kernel<true>, q) : cudaLaunchKernelEx(&lc, compress_kernel<false>, q);
  if (e != cudaSuccess) return e;
  if (cfg.ev_end != nullptr) e = cudaEventRecord(cfg.ev_end, stream);
  return e;
}

}  // namespace c128
