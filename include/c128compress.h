/*
 * libc128compress — GB300 (sm_103a) DeepSeek-V4 C128 sparse-attention KV compressor.
 *
 * One stream-ordered call, compress_norm_rope_store(), does for every active token
 *   1. window gather: the 128 state-cache rows p-127 .. p of the token's request, found through
 *      the paged block table (state block size 8, so 16 whole blocks);
 *   2. a per-column softmax of score (row columns 512..1023) over those 128 rows and the
 *      softmax-weighted sum of kv (row columns 0..511): compressed[512], fp32;
 *   3. RMSNorm with weight rms_w and eps;
 *   4. FP8 e4m3 quantisation of the 448 "nope" columns with one UE8M0 (power-of-two) scale per
 *      64 columns, and interleaved-pair (GPT-J) RoPE of the 64 rope columns, stored as bf16;
 *   5. the paged k_cache store at kv_slot_mapping[t].
 * It follows the fused Triton kernel _fused_kv_compress_norm_rope_insert_sparse_attn and its
 * launcher compress_norm_rope_store_triton on the API page of
 * vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache (sections "Gather state cache
 * entries", "Softmax + weighted sum", "RMSNorm", "KV cache pointers", "FP8 UE8M0 quant",
 * "GPT-J RoPE"), in the C128 layout of vLLM PR #44230 "optimize the compressor 128 split cutedsl
 * kernel" (Summary: head 512, state width 512, compress ratio 128, no overlap, state block 8;
 * Changes: reject unsupported layouts and kv_cache_block_size != k_cache.shape[1]).
 *
 * Arithmetic (where the pages leave precision open): the softmax and weighted sum run in fp32
 * (within 1e-5 relative / 1e-6 absolute of the exact value); from compressed[] on, every step is
 * a fixed IEEE computation, so the bytes are a pure function of compressed[]:
 *   var = RN32(exact(sum c^2) / 512); rrms = RN32(1 / sqrt(double(RN32(var + eps))));
 *   normed = RN32(RN32(c * rrms) * w); nope: bf16 round, absmax (floor RN32(1e-4)),
 *   e = ceil(log2(RN32(absmax * RN32(1/448)))), q = e4m3_rn_satfinite(clamp(x * 2^-e, +-448)),
 *   scale byte = clamp(e + 127, 0, 255), 8th scale byte 0; rope: e' = RN32(RN32(e*C) - RN32(o*S)),
 *   o' = RN32(RN32(o*C) + RN32(e*S)), each stored as bf16 (round to nearest even).
 *
 * A token is active iff slot_mapping[t] >= 0, positions[t] >= 0, (positions[t] + 1) % 128 == 0
 * and kv_slot_mapping[t] >= 0. Inactive tokens write nothing; no byte of k_cache outside the
 * 576 token bytes and 8 scale bytes of an active token's slot is touched.
 *
 * All tensors are caller-owned device memory described by c128_tensor_t (strides in elements).
 * The call is asynchronous on `stream`: it never synchronises the host with the GPU and never
 * reads device memory back to the host.
 * It uses a per-(device, stream) workspace owned by the library (a 256-byte header with the
 * sticky device error bits, then one int32 per token). The first call on a stream, and any call
 * with more tokens than that workspace holds, grows it stream-ordered: a new buffer from the
 * device's default memory pool (cudaMallocAsync on `stream`), the header copied device-to-device
 * on `stream`, the old buffer returned with cudaFreeAsync on `stream`. Nothing waits on the host.
 * A stream that is being captured into a CUDA graph cannot grow its workspace: such a call
 * returns C128_ERR_CAPTURE and enqueues nothing, so call c128_reserve_workspace with the largest
 * batch before capturing. A graph keeps the workspace it was captured with; a later call on the
 * same stream that grows the workspace frees that buffer, so reserve enough before capturing a
 * graph that will be replayed. Calls on the same stream are serialised by the stream; calls on
 * different streams use different workspaces. c128_release_stream returns one stream's workspace
 * (call it before destroying the stream). Two active tokens naming the same kv slot race
 * (undefined which one lands); this is not checked.
 */
#ifndef C128COMPRESS_H
#define C128COMPRESS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* c128_stream_t;

/* Element types of c128_tensor_t. */
enum {
    C128_I32 = 1,
    C128_I64 = 2,
    C128_F32 = 3,
    C128_U8 = 4,
};

/* A strided view of caller-owned device memory. shape/stride beyond ndim are ignored. */
typedef struct c128_tensor {
    void* data;          /* device pointer (may be NULL only when the tensor is empty) */
    int32_t dtype;       /* one of C128_I32, C128_I64, C128_F32, C128_U8 */
    int32_t ndim;        /* 1 .. 4 */
    int64_t shape[4];
    int64_t stride[4];   /* in elements */
} c128_tensor_t;

/* Return codes. Every error is detected on the host before anything is launched, except
 * C128_ERR_CUDA (a CUDA call or launch failed) and C128_ERR_NOMEM (workspace allocation);
 * C128_ERR_CAPTURE is also returned before anything is enqueued. */
enum {
    C128_OK = 0,
    C128_ERR_NULL_PTR = 1,     /* a descriptor, or the data of a non-empty tensor, is NULL */
    C128_ERR_DTYPE = 2,        /* wrong element type */
    C128_ERR_SHAPE = 3,        /* wrong rank / extent, or token counts disagree */
    C128_ERR_STRIDE = 4,       /* innermost dimension not contiguous, or an unusable stride */
    C128_ERR_ALIGN = 5,        /* state_cache or k_cache base/stride not aligned (see below) */
    C128_ERR_UNSUPPORTED = 6,  /* not the C128 layout: state block != 8, row != 1024, head != 512 */
    C128_ERR_ARG = 7,          /* kv_block_size < 1 or != k_cache.shape[1]; too many tokens */
    C128_ERR_CUDA = 8,
    C128_ERR_NOMEM = 9,
    C128_ERR_TOO_MANY_TOKENS = 10, /* c128_compress_norm_rope_store_noalloc: T > C128_NOALLOC_MAX_TOKENS */
    C128_ERR_CAPTURE = 11,     /* the stream is being captured and its workspace would have to grow */
};

/* Device-side error bits (OR-ed into the stream's workspace, sticky until cleared).
 * An active token whose indices fall outside the given tensors is skipped (writes nothing)
 * and reports one of the first five bits; a bounded wait that ran out reports TIMEOUT. */
enum {
    C128_DEV_BAD_REQ = 1,        /* token_to_req_indices[t] outside [0, block_table.shape[0]) */
    C128_DEV_BAD_BT_COL = 2,     /* positions[t] / 8 >= block_table.shape[1] */
    C128_DEV_BAD_BLOCK = 4,      /* a window block id outside [0, state_cache.shape[0]) */
    C128_DEV_BAD_COS_ROW = 8,    /* window start (p/128)*128 >= cos_sin_cache.shape[0] */
    C128_DEV_BAD_KV_SLOT = 16,   /* kv_slot_mapping[t] >= k_cache.shape[0] * kv_block_size */
    C128_DEV_TIMEOUT = 32,       /* a pipeline wait exceeded its time limit; the kernel gave up */
};

/*
 * compress_norm_rope_store — the whole C128 compressor path for one batch of tokens.
 *
 *   token_to_req_indices [T]               int32  request of each token (contiguous)
 *   positions            [T]               int64  absolute position of each token (contiguous)
 *   slot_mapping         [T]               int64  state-cache slot; < 0 marks a padded token
 *   block_table          [R, MB]           int32  state-cache block ids per request; row stride
 *                                                 stride[0] >= MB, stride[1] == 1
 *   state_cache          [NB, 8, 1024]     fp32   row = kv[0:512] | score[512:1024];
 *                                                 stride[2] == 1, stride[1] >= 1024,
 *                                                 data 16-byte aligned, stride[0] and stride[1]
 *                                                 multiples of 4 elements
 *   rms_w                [512]             fp32   RMSNorm weight (contiguous)
 *   eps                                    fp32   RMSNorm epsilon
 *   cos_sin_cache        [MP, 64]          fp32   cos in [0, 32), sin in [32, 64) of row
 *                                                 (p / 128) * 128; stride[1] == 1
 *   k_cache              [NKB, bs, W>=584] uint8  written in place: block b holds bs token
 *                                                 records of 576 bytes (448 e4m3 + 64 bf16 rope)
 *                                                 at b*stride[0] + off*576, then bs x 8 scale
 *                                                 bytes (7 UE8M0 + a zero pad) at
 *                                                 b*stride[0] + bs*576 + off*8; W*bs >= bs*584,
 *                                                 data 16-byte aligned, stride[0] a multiple of 8
 *   kv_slot_mapping      [T]               int64  k_cache slot (block*bs + offset); < 0: no store
 *   kv_block_size                                 must equal k_cache.shape[1]
 *   stream                                        CUDA stream the work is enqueued on
 *
 * Returns C128_OK or a C128_ERR_* code (nothing is launched on an error). T == 0 is a no-op.
 */
int compress_norm_rope_store(const c128_tensor_t* token_to_req_indices,
                             const c128_tensor_t* positions,
                             const c128_tensor_t* slot_mapping,
                             const c128_tensor_t* block_table,
                             const c128_tensor_t* state_cache,
                             const c128_tensor_t* rms_w,
                             float eps,
                             const c128_tensor_t* cos_sin_cache,
                             const c128_tensor_t* k_cache,
                             const c128_tensor_t* kv_slot_mapping,
                             int64_t kv_block_size,
                             c128_stream_t stream);

/*
 * Test of the failure handling, for tests only. Runs compress_norm_rope_store on the same
 * arguments (C128 layout), except that CTA 0 arms the first stage of its first window and never
 * copies into it (the one-CTA-per-token kernel up to 8 tokens per SM, where CTA 0 has a window only
 * if token 0 is active; the compress kernel above).
 * Every wait in the kernels is bounded (1 s), so the consumers of that stage give up, the CTA
 * stops, and the kernel ends with C128_DEV_TIMEOUT in the device error bits (read them with
 * c128_device_errors) instead of hanging; the CUDA context stays usable. Other CTAs store their
 * windows as usual; CTA 0's windows are not stored. Takes about two seconds of GPU time. Returns
 * C128_ERR_ARG when the batch has no more tokens than the GPU has SMs (such batches run the
 * cluster-split kernel, which is not set up for this test), else the codes of
 * compress_norm_rope_store.
 */
int c128_debug_stall_first_window(const c128_tensor_t* token_to_req_indices,
                                  const c128_tensor_t* positions,
                                  const c128_tensor_t* slot_mapping,
                                  const c128_tensor_t* block_table,
                                  const c128_tensor_t* state_cache,
                                  const c128_tensor_t* rms_w,
                                  float eps,
                                  const c128_tensor_t* cos_sin_cache,
                                  const c128_tensor_t* k_cache,
                                  const c128_tensor_t* kv_slot_mapping,
                                  int64_t kv_block_size,
                                  c128_stream_t stream);

/*
 * Same as compress_norm_rope_store, and also writes the fp32 compressed vector (the softmax-
 * weighted sum, before RMSNorm) of every token it stores to comp_out [T, 512] fp32 (contiguous,
 * 16-byte aligned). Rows of other tokens are left as they were. For tests and diagnostics: it
 * exposes the quantity the byte-exact epilogue is a function of.
 */
int c128_compress_norm_rope_store_debug(const c128_tensor_t* token_to_req_indices,
                                        const c128_tensor_t* positions,
                                        const c128_tensor_t* slot_mapping,
                                        const c128_tensor_t* block_table,
                                        const c128_tensor_t* state_cache,
                                        const c128_tensor_t* rms_w,
                                        float eps,
                                        const c128_tensor_t* cos_sin_cache,
                                        const c128_tensor_t* k_cache,
                                        const c128_tensor_t* kv_slot_mapping,
                                        int64_t kv_block_size,
                                        const c128_tensor_t* comp_out,
                                        c128_stream_t stream);

/*
 * c128_compress_norm_rope_store_noalloc — the same operation, for callers that cannot allocate.
 * The pages have no counterpart to this entry point; it exists for the library's users.
 *
 * compress_norm_rope_store keeps its list of active tokens in a workspace that it allocates with
 * cudaMalloc on the first call on a stream and whenever a larger batch arrives. Some callers may
 * not allocate device memory once they are running: a serving engine that hands all free memory
 * to its KV caches at start-up and must never see an allocation (or its implicit device
 * synchronisation) on the decode path, code running inside a memory-pool or allocator callback,
 * or a host that enforces a fixed device-memory budget. This entry point allocates nothing.
 *
 * Its scratch (a 256-byte header, the token list and the planning pass's per-chunk counts) is one
 * static device array for C128_NOALLOC_MAX_TOKENS tokens (256 KiB + 384 B) in the library image;
 * every GPU that loads the library holds it until the process exits. The first call on each
 * device looks up that array's
 * device address (cudaGetSymbolAddress, with that device current) and caches it; make that first
 * call before any stream capture. Arguments, layout and results are exactly those of
 * compress_norm_rope_store; T > C128_NOALLOC_MAX_TOKENS returns C128_ERR_TOO_MANY_TOKENS without
 * launching anything. All calls share the one array: each call clears the counters it needs,
 * and calls that can overlap on the GPU (different streams, or different host threads) race and
 * corrupt each other's work. Device error bits of these calls are not readable through
 * c128_device_errors (tokens with out-of-range indices are still skipped).
 */
#define C128_NOALLOC_MAX_TOKENS 65536
int c128_compress_norm_rope_store_noalloc(const c128_tensor_t* token_to_req_indices,
                                          const c128_tensor_t* positions,
                                          const c128_tensor_t* slot_mapping,
                                          const c128_tensor_t* block_table,
                                          const c128_tensor_t* state_cache,
                                          const c128_tensor_t* rms_w,
                                          float eps,
                                          const c128_tensor_t* cos_sin_cache,
                                          const c128_tensor_t* k_cache,
                                          const c128_tensor_t* kv_slot_mapping,
                                          int64_t kv_block_size,
                                          c128_stream_t stream);

/*
 * compress_norm_rope_store_ex — the same op for the other configurations of the fused kernels
 * on the API page (one launcher, compress_norm_rope_store_triton, serves all three):
 *
 *   C128_FORMAT_SPARSE_FP8    _fused_kv_compress_norm_rope_insert_sparse_attn: head 512, rope 64;
 *                             448 e4m3 + 64 bf16 rope (576 B) then 8 scale bytes per slot
 *   C128_FORMAT_INDEXER_FP8   _fused_kv_compress_norm_rope_insert_indexer_attn: head 128, rope 64;
 *                             RoPE of the last 32 pairs first, bf16 round, one absmax block:
 *                             128 e4m3 bytes per slot, then one fp32 scale 2^e (4 B) per slot
 *   C128_FORMAT_INDEXER_MXFP4 _fused_kv_compress_norm_rope_insert_indexer_mxfp4_attn: head 128;
 *                             RoPE, bf16 round, per 32 values e = ceil(log2(absmax/6)) (absmax
 *                             floor 6*2^-126, e clamped to [-127,127]), E2M1 codes of x*2^-e
 *                             (round to nearest even, saturating), pair j in byte j with the even
 *                             value in the low nibble: 64 bytes per slot, then 4 UE8M0 bytes (e+127)
 *
 * with compress ratio `compress_ratio` (a power of two; window end: (p+1) % ratio == 0) and, when
 * `overlap` is 1, windows of 2*ratio rows whose newer `ratio` rows read kv and score at +head_dim
 * (the C4 layout); rows at negative positions take no weight. A state row is kv[state_width]
 * followed by score[state_width] (state_width >= (1+overlap)*head_dim, a multiple of 4), blocks of
 * any number of rows (state_cache [NB, block, 2*state_width]); cos/sin come from row
 * (p / ratio) * ratio. k_cache blocks hold bs token records then bs scale records, as above.
 * comp_out, if not NULL, receives the fp32 compressed vectors ([T, head_dim], contiguous, 16-byte
 * aligned) of stored tokens.
 * The k_cache block stride (stride[0], bytes) must be a multiple of 8 for the sparse format, 4 for
 * the indexer FP8 format and 2 for MXFP4 (the widest store of each), which the natural layout
 * bs x record bytes always is.
 * Everything else is as for compress_norm_rope_store; the C128 configuration (512, 64, 128, 0, 512,
 * sparse) runs the same kernels as compress_norm_rope_store when its state block is any multiple
 * of 8 rows.
 * Returns C128_ERR_NULL_PTR for a NULL config and C128_ERR_UNSUPPORTED for a configuration outside
 * the ones above (another head or rope size, a head that does not match the format, a ratio that
 * is not a power of two or makes windows longer than 256 rows, overlap other than 0 or 1, a state
 * width below (1 + overlap) * head_dim or not a multiple of 4); the tensor checks and their codes
 * are those of compress_norm_rope_store, with head_dim in place of 512.
 * Kernels: the C128 configuration with a state block that is a multiple of 8 rows runs the C128
 * kernels; windows of at most 8 rows stream through a shared-memory ring (many windows per SM);
 * longer head-128 windows whose state block is a multiple of 8 rows stream in 8-row tiled loads;
 * the rest run a gather kernel. All of them are CUDA-graph capturable.
 */
enum {
    C128_FORMAT_SPARSE_FP8 = 0,
    C128_FORMAT_INDEXER_FP8 = 1,
    C128_FORMAT_INDEXER_MXFP4 = 2,
};
typedef struct c128_config {
    int32_t head_dim;        /* 512 (sparse format) or 128 (indexer formats) */
    int32_t rope_head_dim;   /* 64 */
    int32_t compress_ratio;  /* power of two; (1 + overlap) * ratio <= 256 */
    int32_t overlap;         /* 0 or 1 */
    int32_t state_width;     /* kv columns of a state row; as many score columns follow */
    int32_t cache_format;    /* C128_FORMAT_* */
} c128_config_t;
int compress_norm_rope_store_ex(const c128_config_t* config,
                                const c128_tensor_t* token_to_req_indices,
                                const c128_tensor_t* positions,
                                const c128_tensor_t* slot_mapping,
                                const c128_tensor_t* block_table,
                                const c128_tensor_t* state_cache,
                                const c128_tensor_t* rms_w,
                                float eps,
                                const c128_tensor_t* cos_sin_cache,
                                const c128_tensor_t* k_cache,
                                const c128_tensor_t* kv_slot_mapping,
                                int64_t kv_block_size,
                                const c128_tensor_t* comp_out,
                                c128_stream_t stream);

/*
 * The same test for the other configurations (tests only): compress_norm_rope_store_ex with the
 * small-window kernel (windows of at most 8 rows) leaving the stage of the first listed window
 * unfilled, or the indexer kernel (head-128 windows of more than 8 rows) leaving CTA 0's first
 * stage unfilled, with the same outcome:
 * C128_DEV_TIMEOUT in the device error bits, the other CTAs' windows stored, the context usable.
 * Configurations served by the gather kernel (no copy warp) run normally. Returns the codes of
 * compress_norm_rope_store_ex.
 */
int c128_debug_stall_first_window_ex(const c128_config_t* config,
                                     const c128_tensor_t* token_to_req_indices,
                                     const c128_tensor_t* positions,
                                     const c128_tensor_t* slot_mapping,
                                     const c128_tensor_t* block_table,
                                     const c128_tensor_t* state_cache,
                                     const c128_tensor_t* rms_w,
                                     float eps,
                                     const c128_tensor_t* cos_sin_cache,
                                     const c128_tensor_t* k_cache,
                                     const c128_tensor_t* kv_slot_mapping,
                                     int64_t kv_block_size,
                                     c128_stream_t stream);

/* Human-readable name of a return code (static string, never NULL). */
const char* c128_status_string(int status);

/* Make the workspace of (current device, stream) hold at least max_tokens tokens, growing it
 * stream-ordered as described at the top (cudaMallocAsync / device-to-device header copy /
 * cudaFreeAsync on `stream`, no host synchronisation). Returns C128_ERR_CAPTURE if it would have
 * to grow while `stream` is being captured, C128_ERR_NOMEM if the pool has no room. */
int c128_reserve_workspace(int64_t max_tokens, c128_stream_t stream);

/* Return the workspace and kernel-timer events of (current device, stream) to the library: the
 * workspace is freed with cudaFreeAsync on `stream`, after the work already enqueued there, and
 * the stream's sticky device error bits go with it. Call it before destroying a stream the
 * library was used on (a later call on a stream with the same handle starts a fresh workspace).
 * Does not synchronise. Returns C128_ERR_CAPTURE (and releases nothing) while `stream` is being
 * captured. */
int c128_release_stream(c128_stream_t stream);

/* Synchronise `stream`, store the device error bits (C128_DEV_*) of its workspace in *bits,
 * and clear them when `clear` is non-zero. A stream never used reports 0. */
int c128_device_errors(c128_stream_t stream, uint32_t* bits, int clear);

/* Kernel timer. Between begin and end, every call on `stream` records a CUDA event pair around
 * its compress kernel (the dominant kernel; the planning kernel is outside the pair). end()
 * synchronises the stream and returns the summed kernel time in ms and the number of launches.
 * While the timer runs the compress kernel does not overlap the planning kernel. */
int c128_kernel_timer_begin(c128_stream_t stream);
int c128_kernel_timer_end(c128_stream_t stream, double* total_ms, int64_t* launches);

/* Static launch facts of the compress kernel on the current device. */
typedef struct c128_info {
    int32_t sm_count;        /* streaming multiprocessors */
    int32_t threads;         /* threads per CTA of the compress kernel */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t stages;          /* shared-memory ring depth, 32 KiB (one state block) per stage */
    int32_t ctas_per_sm;     /* resident CTAs per SM */
    int32_t plan_tokens_per_cta;
    int32_t wait_timeout_ms; /* limit of every pipeline wait */
    int32_t version;
} c128_info_t;
int c128_get_info(c128_info_t* info);

/* Read-bandwidth probe (a measurement helper; the pages have no counterpart). It streams `bytes`
 * of the device buffer `buf` once with plain 16-byte loads and XORs every 32-bit word into the
 * device word *xor_out (atomicXor per warp: zero it first and it ends as the XOR of the buffer's
 * words, which proves every byte was read). The compressor's kernels read far more than they
 * write, so this read rate, taken in the same process, is the denominator beside the copy
 * bandwidth for their reported bandwidth fraction.
 *   threads_per_cta   32..1024, a multiple of 32
 *   ctas_per_sm       1..32, with threads_per_cta x ctas_per_sm <= 2048; the grid is #SM x the
 *                     smaller of ctas_per_sm and the CTAs that fit on an SM at once (so all are
 *                     resident), fewer when the buffer holds less than one load per thread
 *   loads_in_flight   16-byte loads each thread issues before it uses them: 1, 2, 4 or 8
 * `buf` 16-byte aligned, `bytes` a multiple of 16; both pointers are caller-owned device memory
 * and nothing is allocated. Stream-ordered and asynchronous. Returns C128_ERR_ARG (bad sizes or
 * launch shape), C128_ERR_NULL_PTR, C128_ERR_ALIGN or C128_ERR_CUDA; bytes == 0 is a no-op. */
int c128_read_probe(const void* buf, int64_t bytes, int32_t threads_per_cta, int32_t ctas_per_sm,
                    int32_t loads_in_flight, uint32_t* xor_out, c128_stream_t stream);

/* Free every workspace and timer the library holds, on every device it was used on
 * (synchronises those devices). */
int c128_release_all(void);

#ifdef __cplusplus
}
#endif
#endif /* C128COMPRESS_H */
