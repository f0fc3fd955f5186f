/*
 * csa2.h - C ABI of the GB300 (sm_103a) CSA2 index + sparse-attention step.
 *
 * The step (one query per decode request, or many queries sharing one cache):
 *   1. csa2_quantize_append  - KV append: RoPE then FP4 (E2M1, one E4M3 scale
 *                              per 16 channels) for the main latent; FP4 for
 *                              indexer K/Q rows; FP8 E4M3 for window latents.
 *   2. csa2_index_full       - Full layer: score every visible entry, keep the
 *                              top pool blocks of 8 by block maximum, and pick
 *                              the top-k positions.
 *   3. csa2_index_reindex    - Reindex layer: re-score only the pool's
 *                              positions with this layer's own indexer query.
 *      (csa2_index_full_bf16 / csa2_index_reindex_bf16 take the indexer
 *      query as bf16 and quantize it themselves, saving its FP4 append.)
 *      (Reuse layers make no call: they pass the previous top-k buffer again.)
 *   4. csa2_sparse_attn      - 64-head attention over the selected FP4 latents
 *                              plus the FP8 sliding window, one merged softmax.
 *
 * Sources, four secondary web pages about DeepSeek-V4.1-Flash:
 *   [T1] "DeepSeek V4.1-Flash 为什么这么强？CED 与 CSA2 架构全拆解"
 *   [T2] the blog post "DeepSeek V4.1 Flash vs V4 Pro"
 *   [T3] "DeepSeek-V4.1-Flash：全局 KV 仅 890 B/token，百万上下文怎么做成的？"
 * The pages fix formats, shapes and modes but no formula; the score, the
 * rounding and every memory layout below are this library's definitions.
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     allocates nothing.  Data pointers must be 16-byte aligned.
 *   - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream).
 *   - Argument errors are detected on the host and return before any launch
 *     (CSA2_ERR_INVALID_ARG / CSA2_ERR_UNSUPPORTED / CSA2_ERR_WORKSPACE).  A
 *     launch failure returns CSA2_ERR_CUDA.
 *   - Values only the device can see (rows, positions, indices held in device
 *     arrays) are checked by the kernels: an offending item is skipped and the
 *     first problem is recorded in the status word at the start of `ws`
 *     (read it with csa2_status_fetch).  No kernel traps or asserts.
 *   - `ws` is caller-provided scratch of csa2_workspace_bytes(...) bytes.  Its
 *     first 256 bytes hold the status word; zero them once with
 *     csa2_status_reset.  Calls sharing one `ws` must be stream-ordered.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int csa2_status;
enum {
    CSA2_OK = 0,
    CSA2_ERR_INVALID_ARG = 1,   /* null pointer, misalignment, bad size      */
    CSA2_ERR_UNSUPPORTED = 2,   /* a shape or format this library does not run */
    CSA2_ERR_CUDA = 3,          /* a CUDA launch or runtime error             */
    CSA2_ERR_TIMEOUT = 4,       /* device: a bounded wait gave up             */
    CSA2_ERR_DEVICE_BOUNDS = 5, /* device: a row/index outside its bounds was skipped */
    CSA2_ERR_WORKSPACE = 6      /* ws smaller than csa2_workspace_bytes()     */
};

/* Shapes fixed by the pages ([T1] §二, layout paragraph; [T1] 层级化稀疏索引器). */
#define CSA2_INDEX_HEADS 32   /* indexer query heads                        */
#define CSA2_INDEX_DIM 128    /* indexer head dim                           */
#define CSA2_ATTN_HEADS 64    /* main attention heads                       */
#define CSA2_LATENT_DIM 512   /* shared main latent (K = V)                 */
#define CSA2_BLOCK 8          /* positions per pool block                   */
#define CSA2_STATUS_BYTES 256 /* status area at the start of every ws       */

/* Formats and layouts for csa2_quantize_append. */
enum { CSA2_FMT_FP4 = 0, CSA2_FMT_FP8 = 1 };
/*
 * CSA2_LAYOUT_ROWS: FP4 codes row-major, codes[row][dim/2] (two codes per
 *   byte, even channel in the low nibble), scales[row][dim/16] (E4M3 bytes).
 *   FP8: bytes[row][dim].  Used for the main latent and the window latents.
 * CSA2_LAYOUT_BLOCK8 (FP4, dim 128 only): rows in blocks of 8; the 64 code
 *   bytes of row r sit at byte (r/8)*512 + c*128 + (r%8)*16 + j for byte
 *   b = 16c + j of the row (c = 0..3).  Scales stay row-major [row][8].  Used
 *   for indexer K and indexer Q: a block of 8 rows is 512 contiguous bytes
 *   holding four 8-row x 16-byte tiles, the shape tensor cores read.
 * CSA2_LAYOUT_BLOCK8R (FP4, dim 128 only): BLOCK8 with each block's scales
 *   beside its codes: block b of 8 rows is a 576-byte record at byte 576*b,
 *   its 512 code bytes as in BLOCK8 followed by the 8 rows x 8 scale bytes
 *   (row r's scale byte g at 576*(r/8) + 512 + (r%8)*8 + g).  dst_scales
 *   must be NULL.  Used for indexer K: a block the index gathers is then one
 *   contiguous read instead of two.
 */
enum { CSA2_LAYOUT_ROWS = 0, CSA2_LAYOUT_BLOCK8 = 1, CSA2_LAYOUT_BLOCK8R = 2 };

/* Output element type of csa2_sparse_attn. */
enum { CSA2_OUT_BF16 = 0, CSA2_OUT_F32 = 1 };

/* Operation ids for csa2_workspace_bytes. */
enum { CSA2_OP_APPEND = 0, CSA2_OP_INDEX_FULL = 1, CSA2_OP_INDEX_REINDEX = 2, CSA2_OP_SPARSE_ATTN = 3 };

typedef void* csa2_stream_t; /* a cudaStream_t */

/* ABI version (increments on any signature change). */
int csa2_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* csa2_status_string(csa2_status status);

/*
 * Bytes of workspace an operation needs for n_q queries whose visible entry
 * counts are at most max_visible, with pool_blocks pool blocks and topk
 * selections.  Always >= CSA2_STATUS_BYTES.  Returns 0 for bad arguments.
 */
size_t csa2_workspace_bytes(int op, int64_t n_q, int32_t max_visible, int pool_blocks, int topk);

/* Zero the status word of `ws` (stream-ordered). */
csa2_status csa2_status_reset(void* ws, csa2_stream_t stream);

/*
 * Copy the status area to host out[4] = {status, detail0, detail1, detail2}
 * and synchronize `stream`.  out[0] is CSA2_OK or the first device-detected
 * problem (CSA2_ERR_DEVICE_BOUNDS: detail0 = which check, detail1 = the query
 * or row, detail2 = the offending value).
 */
csa2_status csa2_status_fetch(const void* ws, int32_t out[4], csa2_stream_t stream);

/*
 * RoPE tables.  [T1] §三 and [T3] 第三刀: the main latent is quantized after
 * RoPE.  Rotation of channel pair (2i, 2i+1) by p * theta^(-2i/dim), p the
 * 0-based position; the angle is split as p = hi*1024 + lo and the table
 * holds cos/sin of hi*1024*w_i and lo*w_i (computed in fp64, stored fp32),
 * combined on the device by angle addition.  The table covers positions
 * [0, max_pos).  csa2_rope_table_init fills a caller-allocated device buffer
 * of csa2_rope_table_bytes(dim, max_pos) bytes.
 */
size_t csa2_rope_table_bytes(int dim, int64_t max_pos);
csa2_status csa2_rope_table_init(float theta, int dim, int64_t max_pos, void* table,
                                 csa2_stream_t stream);

/*
 * KV append ([T1] §三; [T2] 黑科技之三; [T3] 第三刀).
 *   x_bf16     [n][dim] bf16 rows to append.
 *   fmt        CSA2_FMT_FP4: per group of 16 channels s = RNE_E4M3(amax/6)
 *              (saturating at 448), codes = nearest E2M1 of x/s, ties to the
 *              even code, saturating at 6, sign kept; s == 0 gives zero codes.
 *              CSA2_FMT_FP8: each element to E4M3 (nearest-even, saturating).
 *   layout     CSA2_LAYOUT_ROWS, or CSA2_LAYOUT_BLOCK8 / CSA2_LAYOUT_BLOCK8R
 *              (FP4, dim 128).
 *   dim        512 or 128 (FP4 and FP8 rows; BLOCK8 needs 128).
 *   pos        [n] int64 RoPE positions, or NULL for no RoPE.  Needs
 *              rope_table from csa2_rope_table_init for the same dim, covering
 *              rope_max_pos positions; a position outside [0, rope_max_pos)
 *              skips the row and records CSA2_ERR_DEVICE_BOUNDS.
 *   dst_row    [n] int64 destination rows, or NULL for rows 0..n-1.  A row
 *              outside [0, n_rows) is skipped and recorded.
 *   dst_codes  codes plane of n_rows rows (FP4), or the FP8 byte plane.
 *   dst_scales scales plane [n_rows][dim/16] (FP4), NULL for FP8 and for
 *              CSA2_LAYOUT_BLOCK8R (the scales sit in the records).
 *   n_rows     rows in the destination planes (BLOCK8: a multiple of 8).
 *   ws         at least CSA2_STATUS_BYTES bytes (status word).
 */
csa2_status csa2_quantize_append(const void* x_bf16, int64_t n, int dim, int fmt, int layout,
                                 const int64_t* pos, const void* rope_table, int64_t rope_max_pos,
                                 const int64_t* dst_row, int64_t n_rows,
                                 uint8_t* dst_codes, uint8_t* dst_scales,
                                 void* ws, size_t ws_bytes, csa2_stream_t stream);

/*
 * Full-layer hierarchical index ([T1] §二 mode table and 层级化稀疏索引器;
 * [T3] 第二刀, Fig. 5).  For query t with n = n_visible[t] entries at cache
 * rows kv_start[t] .. kv_start[t]+n-1:
 *   I(t,s) = sum_h w[t][h] * max(0, q~[t][h] . k~[s])  for s < n,
 * q~, k~ the dequantized FP4 indexer query and key.  Block b covers positions
 * [8b, 8b+8) (a partial last block uses its visible positions).
 *   out_pool[t][pool_blocks]: the top-min(pool_blocks, ceil(n/8)) blocks by
 *     block maximum, ties to the lower block, ascending, padded with -1.
 *   out_topk[t][topk]: the top-min(topk, n) positions by I over ALL visible
 *     positions, ties to the lower position, ascending, padded with -1.
 *     (Computed exactly by re-scoring the top-max(pool_blocks, topk) blocks,
 *     which contain every top-k position.)
 *   q_codes/q_scales: indexer Q, BLOCK8 layout, n_q*32 rows of 128 channels
 *     (row t*32+h is head h of query t).  w: [n_q][32] fp32.
 *   k_codes/k_scales: indexer K plane, n_rows rows: BLOCK8 codes and
 *     row-major scales, or (k_scales NULL) BLOCK8R records in k_codes.
 *   kv_start [n_q] int64 (multiples of 8), n_visible [n_q] int32, device.
 *   max_visible: host upper bound of n_visible (sizes the launch).
 *   pool_blocks in [1, 4096], topk in [1, 2048].
 * Checked on the device: kv_start % 8 == 0, 0 <= n_visible <= max_visible
 * and kv_start + n_visible <= n_rows; a failing query gets empty (-1) outputs.
 */
csa2_status csa2_index_full(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                            int64_t n_q, const uint8_t* k_codes, const uint8_t* k_scales,
                            int64_t n_rows, const int64_t* kv_start, const int32_t* n_visible,
                            int32_t max_visible, int pool_blocks, int topk,
                            int32_t* out_pool, int32_t* out_topk,
                            void* ws, size_t ws_bytes, csa2_stream_t stream);

/*
 * Reindex layer ([T1] §二 mode table; [T2] 黑科技之二; [T3] 第二刀): the same
 * score with this layer's own q, w against the shared indexer K, over the
 * positions of `pool` (a Full layer's out_pool, [n_q][pool_blocks], -1 pads
 * ignored) only; out_topk[t][topk] = the top-min(topk, |pool positions|)
 * positions, ties to the lower position, ascending, padded with -1.
 * Other arguments as in csa2_index_full.  A pool entry outside
 * [0, ceil(n/8)) is skipped and recorded.
 */
csa2_status csa2_index_reindex(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                               int64_t n_q, const uint8_t* k_codes, const uint8_t* k_scales,
                               int64_t n_rows, const int64_t* kv_start, const int32_t* n_visible,
                               int32_t max_visible, const int32_t* pool, int pool_blocks, int topk,
                               int32_t* out_topk, void* ws, size_t ws_bytes, csa2_stream_t stream);

/*
 * csa2_index_full and csa2_index_reindex with the indexer query given as
 * bf16 rows, q_bf16 [n_q*32][128] (row t*32+h is head h of query t, 16-byte
 * aligned), instead of FP4 codes and scales.  The query is quantized to FP4
 * (E2M1, one E4M3 scale per 16 channels; [T1] 层级化稀疏索引器, [T3] 第二刀:
 * the indexer runs in FP4) inside the call, exactly as csa2_quantize_append
 * with CSA2_FMT_FP4 would, so the results are those of the FP4 calls on that
 * quantization.  Decode batches (fewer than 256 queries) and every Reindex
 * call quantize it in the scoring kernels' prologue, which saves the
 * separate quantization launch; a many-query Full call quantizes it into
 * its workspace first (the workspace size is the same as the FP4 call's).
 * Other arguments, results and errors as in the FP4 calls.
 */
csa2_status csa2_index_full_bf16(const void* q_bf16, const float* w, int64_t n_q, const uint8_t* k_codes,
                                 const uint8_t* k_scales, int64_t n_rows, const int64_t* kv_start,
                                 const int32_t* n_visible, int32_t max_visible, int pool_blocks, int topk,
                                 int32_t* out_pool, int32_t* out_topk, void* ws, size_t ws_bytes,
                                 csa2_stream_t stream);
csa2_status csa2_index_reindex_bf16(const void* q_bf16, const float* w, int64_t n_q, const uint8_t* k_codes,
                                    const uint8_t* k_scales, int64_t n_rows, const int64_t* kv_start,
                                    const int32_t* n_visible, int32_t max_visible, const int32_t* pool,
                                    int pool_blocks, int topk, int32_t* out_topk, void* ws, size_t ws_bytes,
                                    csa2_stream_t stream);

/*
 * csa2_index_reindex without a workspace, for callers that cannot allocate
 * device memory: runtimes without a device allocator, callers whose memory
 * is fixed before the model starts, or code running where cudaMalloc is not
 * permitted.  The pages describe nothing like it; it exists only for such
 * callers.  Arguments and results are those of csa2_index_reindex, except:
 *   - the per-position scores go to one library-owned device array of 2 MiB
 *     (held by every GPU that loads the library until the process exits):
 *     n_q * 8 * pool_blocks must be at most 524,288, else the call returns
 *     CSA2_ERR_UNSUPPORTED without launching (e.g. 32 queries at 2048 pool
 *     blocks);
 *   - status: a caller-owned device int32[4] that receives the first
 *     device-detected problem (as the status word of a workspace), or NULL.
 *     It is not cleared by the call.
 * The first call on a device looks up the array's device address (one
 * runtime query); make that first call before any stream capture.  Every
 * call shares the array, whose contents are fully rewritten by each call;
 * calls that overlap on the GPU (other streams, other threads) race on it.
 * The call allocates nothing.
 */
csa2_status csa2_index_reindex_noalloc(const uint8_t* q_codes, const uint8_t* q_scales,
                                       const float* w, int64_t n_q, const uint8_t* k_codes,
                                       const uint8_t* k_scales, int64_t n_rows,
                                       const int64_t* kv_start, const int32_t* n_visible,
                                       int32_t max_visible, const int32_t* pool, int pool_blocks,
                                       int topk, int32_t* out_topk, int32_t* status,
                                       csa2_stream_t stream);

/*
 * Sparse attention with one merged softmax ([T1] §二: 64 heads over a
 * 512-dim latent, every layer has its own Q and window KV; [T3] 第三刀: FP4
 * main KV dequantized before attention, window kept in FP8).  For query t,
 * head h, with E = {selected entries} U {window entries} (no dedup):
 *   l_j = sm_scale * q[t][h] . c_j,  p = softmax over E,  o[t][h] = sum p_j c_j
 * where selected entry j is main-KV row kv_start[t] + topk[t][j] (FP4,
 * dequantized; -1 pads skipped) and the window is the last min(window, n)
 * positions p of the query, read from swa[t][p mod window] (E4M3).
 *   q_bf16   [n_q][64][512] bf16.
 *   kv_codes [n_rows][256], kv_scales [n_rows][32]: main latent, ROWS layout.
 *   topk     [n_q][k] int32 positions (a Full/Reindex layer's out_topk).
 *   swa      [n_q][window][512] E4M3 ring (slot = position mod window).
 *   swa_new_bf16  [n_q][512] bf16 window latent of each query's current
 *            token (position n-1), or NULL.  When given, the kernel rounds it
 *            to E4M3 exactly as csa2_quantize_append (CSA2_FMT_FP8) would,
 *            stores it to ring slot (n-1) mod window and uses it: the
 *            window append fused into the attention call.
 *   window   0..128.
 *   out      [n_q][64][512], bf16 (out_dtype CSA2_OUT_BF16) or fp32
 *            (CSA2_OUT_F32); the result is rounded once, from fp32.  bf16's
 *            unit roundoff is 2^-8, so the fp32 form carries the kernels'
 *            own accuracy (about 1e-6 relative).
 *   out_lse  [n_q][64] fp32 natural-log log-sum-exp of the scaled logits,
 *            or NULL.
 * An empty E gives zeros and lse = -inf.  A topk entry outside [-1, n) is
 * skipped and recorded.
 */
csa2_status csa2_sparse_attn(const void* q_bf16, int64_t n_q,
                             const uint8_t* kv_codes, const uint8_t* kv_scales, int64_t n_rows,
                             const int64_t* kv_start, const int32_t* n_visible,
                             const int32_t* topk, int k, uint8_t* swa, const void* swa_new_bf16,
                             int window, float sm_scale, void* out, int out_dtype, float* out_lse,
                             void* ws, size_t ws_bytes, csa2_stream_t stream);

/*
 * Prefill sparse attention over a shared sequence ([T1] §二 layout paragraph:
 * the encoder runs CSA2 at m = 2 in groups of one Full and five Reuse
 * layers, over a prefill chunk of many query tokens).  As csa2_sparse_attn,
 * except that each query's window is its own causal window over the
 * sequence the queries share: the last min(window, n) positions p < n of
 * query t, read from
 *   swa_rows [n_rows][512] E4M3, row kv_start[t] + p
 * (the same row numbering as the main latent; one array per layer, written
 * with csa2_quantize_append CSA2_FMT_FP8), instead of a ring per query.
 * There is no current-token append.  The workspace is that of
 * csa2_sparse_attn (CSA2_OP_SPARSE_ATTN).
 */
csa2_status csa2_sparse_attn_prefill(const void* q_bf16, int64_t n_q,
                                     const uint8_t* kv_codes, const uint8_t* kv_scales, int64_t n_rows,
                                     const int64_t* kv_start, const int32_t* n_visible,
                                     const int32_t* topk, int k, const uint8_t* swa_rows, int window,
                                     float sm_scale, void* out, int out_dtype, float* out_lse,
                                     void* ws, size_t ws_bytes, csa2_stream_t stream);

/*
 * Instrumentation (off by default; the compute path never depends on it).
 * csa2_launch_count: kernels launched through the library by this process.
 * csa2_timer_enable: bracket the next max_launches launches of kernel
 *   `kernel_id` (0 scan_blockmax, 1 select_blocks, 2 pool_score,
 *   3 select_topk, 4 attn_split (either attention kernel), 5 attn_merge, 6 quantize_fp4,
 *   7 quantize_fp8, 8 rope_table) with CUDA events on their stream.  Not for
 *   use during stream capture.
 * csa2_timer_read: wait for those events, return the summed device time and
 *   the number of launches timed, and switch the timer off.
 */
int64_t csa2_launch_count(void);

/*
 * Test hook for the device give-up paths.  Every wait of a library kernel on
 * a barrier (copies arriving, MMAs completing) is bounded: after 2 s it
 * records CSA2_ERR_TIMEOUT in the status word, stops issuing work, waits for
 * the copies and MMAs it already started, and returns.  csa2_debug_wait_limit
 * sets that limit (in nanoseconds) for kernels launched afterwards, on every
 * device (it is a launch argument: a graph captured earlier keeps the limit
 * it was captured with); 0 restores 2 s.  A limit under 1 ms makes every
 * bounded wait give up at once, so a test can check the status, that the
 * copies and MMAs in flight were waited for, and that the next normal call
 * is correct.  Not for production use and not during stream capture.
 */
csa2_status csa2_debug_wait_limit(int64_t ns);
const char* csa2_kernel_name(int kernel_id);
csa2_status csa2_timer_enable(int kernel_id, int max_launches);
csa2_status csa2_timer_read(int kernel_id, double* total_ms, int32_t* launches);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
