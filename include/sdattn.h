/*
 * sdattn.h - C ABI of the GB300 (sm_103a) DSA sparse decode attention library.
 *
 * The operation is the one of the vLLM API page
 * "vllm.models.step5.nvidia.ops.sparse_decode_attention" (function
 * `sparse_decode_attention` and its module docstring): for every
 * (token, KV group) row, all query heads of that group attend over only the
 * row's selected KV regions, read in place from a paged cache through
 * block_table, with FP8 dequantised, tokens past the row's position masked,
 * split-KV partials merged through their log-sum-exp, an optional headwise
 * sigmoid gate applied with bf16 rounding (the page's `_gate`), and inactive
 * rows cleared.
 *
 * Conventions for every entry point:
 *   - Pointers inside `sda_tensor` are DEVICE pointers of the current CUDA
 *     device; shapes and strides are in elements (not bytes).
 *   - The caller owns every buffer.  The library allocates no device memory,
 *     never synchronises the stream (except sparse_decode_read_errors) and
 *     returns a status instead of aborting.  A launch is asynchronous: results
 *     are valid once the stream has reached that point.
 *   - Inputs are read only; only `output` and `workspace` are written, and
 *     neither may overlap an input.
 */
#ifndef SDATTN_H
#define SDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SDA_OK = 0,
    SDA_ERR_INVALID = 1,      /* an argument breaks the documented contract            */
    SDA_ERR_UNSUPPORTED = 2,  /* well formed, but outside what the kernels handle      */
    SDA_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small            */
    SDA_ERR_CUDA = 4,         /* a CUDA runtime or driver call failed                  */
    SDA_ERR_TIMEOUT = 5,      /* device flag: a bounded wait inside a kernel gave up   */
    SDA_ERR_BOUNDS = 6        /* device flag: an index read from the inputs was bad    */
} sda_status;

typedef enum {
    SDA_DTYPE_BF16 = 1,
    SDA_DTYPE_FP8_E4M3 = 2,   /* OCP E4M3 "fn" (finite, bias 7)                        */
    SDA_DTYPE_UINT8 = 3,      /* raw bytes; an FP8 cache may be passed as uint8        */
    SDA_DTYPE_INT32 = 4,
    SDA_DTYPE_BOOL = 5,       /* one byte, nonzero = true                              */
    SDA_DTYPE_FP32 = 6
} sda_dtype;

/* A strided view of device memory.  Unused trailing shape/stride entries are
 * ignored.  `data` may be NULL only where an argument is documented optional. */
typedef struct {
    const void *data;
    int32_t dtype;            /* sda_dtype */
    int32_t ndim;
    int64_t shape[4];
    int64_t stride[4];        /* in elements */
} sda_tensor;

/* Device error flags accumulated in the workspace header (bit values). */
#define SDA_FLAG_BOUNDS  0x1u  /* a region id < -1, a table column past the table width, or a
                                  table entry outside [0, pages) was met; that piece was skipped */
#define SDA_FLAG_TIMEOUT 0x2u  /* a pipeline wait exceeded its limit; the row's output is invalid */

/*
 * Split count per row: start at 1 and double while below 32 and
 * rows * splits * 2 <= 256, i.e. about 256 split programs per call.
 * Follows `sparse_decode_splits` on the page named above (the split cannot
 * follow context length because CUDA graphs are captured per batch size).
 * rows < 0 returns 1.
 */
int sparse_decode_splits(int rows);

/*
 * Bytes of workspace `sparse_decode_attention` needs for `rows` rows of
 * `heads` heads with `splits` splits: a 256-byte header (device error flags)
 * plus, when splits > 1, fp32 partial outputs [rows*splits*heads, 192] and
 * fp32 log-sum-exps [rows*splits*heads] (the page's `partial` and `lse`).
 * Returns 0 for arguments out of range.
 */
size_t sparse_decode_workspace_bytes(int rows, int heads, int splits);

/*
 * Sparse decode attention (page above, function `sparse_decode_attention`).
 *
 *   query        [rows, H, 192] bf16, stride[2] == 1, H in 1..16.
 *                rows = tokens * G; row r is KV group r % G of token r / G.
 *   cache        [pages, G, B, 384] bf16, FP8_E4M3 or UINT8 (E4M3 bytes);
 *                K in elements 0..191 and V in 192..383 of a token's row.
 *                stride[3] == 1; any page / group / token strides whose byte
 *                sizes are multiples of 16 (and a 16-byte aligned base).
 *   regions      [rows, R] int32, stride[1] == 1, R <= 16384 (else
 *                SDA_ERR_UNSUPPORTED).  Region ids of the row, any order; -1
 *                marks an unused slot.  Id `id` covers the request's logical
 *                tokens [id*RT, (id+1)*RT), RT = region_tokens.
 *   block_table  [requests, W] int32, stride[1] == 1.  Logical block c of
 *                request q lives in page block_table[q, c].  The G*query_len
 *                consecutive rows of one request share its table row:
 *                request = r / (G * query_len).
 *   positions    [rows] int32: the row's token position (0-based); a token t
 *                is visible iff t <= position.
 *   active       [rows] BOOL or UINT8: zero rows are not computed; with
 *                clear_inactive their output is written as +0.0.
 *   output       [rows, H, 192] bf16, stride[2] == 1 (written).
 *   scale        softmax scale applied to q.k (e.g. 1/sqrt(192)).
 *   query_len    tokens per request (>= 1).
 *   splits       split-KV programs per row, 1..64 (see sparse_decode_splits).
 *                Each split takes a contiguous chunk [s*n/S, (s+1)*n/S) of the
 *                row's live regions; splits > 1 adds the combine kernel.
 *   k_scale, v_scale  device fp32 scalars; required for an FP8 cache, ignored
 *                for bf16.  K = decode(byte) * k_scale, V = decode(byte) * v_scale.
 *   gate         NULL (or data == NULL) for no gate, else [tokens, G*H] bf16:
 *                head h of row r is multiplied by bf16(sigmoid(gate[r/G,
 *                (r%G)*H + h])) computed in fp32 (the page's `_gate`).
 *   clear_inactive  nonzero: inactive rows are written as +0.0; zero: left as is.
 *                (The adapter page's decode path passes clear_inactive || gate,
 *                so gated layers always clear; that policy is the caller's.)
 *   region_tokens   RT; 0 means RT = B.  min(RT, B, 64) must be a multiple of 8
 *                and divide both RT and B.
 *   workspace    device buffer of >= sparse_decode_workspace_bytes(rows, H,
 *                splits) bytes, 256-byte aligned; its first 4 bytes are error
 *                flags the kernels OR into (zero them once before first use;
 *                see sparse_decode_read_errors).  Calls that overlap on the
 *                GPU must not share a workspace.
 *   stream       cudaStream_t (NULL = legacy default stream).
 *
 * Returns SDA_OK after enqueueing the kernels (rows == 0 enqueues nothing),
 * SDA_ERR_INVALID / SDA_ERR_UNSUPPORTED / SDA_ERR_WORKSPACE without touching
 * the GPU, or SDA_ERR_CUDA when a launch failed.  Device-side problems are
 * reported through the workspace flags, never by a trap.
 *
 * FP8 note: the kernels convert E4M3 to fp16 exactly; the two NaN codes
 * (S.1111.111) are not meaningful cache contents and are not special-cased.
 * The FP8 path multiplies in fp16: each row's q is first scaled by a power of
 * two that puts its largest |q| in [2^14, 2^15), and the factor is undone in
 * the fp32 logit scale, so any finite bf16 query is taken at full precision
 * (values more than 2^31 below the row's largest lose low bits) as long as
 * the logits scale * q.k * k_scale fit in fp32.
 */
sda_status sparse_decode_attention(const sda_tensor *query, const sda_tensor *cache,
                                   const sda_tensor *regions, const sda_tensor *block_table,
                                   const sda_tensor *positions, const sda_tensor *active,
                                   const sda_tensor *output, float scale, int query_len,
                                   int splits, const float *k_scale, const float *v_scale,
                                   const sda_tensor *gate, int clear_inactive, int region_tokens,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * Split count for the sliding-window decode below (a reading of its own: the
 * page's `swa_decode_plan` body is not shown).  Starts from
 * sparse_decode_splits(rows) and halves while a split would cover fewer than
 * 256 window tokens.
 */
int sparse_decode_swa_splits(int rows, int window);

/*
 * Gated sliding-window decode over the same packed cache: the non-DSA layers'
 * fused path of the vLLM page "vllm.models.step5.nvidia.sparse_attention"
 * (`Step5SplitKVFlashAttentionImpl.forward_with_headwise_gate`, which calls
 * `swa_decode_gated` with window = sliding_window[0] + 1, GQA packing and a
 * split window, bf16, query_len <= 4 there).
 *
 *   query, cache, block_table, output, scale, query_len, splits, k_scale,
 *   v_scale, gate, workspace, stream: as in sparse_decode_attention
 *                (rows = tokens * G; FP8 caches are accepted as well).
 *   seq_lens     [requests] int32: tokens of each request including the ones
 *                being decoded.  Token j of request q sits at position
 *                p = seq_lens[q] - query_len + j and attends over the `window`
 *                tokens [max(0, p - window + 1), p] of its request (none when
 *                p < 0: zeros).
 *   window       >= 1 (at most 2^30).
 * Every row is active.  The window is walked in pieces of min(B, 64) (FP8) or
 * min(B, 32) (bf16) tokens, which must be a multiple of 8 dividing B.  Splits
 * take contiguous chunks of the window's pieces.  Errors as for
 * sparse_decode_attention.
 */
sda_status sparse_decode_swa_attention(const sda_tensor *query, const sda_tensor *cache,
                                       const sda_tensor *block_table, const sda_tensor *seq_lens,
                                       const sda_tensor *output, float scale, int window, int query_len,
                                       int splits, const float *k_scale, const float *v_scale,
                                       const sda_tensor *gate, void *workspace, size_t workspace_bytes,
                                       void *stream);

/*
 * Region selection for decode rows: the step before sparse_decode_attention
 * on the vLLM page "vllm.models.step5.nvidia.flashinfer_sparse"
 * (`select_and_run_decode_attention` calls `select_regions(scores, current,
 * topk, topk_lengths=..., sort=False)`; its body is not on the page, so the
 * rule below is a reading).
 *
 *   scores        [rows, N] fp32, stride[1] == 1: a score per region id.
 *   current       [rows] int32: the region holding the row's own token; it is
 *                 always kept when 0 <= current < length.
 *   topk_lengths  [rows] int32 or NULL (every row has N candidates): the row
 *                 considers region ids [0, min(length, N)).
 *   topk          regions per row (>= 1).
 *   regions       [rows, topk] int32, stride[1] == 1 (written): the current
 *                 region first, then the topk - 1 best-scoring other
 *                 candidates in ascending id order, then -1 padding.  NaN
 *                 scores rank lowest; equal scores go to the lower id.
 * No workspace; returns SDA_ERR_INVALID for shapes, dtypes or strides outside
 * this contract, SDA_ERR_CUDA if the launch failed.
 */
sda_status sparse_decode_select_regions(const sda_tensor *scores, const sda_tensor *current,
                                        const sda_tensor *topk_lengths, int topk,
                                        const sda_tensor *regions, void *stream);

/*
 * Indexer decode scores: a score per 8-token region for every (token, KV
 * group) row, the input of sparse_decode_select_regions.  The adapter page
 * "vllm.models.step5.nvidia.flashinfer_sparse" computes this in
 * `decode_logits` (fast path `decode_summary_scores`, for FP8 queries of 8
 * heads x 256 and uint8 summaries [*, G, 256]) through an FP8 paged
 * MQA-logits kernel whose formula is not on the page; the reading taken is
 *     score[row, j] = sum_h weights[token, g, h] * max(0, <q_h, m_j>)
 * over the 8 index heads h, with q_h = query[token, g, h, :] and m_j the
 * summary of region j of group g, both decoded from E4M3 (no scale), the
 * product accumulated in fp32.
 *
 *   query        [tokens, G, 8, 256] FP8 E4M3 (or uint8 holding E4M3 bytes);
 *                stride[3] == 1, stride[2] == 256, stride[0] and stride[1]
 *                multiples of 16, base 16-byte aligned.  Row r = t * G + g.
 *   weights      [tokens, G, 8] fp32, stride[2] == 1.
 *   summaries    [slots, G, 256] FP8 E4M3 / uint8, stride[2] == 1,
 *                stride[1] == 256, stride[0] a multiple of 16, base 16-byte
 *                aligned.  Slot page * (block_size / 8) + k holds the summary
 *                of tokens [8k, 8k + 8) of that page.
 *   block_table  [reqs, W] int32, stride[1] == 1: the request's pages.
 *   seq_lens     [>= reqs] int32: request lengths; the query_len tokens of
 *                request q are tokens q * query_len + i at position
 *                seq_lens[q] - query_len + i.
 *   block_size   tokens per page, a multiple of 8.
 *   query_len    tokens per request, 1..4; tokens must be a multiple of it.
 *   scores       [tokens * G, N] fp32, stride[1] == 1 (written): columns
 *                j < min(pos / 8 + 1, N) hold the score of region j, the
 *                rest -inf (all -inf when pos < 0).  Region j's page is
 *                block_table[req, 8j / block_size].
 *   current      [tokens * G] int32 or NULL (written): pos / 8, -1 if pos < 0.
 *   lengths      [tokens * G] int32 or NULL (written): the number of scored
 *                columns, min(pos / 8 + 1, N) (0 if pos < 0).
 *   workspace    NULL, or >= 256 bytes, 256-byte aligned: receives
 *                SDA_FLAG_BOUNDS when a scored region's table column is past
 *                W or its page has no slots in `summaries` (that region
 *                scores -inf); read it with sparse_decode_read_errors.
 * Every summary is read from HBM once per (request, group): the query_len
 * tokens share it.  Returns SDA_ERR_INVALID for shapes, dtypes or strides
 * outside this contract, SDA_ERR_UNSUPPORTED for query_len > 4 or
 * misaligned operands, SDA_ERR_WORKSPACE for a bad workspace, SDA_ERR_CUDA if
 * the launch failed; tokens == 0 returns SDA_OK with no launch.
 */
sda_status sparse_decode_summary_scores(const sda_tensor *query, const sda_tensor *weights,
                                        const sda_tensor *summaries, const sda_tensor *block_table,
                                        const sda_tensor *seq_lens, int block_size, int query_len,
                                        const sda_tensor *scores, const sda_tensor *current,
                                        const sda_tensor *lengths, void *workspace,
                                        size_t workspace_bytes, void *stream);

/*
 * Reads the device error flags (SDA_FLAG_*) from a workspace into *flags,
 * optionally clearing them.  Synchronises `stream` (it must be the stream the
 * calls ran on).  Returns SDA_ERR_CUDA if a CUDA call failed.
 */
sda_status sparse_decode_read_errors(const void *workspace, uint32_t *flags, int clear, void *stream);

/*
 * Upper bound in nanoseconds for every pipeline wait inside the kernels
 * (default 1e9).  A wait that runs out sets SDA_FLAG_TIMEOUT, stops the row,
 * lets in-flight copies land and returns.  Applies to launches made after the
 * call, process-wide.  Meant for failure-detection tests.
 */
void sparse_decode_set_wait_limit_ns(uint64_t ns);

/*
 * Allocation-free variant of sparse_decode_attention.  The page has no
 * counterpart for it.
 *
 * For callers that cannot obtain device memory for a workspace: plugin or
 * FFI hosts that are handed tensor pointers by another runtime but no
 * allocator, and code that must not call cudaMalloc while other work is in
 * flight (an allocation can synchronise the device).  Arguments and results
 * are those of sparse_decode_attention without `workspace` /
 * `workspace_bytes`: the scratch (flag header, split partials and LSEs) lives
 * in an 8 MiB static device array inside the library, which every GPU that
 * loads the library holds until the process exits.
 *   - Limit: sparse_decode_workspace_bytes(rows, H, splits) must be at most
 *     8 MiB (8388608), else SDA_ERR_WORKSPACE is returned and nothing is
 *     enqueued.  splits == 1 needs 256 bytes, so any row count fits; with
 *     16 heads, rows * splits up to 679 fits.  Arguments outside the contract
 *     get the statuses of sparse_decode_attention, checked first, also with
 *     nothing enqueued.
 *   - The first call on a device (of this function or of
 *     sparse_decode_no_alloc_read_errors) looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and zeroes its flag
 *     header with an async memset on `stream`; make that first call before
 *     any stream capture on the device.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents.  Calls whose kernels overlap on the GPU (different
 *     streams, no ordering between them) race on it: serialise them.
 *   - Device flags (SDA_FLAG_*) collect in the array's header over calls, as
 *     in a caller's workspace; read and clear them with
 *     sparse_decode_no_alloc_read_errors.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 */
sda_status sparse_decode_attention_no_alloc(const sda_tensor *query, const sda_tensor *cache,
                                            const sda_tensor *regions, const sda_tensor *block_table,
                                            const sda_tensor *positions, const sda_tensor *active,
                                            const sda_tensor *output, float scale, int query_len,
                                            int splits, const float *k_scale, const float *v_scale,
                                            const sda_tensor *gate, int clear_inactive,
                                            int region_tokens, void *stream);

/*
 * The device flags of sparse_decode_attention_no_alloc on the current device
 * (the page has no counterpart): as sparse_decode_read_errors on the static
 * array's header.  Synchronises `stream`, which must be ordered after the
 * calls whose flags are wanted; with `clear` the header is zeroed afterwards.
 * Returns SDA_ERR_INVALID for a NULL `flags`, SDA_ERR_CUDA if a CUDA call
 * failed.
 */
sda_status sparse_decode_no_alloc_read_errors(uint32_t *flags, int clear, void *stream);

/*
 * Diagnostic builds only (the library compiled with SDA_TIMELINE): registers a
 * device buffer of at least 83886080 bytes (10 x 2^20 uint64) into which the
 * split and combine kernels of later launches write %globaltimer stamps (ns) at
 * their phase boundaries: split CTA u at entries u * 8 + k (k = 0 start, 1 the
 * consumers released with the row's live regions, 2 first K|V stage landed, 3
 * stage loop done, 4 output writes start, 5 done), combine CTA r at entries
 * 2^23 + r * 2 + k (k = 0 start, 1 past its wait on the split kernel).  NULL
 * stops the stamps.  Not thread-safe, synchronous.  The regular library returns
 * SDA_ERR_UNSUPPORTED and does nothing; its kernels carry no stamps.  No
 * counterpart on the pages: it is a measurement aid.
 */
sda_status sparse_decode_timeline_buffer(void *buffer, size_t bytes);

/* A static description of a status code. */
const char *sparse_decode_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SDATTN_H */
