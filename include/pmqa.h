/*
 * pmqa.h -- C ABI of libpmqa: the FP8 paged MQA-logits indexer and its per-row
 * top-k, the non-paged (prefill) MQA logits, and the sparse MLA decode that
 * consumes the top-k positions, as hand-written CUDA kernels for sm_103a
 * (GB300).
 *
 * What is computed. Sources: the page "[Bug] aiter ops triton attention pa"
 * (stepcodex.com issue mirror), section "Minimal reproduction" (the reference
 * function `torch_ref` and the `test` driver); the page "[Bugfix][Hardware][AMD]
 * Fix last_page_len calculation in AITER MLA decode" (vLLM PR 31282), section
 * "Comparison with Other Backends" (tokens held by a request's last page).
 *
 *   For request i < bs, draft row j < next_n (row r = i*next_n + j) and
 *   logical token t:
 *     valid(r, t)  <=>  t < ctx_i  and  t <= ctx_i - next_n + j
 *     phys         =   block_tables[i][t / P] * P + t % P
 *     k_t          =   kv_cache[phys][0..127] as fp8 e4m3fn
 *     s_t          =   fp32 whose little-endian bytes are kv_cache[phys][128..131]
 *     logits[r][t] =   sum_h weights[r][h] * relu(s_t * dot(q[i][j][h], k_t))
 *                      if valid(r, t), else -inf, for 0 <= t < max_model_len
 *   Top-k of row r: the positions of the min(k, valid_len(r)) largest logits
 *   among t < valid_len(r) = clamp(ctx_i - next_n + j + 1, 0, ctx_i); remaining
 *   slots hold -1. The order of positions within a row is unspecified; among
 *   equal values any choice is returned. The last page of a request holds
 *   ((ctx_i - 1) mod P) + 1 tokens; its other slots are never read.
 *
 * Memory. Every pointer is a DEVICE pointer owned by the caller. The library
 * allocates nothing, keeps no global state between calls (the one exception is
 * the built-in scratch of pmqa_logits_topk_noalloc), never synchronises the
 * stream (except pmqa_read_device_status) and enqueues its work on the given
 * stream. Calls that share one workspace must not overlap on the GPU.
 *
 * Errors. Functions return PMQA_OK (0) or a negative PMQA_ERR_* code; on an
 * error nothing has been enqueued. Faults the host cannot see (a block table
 * entry outside the pool, a context longer than max_model_len or than the
 * table covers, a pipeline wait that ran out) never trap: the kernel skips the
 * access (a bad table entry reads as zeros), records a PMQA_DEV_* bit in the
 * workspace status word and finishes; pmqa_read_device_status reports it.
 */
#ifndef PMQA_H
#define PMQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *pmqa_stream_t;

enum {
    PMQA_OK = 0,
    PMQA_ERR_INVALID_ARG = -1,  /* null pointer, negative size, misalignment, k < 1 */
    PMQA_ERR_UNSUPPORTED = -2,  /* head_dim != 128, heads not in {16,32,64,128},
                                   next_n not in 1..4, k too large for the kernel */
    PMQA_ERR_WORKSPACE = -3,    /* workspace smaller than pmqa_workspace_bytes */
    PMQA_ERR_CUDA = -4,         /* a CUDA runtime call or a launch failed */
    PMQA_ERR_DEVICE = -5        /* reported by pmqa_read_device_status only */
};

/* Bits of the device status word. */
#define PMQA_DEV_BAD_BLOCK_ID 0x1u /* a block table entry outside [0, num_blocks) */
#define PMQA_DEV_BAD_CONTEXT 0x2u  /* ctx < 0, ctx > max_model_len, or ctx > P * max_blocks_per_seq;
                                      the kernel clamps it */
#define PMQA_DEV_TIMEOUT 0x4u      /* a pipeline wait exceeded its limit; results are invalid */
#define PMQA_DEV_OVERFLOW 0x8u     /* top-k candidate storage exceeded; results are invalid */
#define PMQA_DEV_INTERNAL 0x10u    /* a kernel found its shared memory misaligned and did no work;
                                      results are invalid */

/* Workspace-size selector for pmqa_workspace_bytes. For PMQA_OP_MQA_LOGITS (the
   prefill entry point) bs is the number of query rows m and the other sizes
   are ignored. */
enum { PMQA_OP_LOGITS = 0, PMQA_OP_TOPK = 1, PMQA_OP_LOGITS_TOPK = 2, PMQA_OP_MQA_LOGITS = 3 };

/*
 * One decode-step problem, in the argument order of the reference function
 * (q, kv_cache, weights, context_lens, block_tables, max_model_len) plus sizes.
 *   q             fp8 e4m3fn [bs, next_n, heads, head_dim], contiguous, 16-byte aligned
 *   kv_cache      uint8 [num_blocks, block_size, head_dim + 4], contiguous, 16-byte
 *                 aligned (rows are read as 16-byte aligned windows): per token
 *                 head_dim fp8 bytes then a little-endian fp32 scale
 *   weights       fp32 [bs * next_n, heads], contiguous, 16-byte aligned
 *   context_lens  int32 [bs]
 *   block_tables  int32 [bs, max_blocks_per_seq], row-major; only the first
 *                 ceil(ctx_i / block_size) entries of row i are read
 */
typedef struct pmqa_problem {
    const void *q;
    const void *kv_cache;
    const float *weights;
    const int32_t *context_lens;
    const int32_t *block_tables;
    int32_t bs;
    int32_t next_n;
    int32_t heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t max_blocks_per_seq;
    int32_t max_model_len;
    int64_t num_blocks;
} pmqa_problem;

/*
 * Bytes of device workspace an operation needs for rows = bs * next_n rows of
 * width max_model_len and top-k size k (k is ignored for PMQA_OP_LOGITS).
 * Returns 0 for invalid arguments. The workspace must be 256-byte aligned and
 * zero-filled before its first use (pmqa_workspace_init); every call leaves it
 * zero-filled again except for the status word.
 */
size_t pmqa_workspace_bytes(int32_t bs, int32_t next_n, int32_t max_model_len, int32_t k, int op);

/* Zero-fill a workspace (cudaMemsetAsync on the stream). */
int pmqa_workspace_init(void *ws, size_t ws_bytes, pmqa_stream_t stream);

/*
 * Logits, the definition above. logits: fp32 [bs * next_n, max_model_len],
 * 4-byte aligned; every entry of every row is written (-inf outside the mask),
 * so no caller pre-fill is needed.
 */
int pmqa_logits(const pmqa_problem *p, float *logits, void *ws, size_t ws_bytes,
                pmqa_stream_t stream);

/*
 * Per-row top-k of existing logits rows. logits: fp32 [bs * next_n, max_model_len];
 * only t < valid_len(r) is read (entries beyond are ignored whatever they hold).
 * idx: int32 [bs * next_n, k], -1 past min(k, valid_len(r)).
 * vals: fp32 [bs * next_n, k] or NULL; the logits at idx (-inf where idx is -1).
 */
int pmqa_topk(const float *logits, const int32_t *context_lens, int32_t bs, int32_t next_n,
              int32_t max_model_len, int32_t k, int32_t *idx, float *vals, void *ws,
              size_t ws_bytes, pmqa_stream_t stream);

/*
 * Fused logits + top-k in one pass over the KV cache: the logits rows need not
 * be written to memory. idx and vals as for pmqa_topk; logits may be NULL, or
 * a [bs * next_n, max_model_len] buffer that then receives the full logits.
 */
int pmqa_logits_topk(const pmqa_problem *p, int32_t k, int32_t *idx, float *vals, float *logits,
                     void *ws, size_t ws_bytes, pmqa_stream_t stream);

/*
 * pmqa_logits_topk in its two kernel launches, for callers that schedule or
 * time them apart. stages: PMQA_STAGE_SCORE (the KV pass: logits into the
 * workspace, or into logits when given, plus one key histogram per row),
 * PMQA_STAGE_SELECT (the per-row selection from that state, which also clears
 * it), or both (= pmqa_logits_topk). A SELECT call must follow the SCORE call
 * with the same arguments and workspace, with no other call on that workspace
 * in between; arguments are checked as for pmqa_logits_topk. The pages have no
 * counterpart: the split is the fused call's own launch boundary.
 */
enum { PMQA_STAGE_SCORE = 1, PMQA_STAGE_SELECT = 2 };
int pmqa_logits_topk_stages(const pmqa_problem *p, int32_t k, int32_t *idx, float *vals,
                            float *logits, void *ws, size_t ws_bytes, pmqa_stream_t stream,
                            int32_t stages);

/*
 * pmqa_logits_topk without a caller-supplied workspace. The pages have no
 * counterpart to this entry point: it exists for callers that are given device
 * buffers for their inputs and outputs but cannot allocate device memory of
 * their own (for example a plugin inside a host program that owns the whole
 * device-memory pool and offers no allocation hook, or a latency-critical loop
 * that must not call cudaMalloc, which may synchronise the device).
 * The workspace is a 32 MiB array that the library keeps in device memory on
 * every GPU where it is loaded, until the process exits. Problems whose
 * pmqa_workspace_bytes(bs, next_n, max_model_len, k, PMQA_OP_LOGITS_TOPK)
 * exceeds 32 MiB return PMQA_ERR_WORKSPACE with nothing enqueued: that size is
 * 12 bytes per (row, position) -- an 8-byte candidate entry and a 4-byte
 * compact logit -- plus 8 KB of histogram and 12 bytes of counters per row and
 * 256 bytes of status, so for example 16 rows of 131072 positions fit and 16
 * rows of 202752 do not.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before capturing
 * any stream. Every call shares the one array and clears its counters at the
 * start, so calls that overlap on the GPU (other streams, other threads) race
 * and must be serialised by the caller. Device-side status bits of these calls
 * are not reported. Allocates nothing: no cudaMalloc, cudaFree or allocating
 * library call.
 */
int pmqa_logits_topk_noalloc(const pmqa_problem *p, int32_t k, int32_t *idx, float *vals,
                             float *logits, pmqa_stream_t stream);

/*
 * The fused call restricted to a slice of every request's tokens: request i
 * scores only tokens token_begin[i] <= t < token_end[i] (device int32 [bs]
 * each, clamped to [0, ctx_i]; an empty slice scores nothing), with the
 * request's full context for the causal window, and selects per row the
 * positions (global t) of the min(k, admitted tokens of the slice) largest
 * logits; idx and vals as for pmqa_logits_topk. The block table is read only
 * for pages that hold tokens of the slice, so a GPU that keeps only its
 * slice's pages may leave the other entries unset. This is the per-GPU step
 * of a context-parallel split, whose lists pmqa_topk_merge combines; a call on
 * the whole range [0, ctx_i) equals pmqa_logits_topk. Workspace as for
 * PMQA_OP_LOGITS_TOPK; two kernel launches, as pmqa_logits_topk.
 */
int pmqa_logits_topk_range(const pmqa_problem *p, const int32_t *token_begin,
                           const int32_t *token_end, int32_t k, int32_t *idx, float *vals,
                           void *ws, size_t ws_bytes, pmqa_stream_t stream);

/*
 * Top-k of the union of candidate lists, per row: the merge step of a
 * context-parallel split of the indexer, in which each GPU holds a slice of
 * every request's tokens, scores it (pmqa_logits_topk_range) and keeps the
 * slice's top-k positions and logits; the lists are gathered from the GPUs
 * (an all-gather) and merged here. Every one of a row's k largest logits lies
 * in its own slice's top-k, so the union's top-k is the row's top-k. The pages
 * name decode context parallelism (DCP) among the configurations of the
 * sparse-MLA decode path (page "[Bug][ROCm]: ROCM_AITER_MLA can select an aiter
 * MLA decode kernel that silently returns uncorrelated output", chat-gpts.plus
 * summary, closing notes); the split and this merge are the library's design.
 *   idx       int32 [lists, rows, k_in]: positions, -1 for an empty slot (skipped)
 *   vals      fp32 [lists, rows, k_in]: their logits
 *   out_idx   int32 [rows, k]: the positions of the min(k, valid candidates)
 *             largest logits (order unspecified, ties either way), then -1
 *   out_vals  fp32 [rows, k] or NULL: their logits, then -inf
 * A position may appear in at most one of a row's lists. lists * k_in < 2^31
 * (PMQA_ERR_UNSUPPORTED otherwise). No workspace; one kernel launch.
 */
int pmqa_topk_merge(const int32_t *idx, const float *vals, int32_t lists, int32_t rows,
                    int32_t k_in, int32_t k, int32_t *out_idx, float *out_vals,
                    pmqa_stream_t stream);

/*
 * Prefill (non-paged) logits. Source: the page "[Bug] aiter ops triton
 * attention pa", section "Observations while narrowing it down", which names
 * the prefill indexer `fp8_mqa_logits` (heads 32, head_dim 128, up to 8192 keys,
 * query lengths up to 4096) beside the paged decode kernel. The pages give only
 * its name and shapes; it is read as the decode definition with the paging
 * removed and one key range per query row:
 *   logits[r][t] = sum_h weights[r][h] * relu(k_scale[t] * dot(q[r][h], k_t))
 *                  for max(ks[r], 0) <= t < min(ke[r], n), else -inf,
 * for every query row r < m and key t < n.
 *   q        fp8 e4m3fn [m, heads, head_dim], contiguous, 16-byte aligned
 *   k        fp8 e4m3fn [n, head_dim], contiguous, 16-byte aligned
 *   k_scale  fp32 [n], 4-byte aligned
 *   weights  fp32 [m, heads], contiguous, 16-byte aligned
 *   ks, ke   int32 [m]: row r's key range [ks[r], ke[r]); values outside [0, n]
 *            are clamped, ks >= ke gives an all -inf row
 * head_dim must be 128 and heads one of 16, 32, 64, 128; m * heads < 2^31 and
 * n <= 2^31 - 129 (PMQA_ERR_UNSUPPORTED otherwise).
 */
typedef struct pmqa_mqa_problem {
    const void *q;
    const void *k;
    const float *k_scale;
    const float *weights;
    const int32_t *ks;
    const int32_t *ke;
    int32_t m;
    int32_t n;
    int32_t heads;
    int32_t head_dim;
} pmqa_mqa_problem;

/*
 * logits: fp32 [m, n], 4-byte aligned; every entry is written. ws: at least
 * pmqa_workspace_bytes(m, 1, n, 0, PMQA_OP_MQA_LOGITS) bytes (256 + 8 per 4
 * query rows, rounded up to 256), 256-byte aligned, zero-filled before first
 * use; it holds the status word (a pipeline wait that ran out sets
 * PMQA_DEV_TIMEOUT) and per-call scratch. Two kernel launches.
 */
int pmqa_mqa_logits(const pmqa_mqa_problem *p, float *logits, void *ws, size_t ws_bytes,
                    pmqa_stream_t stream);

/*
 * Sparse MLA decode over the indexer's top-k positions: the attention step of
 * the same decode step, which attends only to the positions the top-k
 * selected. Sources: the page "[Bug] aiter ops triton attention pa", section
 * "Downstream impact" (the sparse MLA attention attends to the indexer's top-k
 * positions); the page "[Bug][ROCm]: ROCM_AITER_MLA can select an aiter MLA
 * decode kernel that silently returns uncorrelated output" (chat-gpts.plus
 * summary: fp8 Q and fp8 KV, 16 query heads per latent KV head, 1..4 query
 * rows per request, a log-sum-exp output for decode context parallelism); the
 * page "[Bugfix][Hardware][AMD] Fix last_page_len calculation in AITER MLA
 * decode", section "The Bug" (the MLA cache in pages of one token; larger
 * pages use the same lookup). The pages give no widths: a cached token is one
 * latent row of 576 fp8 values whose first 512 are its value vector (the MLA
 * layout of a 512-wide compressed KV plus a 64-wide rotary key), and q and the
 * cache carry one fp32 scale each.
 *
 *   For query row r = i*next_n + j, head h and each listed position t of row r
 *   (indices[r][e] >= 0; a position listed twice counts twice):
 *     phys    = block_tables[i][t / block_size] * block_size + t % block_size
 *     s_t     = sm_scale * sum_d (q_scale * q[r][h][d]) * (kv_scale * kv[phys][d]),  d < 576
 *     out[r][h][d] = sum_t softmax(s)_t * kv_scale * kv[phys][d],   d < 512
 *     lse[r][h]    = ln sum_t exp(s_t)
 *   A row with no listed position gives out = 0 and lse = -inf.
 *
 *   q             fp8 e4m3fn [bs * next_n, heads, head_dim], contiguous, 16-byte aligned
 *   kv_cache      fp8 e4m3fn [num_blocks, block_size, head_dim], contiguous,
 *                 16-byte aligned; only the rows of listed positions are read
 *   indices       int32 [bs * next_n, topk]: positions in the row's request
 *                 (what pmqa_logits_topk returns), -1 for an empty entry
 *   block_tables  int32 [bs, max_blocks_per_seq], row-major
 * heads must be 16, head_dim 576 and v_head_dim 512 (PMQA_ERR_UNSUPPORTED
 * otherwise); the scales must be finite.
 */
typedef struct pmqa_mla_problem {
    const void *q;
    const void *kv_cache;
    const int32_t *indices;
    const int32_t *block_tables;
    float q_scale;
    float kv_scale;
    float sm_scale;
    int32_t bs;
    int32_t next_n;
    int32_t heads;
    int32_t head_dim;
    int32_t v_head_dim;
    int32_t topk;
    int32_t block_size;
    int32_t max_blocks_per_seq;
    int64_t num_blocks;
} pmqa_mla_problem;

/* Bytes of workspace for pmqa_sparse_mla_decode over `rows` query rows (about
   17 MB, whatever the row count); 0 for rows < 0. */
size_t pmqa_sparse_mla_workspace_bytes(int32_t rows);

/*
 * out: bf16 [bs * next_n, heads, 512], 4-byte aligned; lse: fp32
 * [bs * next_n, heads] or NULL. ws: pmqa_sparse_mla_workspace_bytes(rows)
 * bytes, 256-byte aligned, its status word zero before the first use
 * (pmqa_workspace_init). A listed position past the block table sets
 * PMQA_DEV_BAD_CONTEXT, a table entry outside [0, num_blocks)
 * PMQA_DEV_BAD_BLOCK_ID (the position is then skipped); a pipeline wait that
 * ran out sets PMQA_DEV_TIMEOUT (results invalid). Two kernel launches: the
 * attention, and the combination of rows whose tiles were split over CTAs.
 */
int pmqa_sparse_mla_decode(const pmqa_mla_problem *p, void *out, float *lse, void *ws,
                           size_t ws_bytes, pmqa_stream_t stream);

/*
 * The decode restricted to a slice of every request's tokens: request i's rows
 * attend only to their listed positions t with token_begin[i] <= t <
 * token_end[i] (device int32 [bs] each); the other listed positions are
 * skipped, so the block table need only map the slice's pages. This is one
 * GPU's step of a decode split by context (decode context parallelism: the
 * chat-gpts.plus summary names an LSE output for it): the slices' outputs and
 * log-sum-exps are gathered and combined by pmqa_sparse_mla_merge. Otherwise
 * as pmqa_sparse_mla_decode; a row with no position in its slice gives out = 0
 * and lse = -inf.
 */
int pmqa_sparse_mla_decode_range(const pmqa_mla_problem *p, const int32_t *token_begin,
                                 const int32_t *token_end, void *out, float *lse, void *ws,
                                 size_t ws_bytes, pmqa_stream_t stream);

/*
 * Merge of `parts` partial decodes of the same rows (each over a disjoint part
 * of every row's listed positions, e.g. the slices of a context split):
 *   outs  bf16 [parts, rows, heads, 512]; lses fp32 [parts, rows, heads]
 *   out   bf16 [rows, heads, 512] = sum_g w_g outs[g] / sum_g w_g,
 *         w_g = exp(lses[g] - max_g lses[g]) (a part with lse -inf weighs 0)
 *   lse   fp32 [rows, heads] or NULL: max_g lses[g] + ln sum_g w_g
 * heads must be 16. No workspace; one kernel launch.
 */
int pmqa_sparse_mla_merge(const void *outs, const float *lses, int32_t parts, int32_t rows,
                          int32_t heads, void *out, float *lse, pmqa_stream_t stream);

/*
 * Measurement aid beside the decode path (computes nothing of the method): reads
 * the rows rows[0..n) of a pool of fixed-pitch rows, each as its 16-byte aligned
 * window (144 bytes for row_pitch 132, the token row of the KV cache; 576 bytes
 * for row_pitch 576, the latent row of the MLA cache), to time how fast the GPU
 * gathers such rows. One launch, one CTA per SM.
 *   pool      device, 16-byte aligned, pool_bytes long; a window that would pass
 *             its end, and a negative row, is skipped (PMQA_DEV_BAD_CONTEXT in out[0])
 *   rows      device int32 [n]
 *   method    0: 16-byte loads into registers; 1: 16-byte cp.async into shared
 *             memory; 2: one bulk copy (cp.async.bulk) per window into shared memory
 *   out       device uint32 [2], zeroed by the caller: out[0] |= status bits
 *             (PMQA_DEV_TIMEOUT for a wait that ran out), out[1] ^= the XOR of
 *             every 32-bit word read (method 0) or of each window's first
 *             word (methods 1, 2)
 * Returns PMQA_ERR_UNSUPPORTED for another pitch, PMQA_ERR_INVALID_ARG for
 * n < 0, a method outside 0..2, a null or misaligned pointer (n = 0 launches
 * nothing and returns PMQA_OK).
 */
int pmqa_gather_probe(const void *pool, uint64_t pool_bytes, const int32_t *rows, int64_t n,
                      int32_t row_pitch, int32_t method, uint32_t *out, pmqa_stream_t stream);

/*
 * Synchronise the stream, return the device status bits recorded since the
 * last read (>= 0) and clear them, or a negative PMQA_ERR_* code.
 */
int pmqa_read_device_status(void *ws, pmqa_stream_t stream);

/* Static text for a return code. */
const char *pmqa_status_string(int code);

/* Library version, major * 10000 + minor * 100 + patch. */
int pmqa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PMQA_H */
