/*
 * hisa.h -- C ABI of the GB300 (sm_103a) HiSA sparse-attention step.
 *
 * The step is the one described on the page "feat(deepseek-v4): implement HiSA
 * hierarchical sparse attention" (cited as [HiSA issue] with its section): score
 * pooled indexer keys, select index_topk pooled rows (flat or hierarchical), gather
 * the selected pooled KV rows and combine them with the local window and the
 * per-head sinks in one split softmax.
 *
 * Conventions shared by every entry point
 *  - Tensor pointers are DEVICE pointers owned by the caller; tensors are dense,
 *    row-major, with the shapes written beside each argument. The library never
 *    allocates, never frees, never synchronises the stream and keeps no state
 *    between calls; it is safe to call from several host threads on different
 *    streams with different workspaces.
 *  - Consecutive calls may overlap, on request: a call whose descriptor sets
 *    HISA_FLAG_CHAINED launches its kernels as programmatic dependents of the
 *    kernel before it on the stream, so it may start while that kernel finishes.
 *    hisa_select_topk then reads q, w, key_off and t0, and hisa_sparse_attend reads
 *    q, local_kv, local_len, local_pos0, kv_off, t0 and sinks before that kernel has
 *    completed; each waits for it before reading top_blk / I and before writing any
 *    output. Set the flag only when the kernel just before the call on the stream is
 *    another libhisa call and none of those early-read inputs is written by it (the
 *    usual chain: hisa_block_filter(_append) -> hisa_select_topk -> hisa_sparse_attend).
 *    Without the flag (flags = 0) a call's kernels start after the previous work on the
 *    stream has completed, as with any ordinary launch, except kernels that read nothing
 *    before the previous grid has completed (the coarse stage's pipeline, and the selects
 *    and merges that follow a call's scoring or combine kernel), which may always overlap
 *    its end.
 *  - Ragged batches: sequence b owns pooled rows [key_off[b], key_off[b+1]) of the
 *    packed key / KV arrays, so Np_b = key_off[b+1] - key_off[b] (int64, device).
 *  - Positions: t0[b] (int32, device) is the absolute token position of query
 *    row 0 of sequence b; row j sits at t = t0[b] + j ([HiSA issue] "Conventions").
 *    The visible pooled prefix is V(t) = min(Np_b, floor((t+1)/r)) ([HiSA issue]
 *    "The pooled stream and positions"). As on the page, the causal pooled mask
 *    is applied only when L > 1; single-row calls treat all Np_b rows as visible.
 *  - Head weights w are the RAW weights_proj(x) outputs (f32); the library applies
 *    H_i^-1/2 * D_i^-1/2 once per head ([HiSA issue] "The indexer query and
 *    per-head weights"). All selection scoring accumulates in f32.
 *  - Selections are sets: entries of I / top_blk are written in ascending id order,
 *    equal scores are broken by ascending id, -0.0 equals +0.0, and rows that have
 *    fewer than k candidates are padded with -1.
 *  - Host validation is synchronous: a bad argument returns HISA_EINVAL /
 *    HISA_EDTYPE / HISA_EWORKSPACE before anything is enqueued. Kernels then run
 *    asynchronously on `stream`; a failed launch returns HISA_ECUDA.
 *  - Data the host cannot see (offsets, ids, per-sequence gates) is checked on the
 *    device. A violation never faults: the kernel skips the access, writes -1 /
 *    NEG where the page defines a neutral value, and ORs a HISA_DEV_* bit into the
 *    status word held in the first 256 bytes of the workspace. Read it with
 *    hisa_device_status(); clear it with hisa_workspace_init().
 *  - Workspace: `ws` is device memory of at least hisa_workspace_bytes(op, desc)
 *    bytes, 256-byte aligned. One workspace sized for the largest op may be shared
 *    by consecutive calls on the same stream.
 */
#ifndef HISA_H
#define HISA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define HISA_API __attribute__((visibility("default")))
#else
#define HISA_API
#endif

struct CUstream_st;                  /* the type behind cudaStream_t */
typedef struct CUstream_st *hisa_stream_t;

typedef enum {
    HISA_OK = 0,
    HISA_EINVAL = -1,     /* bad descriptor field, pointer, alignment or a host-checkable gate */
    HISA_EDTYPE = -2,     /* dtype or shape combination without a kernel */
    HISA_EWORKSPACE = -3, /* workspace missing, misaligned or too small */
    HISA_ECUDA = -4,      /* a CUDA runtime call or a kernel launch failed */
    HISA_EDEVICE = -5     /* hisa_device_status(): a kernel flagged bad data */
} hisa_status;

typedef enum { HISA_F32 = 0, HISA_BF16 = 1 } hisa_dtype;

/* Bits of the device status word. */
#define HISA_DEV_BAD_OFFSETS 0x1u /* offsets not monotone, past keys_rows / means_rows / kv_rows, Np_b > Np_max,
                                    or a capacity too small; the sequence is skipped */
#define HISA_DEV_GATE        0x2u /* a sequence failed Np_b >= index_block*index_keep; rows are -1 */
#define HISA_DEV_BAD_ID      0x4u /* a selected id outside [-1, Np_b) reached the combine; skipped */
#define HISA_DEV_NONFINITE   0x8u /* a select saw a non-finite score */
#define HISA_DEV_BAD_BLOCK   0x10u /* a top_blk entry outside [0, nb_b); that row is written as -1 */
#define HISA_DEV_TIMEOUT     0x20u /* a kernel gave up on a bounded wait; its outputs are incomplete */

/* Bits of hisa_index_desc.flags / hisa_attn_desc.flags (all others must be 0). */
#define HISA_FLAG_CHAINED    0x1u /* may overlap the previous libhisa call on the stream (see above) */

/* Operation ids for hisa_workspace_bytes. */
#define HISA_OP_INDEX_SCORES  0
#define HISA_OP_BLOCK_MEANS   1
#define HISA_OP_BLOCK_FILTER  2
#define HISA_OP_SELECT_TOPK   3
#define HISA_OP_FLAT_TOPK     4
#define HISA_OP_SPARSE_ATTEND 5
#define HISA_OP_COMPRESS      6

/* Indexer problem ([HiSA issue] "Configuration", "Flat selection", "HiSA decode path"). */
typedef struct {
    int32_t B;            /* sequences (>= 1) */
    int32_t L;            /* query rows per sequence (>= 1; 1 = decode) */
    int32_t H_i;          /* indexer heads, index_n_heads */
    int32_t D_i;          /* indexer head dim, index_head_dim: 32, 64 or 128 */
    int32_t r;            /* compress ratio (>= 1) */
    int32_t index_topk;   /* k: pooled rows kept per query (1..2048) */
    int32_t index_block;  /* b: HiSA block size in pooled rows (0 disables the hierarchy) */
    int32_t index_keep;   /* keep: blocks kept by the coarse stage */
    int64_t Np_max;       /* an upper bound of Np_b over the batch (sizes grids and workspace) */
    int64_t keys_rows;    /* rows allocated in keys (>= key_off[B]); no key read goes past it */
    int64_t means_rows;   /* rows allocated in the block-mean array; no block-mean read or
                             write goes past it (0 for calls that take no means) */
    int32_t q_dtype;      /* hisa_dtype of q: HISA_F32 or HISA_BF16 */
    int32_t k_dtype;      /* hisa_dtype of the pooled indexer keys */
    int32_t flags;        /* HISA_FLAG_* bits (0 = none) */
} hisa_index_desc;

/* Attention problem ([HiSA issue] "Consuming the selection: sparse combine"). */
typedef struct {
    int32_t B, L;         /* sequences, query rows per sequence */
    int32_t H;            /* query heads sharing the single KV head: 8, 16 or 64 */
    int32_t Dh;           /* head dim: 64, 128 or 512 (with H = 8, 16, 64 respectively) */
    int32_t window;       /* sliding window: local row s is visible to t iff 0 <= t-s < window */
    int32_t W_max;        /* rows allocated per sequence in local_kv */
    int32_t r;            /* compress ratio, for V(t) */
    int32_t k;            /* width of I (ignored when I == NULL) */
    int64_t Np_max;       /* an upper bound of Np_b over the batch */
    int64_t kv_rows;      /* rows allocated in pooled_kv (>= kv_off[B]); no read goes past it */
    float scale;          /* softmax scale; <= 0 selects Dh^-1/2 */
    int32_t q_dtype;      /* hisa_dtype of q; must equal kv_dtype */
    int32_t kv_dtype;     /* hisa_dtype of local_kv and pooled_kv */
    int32_t flags;        /* HISA_FLAG_* bits (0 = none) */
    int32_t out_dtype;    /* hisa_dtype of out: HISA_F32 (0, the default) or HISA_BF16, the
                             f32 result rounded to nearest even once, after the combine */
} hisa_attn_desc;

/* The indexer's compressor ([HiSA issue] "The pooled stream and positions", "Configuration":
 * compressor.{wkv, wgate, ape, norm}, compress_rope_theta, qk_rope_head_dim). */
typedef struct {
    int32_t B;            /* sequences (>= 1) */
    int32_t D_i;          /* pooled key dim: 32, 64 or 128 */
    int32_t r;            /* compress ratio: tokens per window (1..128) */
    int32_t overlap;      /* 1: the overlap variant, projections 2*D_i wide (channels [0, D_i) pool
                             the previous window, [D_i, 2*D_i) the row's own window); 0: plain, D_i wide */
    int32_t rope_dims;    /* trailing dims rotated, even, 0..D_i (64) */
    int32_t index_block;  /* b: block size of the block-mean cache (0: no means kept) */
    int32_t n_new_max;    /* an upper bound of n_new[b] (0..1048576) */
    int32_t k_dtype;      /* hisa_dtype of the pooled key cache */
    float rope_theta;     /* RoPE base (> 1): compress_rope_theta = 160000 */
    float eps;            /* RMSNorm epsilon (> 0) */
    int64_t tok_rows;     /* rows allocated in kv and gate */
    int64_t keys_rows;    /* rows allocated in keys; no key read or write goes past it */
    int64_t means_rows;   /* rows allocated in means (0 when means is NULL) */
    int32_t flags;        /* HISA_FLAG_* bits (0 = none) */
} hisa_compress_desc;

/* Bytes of device workspace `op` needs for `desc` (a hisa_index_desc* for ops 0-4,
 * a hisa_attn_desc* for op 5, a hisa_compress_desc* for op 6). Always >= 256 for a valid desc; 0 for an invalid one.
 * Pure host arithmetic: needs no GPU. */
HISA_API size_t hisa_workspace_bytes(int32_t op, const void *desc);

/* Clears the device status word of `ws` (asynchronous memset on `stream`). */
HISA_API hisa_status hisa_workspace_init(void *ws, size_t ws_bytes, hisa_stream_t stream);

/* Synchronises `stream`, then copies the status word of `ws` into *flags.
 * Returns HISA_EDEVICE when any bit is set, HISA_OK otherwise. */
HISA_API hisa_status hisa_device_status(const void *ws, hisa_stream_t stream, uint32_t *flags);

/* A static, human-readable name for a status code. */
HISA_API const char *hisa_status_string(int32_t status);

/* Flat indexer scores ([HiSA issue] "Flat selection (baseline path)": s = relu(q.k),
 * score = sum_h s * scale * w; NEG = -1e30 where p >= V(t0+j) when L > 1).
 *   q      [B, L, H_i, D_i]  q_dtype      keys    [sum Np_b, D_i]  k_dtype
 *   w      [B, L, H_i]       f32 raw      key_off [B+1] int64; t0 [B] int32
 *   scores [B*L, ld_scores]  f32 out: row b*L+j holds Np_b scores; columns
 *          [Np_b, ld_scores) are not written. ld_scores >= Np_max.
 * With L > 1 this is the dense L x Np x (H_i*D_i) prefill contraction. */
HISA_API hisa_status hisa_index_scores(const hisa_index_desc *desc, const void *q, const float *w,
                              const void *keys, const int64_t *key_off, const int32_t *t0,
                              float *scores, int64_t ld_scores, void *ws, size_t ws_bytes,
                              hisa_stream_t stream);

/* Block-mean representatives ([HiSA issue] "HiSA decode path": rep = mean over the
 * index_block rows of each complete block; the tail [nb*b, Np) has no block).
 *   means     [*, D_i] f32 out; sequence b's nb_b = floor(Np_b / b) means occupy rows
 *             [means_off[b], means_off[b] + nb_b); means_off [B+1] int64 (device) must
 *             leave room for nb_b rows (else HISA_DEV_BAD_OFFSETS and nothing is written).
 *   first_block [B] int32 or NULL: blocks [first_block[b], nb_b) are (re)computed, so
 *             a decode loop appends the newly completed blocks only. NULL = from 0.
 * f32 sums: for each dimension, eight partial sums over the rows i = k (mod 8) in row
 * order, combined as ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)), divided by b
 * (blocks of more than 8192 keys: one sum in row order). */
HISA_API hisa_status hisa_block_means(const hisa_index_desc *desc, const void *keys,
                             const int64_t *key_off, const int64_t *means_off,
                             const int32_t *first_block, float *means, void *ws, size_t ws_bytes,
                             hisa_stream_t stream);

/* Coarse stage ([HiSA issue] "HiSA decode path" / "HiSA batched path": cscore over
 * block means, top Kb = min(keep, nb) blocks; with L > 1 a block is eligible iff its
 * first row is visible, else cscore = NEG).
 *   means/means_off as written by hisa_block_means.
 *   top_blk  [B, L, index_keep] int32 out, ascending block ids.
 *   cscores  [B*L, ld_cscores] f32 out, optional (NULL): nb_b coarse scores per row.
 * Host gate: index_block > 0 and index_block*index_keep >= index_topk, else
 * HISA_EINVAL. Device gate: Np_b >= index_block*index_keep, else HISA_DEV_GATE and a
 * row of -1. */
HISA_API hisa_status hisa_block_filter(const hisa_index_desc *desc, const void *q, const float *w,
                              const float *means, const int64_t *means_off,
                              const int64_t *key_off, const int32_t *t0, int32_t *top_blk,
                              float *cscores, int64_t ld_cscores, void *ws, size_t ws_bytes,
                              hisa_stream_t stream);

/* hisa_block_means, then hisa_block_filter, as one call: the block means of blocks
 * [first_block[b], nb_b) are appended to `means` (same values as hisa_block_means), then
 * the coarse stage runs over all nb_b means. Arguments as in those two calls. For decode
 * (L = 1) with the DeepSeek-V4 indexer shape (H_i = 64, D_i = 128, index_block = 64, bf16
 * keys) it is one kernel, in which the new means are computed while the older means
 * stream into the coarse scoring; otherwise it makes the two calls in turn. ws must hold
 * hisa_workspace_bytes(HISA_OP_BLOCK_FILTER, desc) bytes. */
HISA_API hisa_status hisa_block_filter_append(const hisa_index_desc *desc, const void *q,
                                     const float *w, const void *keys, const int64_t *key_off,
                                     float *means, const int64_t *means_off,
                                     const int32_t *first_block, const int32_t *t0,
                                     int32_t *top_blk, float *cscores, int64_t ld_cscores,
                                     void *ws, size_t ws_bytes, hisa_stream_t stream);

/* Fine stage ([HiSA issue] "HiSA decode path" / "HiSA batched path": candidates
 * pos = top_blk[c / b]*b + c % b, exact rescoring, NEG where pos >= V(t0+j) when
 * L > 1, top k, I = pos[sel]).
 *   top_blk  [B, L, index_keep] int32 (any order; each entry in [0, nb_b)).
 *   I        [B, L, index_topk] int32 out: absolute pooled ids, ascending.
 *   fscores  [B*L, index_keep*index_block] f32 out, optional (NULL): candidate scores
 *            in ascending pos order.
 * Gates as hisa_block_filter. */
HISA_API hisa_status hisa_select_topk(const hisa_index_desc *desc, const void *q, const float *w,
                             const void *keys, const int64_t *key_off, const int32_t *t0,
                             const int32_t *top_blk, int32_t *I, float *fscores, void *ws,
                             size_t ws_bytes, hisa_stream_t stream);

/* Flat selection ([HiSA issue] "Flat selection (baseline path)": top k = min(index_topk,
 * Np_b) of the flat scores; the exact baseline and the path for 512 < Np < 1024).
 *   I [B, L, index_topk] int32 out, ascending ids, -1 beyond min(index_topk, Np_b). */
HISA_API hisa_status hisa_flat_topk(const hisa_index_desc *desc, const void *q, const float *w,
                           const void *keys, const int64_t *key_off, const int32_t *t0,
                           int32_t *I, void *ws, size_t ws_bytes, hisa_stream_t stream);

/* Allocation-free flat selection. The paper has no counterpart: this entry point exists
 * for callers that cannot allocate device memory (hosts whose runtime owns all device
 * memory through its own pool, plugins that may not allocate outside the framework's
 * allocator, loops where cudaMalloc / cudaFree would synchronise the device) and so
 * cannot pass the workspace hisa_flat_topk needs. It computes exactly what
 * hisa_flat_topk computes, with the same arguments and errors, but keeps the scores in
 * a fixed array of device memory declared inside libhisa (16 MiB + 256 bytes), which
 * every GPU that loads the library holds until the process exits. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   B * L * Np_max must not exceed HISA_FLAT_NOALLOC_MAX_SCORES, else HISA_EWORKSPACE
 *   before anything is enqueued.
 *   dev_status: optional (NULL) device pointer to one uint32 that receives this call's
 *   HISA_DEV_* bits (the status is cleared at the start of every call).
 * Runs on the current device. The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress); make that first call before any stream capture.
 * All calls on one device share the one array: calls that may overlap on the GPU (on
 * different streams, or from several host threads without ordering) race and give
 * undefined results; order them on one stream. */
#define HISA_FLAT_NOALLOC_MAX_SCORES 4194304
HISA_API hisa_status hisa_flat_topk_noalloc(const hisa_index_desc *desc, const void *q,
                                   const float *w, const void *keys, const int64_t *key_off,
                                   const int32_t *t0, int32_t *I, uint32_t *dev_status,
                                   hisa_stream_t stream);

/* Indexer compressor ([HiSA issue] "The pooled stream and positions"): appends n_new[b]
 * pooled rows p = p_first[b] .. p_first[b] + n_new[b] - 1 to sequence b's pooled key cache,
 * each anchored at the token window [p r, p r + r - 1]: per output dim d, one softmax over
 * the gate logits gate[t] + ape[t - window start] of the window's tokens (with the overlap
 * variant also the previous window's, through their first D_i channels; row 0 has no
 * previous window) weighs their kv values; then RMSNorm with norm_w and eps, then RoPE of
 * the trailing rope_dims dims, pairs (2m, 2m+1), by the angle (p r) * rope_theta^(-2i /
 * rope_dims) for the i-th rotated pair. Afterwards every block of index_block rows that
 * the new rows complete gets its mean in `means`, with the bits hisa_block_means writes.
 *   kv, gate   [tok_rows, C] f32: wkv(x) and wgate(x) of the tokens, C = 2*D_i (overlap) or
 *              D_i. Sequence b's rows [tok_off[b], tok_off[b+1]) hold (n_new[b] + 1) * r
 *              tokens: the window before row p_first[b] (ignored when p_first[b] == 0 or
 *              without overlap), then the windows of the new rows, in token order.
 *   tok_off    [B+1] int64;  p_first, n_new [B] int32 (n_new <= n_new_max; 0 = nothing)
 *   ape        [r, C] f32;   norm_w [D_i] f32
 *   keys       [keys_rows, D_i] k_dtype in/out: pooled row p of sequence b is row
 *              key_off[b] + p; rows below p_first[b] are read for block means, and
 *              key_off[b] + p_first[b] + n_new[b] must not pass key_off[b+1].
 *   means      [means_rows, D_i] f32 out or NULL; block beta of sequence b at
 *              means_off[b] + beta (means_off [B+1] int64 must leave room for every complete
 *              block). NULL, or index_block == 0, keeps no means.
 * Offsets or counts that do not fit set HISA_DEV_BAD_OFFSETS; that sequence is skipped. */
HISA_API hisa_status hisa_compress_append(const hisa_compress_desc *desc, const float *kv,
                                 const float *gate, const int64_t *tok_off,
                                 const int32_t *p_first, const int32_t *n_new, const float *ape,
                                 const float *norm_w, void *keys, const int64_t *key_off,
                                 float *means, const int64_t *means_off, void *ws,
                                 size_t ws_bytes, hisa_stream_t stream);

/* Sparse combine ([HiSA issue] "Consuming the selection: sparse combine"): one softmax
 * over the visible local rows, the gathered pooled rows P = pooled_kv[I] and the
 * per-head sink, which joins the normaliser and carries no value; K = V.
 *   q          [B, L, H, Dh]  q_dtype (already roped)
 *   local_kv   [B, W_max, Dh] kv_dtype; local_len [B] int32 rows present (<= W_max);
 *              local_pos0 [B] int32 absolute position of local row 0
 *   pooled_kv  [sum Np_b, Dh] kv_dtype; kv_off [B+1] int64
 *   I          [B, L, k] int32 pooled ids (-1 = skip), or NULL for the dense branch over
 *              all Np_b rows. With L > 1 ids >= V(t0+j) are masked.
 *   sinks      [H] f32;  t0 [B] int32
 *   out        [B, L, H, Dh] out, f32 or bf16 as desc->out_dtype says (any device-accessible
 *              address, 16-byte aligned: device memory, or the device address of page-locked
 *              host memory, which the kernels then write directly over the host link)
 * Np_b == 0 gives local-only attention (branch 1 of the three-way branch). */
HISA_API hisa_status hisa_sparse_attend(const hisa_attn_desc *desc, const void *q, const void *local_kv,
                               const int32_t *local_len, const int32_t *local_pos0,
                               const void *pooled_kv, const int64_t *kv_off, const int32_t *I,
                               const float *sinks, const int32_t *t0, void *out, void *ws,
                               size_t ws_bytes, hisa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HISA_H */
