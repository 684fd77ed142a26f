// C ABI entry points of libhisa: host-side validation, workspace layout and kernel
// dispatch. Declarations and the contract live in include/hisa.h.
#include <cmath>
#include <cstring>

#include "hisa_internal.cuh"

using namespace hisa;

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool dtype_ok(int32_t d) { return d == HISA_F32 || d == HISA_BF16; }


// Host-checkable validity of an indexer descriptor.
hisa_status check_index_desc(const hisa_index_desc *d) {
    if (!d) return HISA_EINVAL;
    if (d->B < 1 || d->L < 1 || d->H_i < 1 || d->H_i > 128 || d->r < 1) return HISA_EINVAL;
    if (d->index_topk < 1 || d->index_topk > kMaxTopk) return HISA_EINVAL;
    if (d->index_block < 0 || d->index_keep < 0 || d->index_keep > 64) return HISA_EINVAL;
    if (d->Np_max < 0 || d->Np_max > (int64_t)65535 * 256) return HISA_EINVAL;
    if (d->keys_rows < 0 || d->keys_rows > 0x7fffffffLL) return HISA_EINVAL;
    if (d->means_rows < 0 || d->means_rows > 0x7fffffffLL) return HISA_EINVAL;
    if ((int64_t)d->B * d->L > 0x7fffffffLL) return HISA_EINVAL;
    if (d->flags & ~(int32_t)HISA_FLAG_CHAINED) return HISA_EINVAL;
    if (!dtype_ok(d->q_dtype) || !dtype_ok(d->k_dtype)) return HISA_EDTYPE;
    if (d->D_i != 32 && d->D_i != 64 && d->D_i != 128) return HISA_EDTYPE;
    return HISA_OK;
}

// Gate conditions the host can see ([HiSA issue] "HiSA decode path": index_block > 0
// and index_block * index_keep >= k). Np_b >= index_block * index_keep is checked on
// the device per sequence.
hisa_status check_hisa_gate(const hisa_index_desc *d) {
    if (d->index_block < 1 || d->index_keep < 1) return HISA_EINVAL;
    if ((int64_t)d->index_block * d->index_keep < d->index_topk) return HISA_EINVAL;
    if ((int64_t)d->index_block * d->index_keep > (int64_t)1 << 20) return HISA_EINVAL;
    return HISA_OK;
}

hisa_status check_attn_desc(const hisa_attn_desc *d) {
    if (!d) return HISA_EINVAL;
    if (d->B < 1 || d->L < 1 || d->window < 0 || d->W_max < 0 || d->r < 1 || d->k < 0 ||
        d->k > kMaxTopk)
        return HISA_EINVAL;
    if (d->Np_max < 0 || d->Np_max > 0x7fffffffLL) return HISA_EINVAL;
    if (d->kv_rows < 0 || d->kv_rows > 0x7fffffffLL) return HISA_EINVAL;
    if ((int64_t)d->B * d->L > 0x7fffffffLL) return HISA_EINVAL;
    if (d->flags & ~(int32_t)HISA_FLAG_CHAINED) return HISA_EINVAL;
    if (!dtype_ok(d->q_dtype) || !dtype_ok(d->kv_dtype) || d->q_dtype != d->kv_dtype ||
        !dtype_ok(d->out_dtype))
        return HISA_EDTYPE;
    if (!attend_simt_supported(d->H, d->Dh)) return HISA_EDTYPE;
    return HISA_OK;
}

hisa_status check_compress_desc(const hisa_compress_desc *d) {
    if (!d) return HISA_EINVAL;
    if (d->B < 1 || d->r < 1 || d->r > 128 || (d->overlap != 0 && d->overlap != 1)) return HISA_EINVAL;
    if (d->rope_dims < 0 || d->rope_dims > d->D_i || (d->rope_dims & 1)) return HISA_EINVAL;
    if (d->index_block < 0 || d->index_block > 8192) return HISA_EINVAL;
    if (d->n_new_max < 0 || d->n_new_max > (1 << 20)) return HISA_EINVAL;
    if (!(d->rope_theta > 1.f) || !(d->eps > 0.f)) return HISA_EINVAL;
    if (d->tok_rows < 0 || d->keys_rows < 0 || d->means_rows < 0) return HISA_EINVAL;
    if (d->flags & ~(int32_t)HISA_FLAG_CHAINED) return HISA_EINVAL;
    if (!dtype_ok(d->k_dtype)) return HISA_EDTYPE;
    if (d->D_i != 32 && d->D_i != 64 && d->D_i != 128) return HISA_EDTYPE;
    if ((int64_t)d->B * (d->n_new_max / (d->index_block > 0 ? d->index_block : 64) + 2) >
        ((int64_t)1 << 31))
        return HISA_EINVAL;
    if (d->B > 65535) return HISA_EINVAL;
    return HISA_OK;
}

int64_t n_rows(const hisa_index_desc *d) { return (int64_t)d->B * d->L; }

// The coarse stage of many bf16 query rows (batched prefill) runs as a dense contraction
// over the block means split into bf16 planes (launch_coarse_gemm), then a select; fewer
// or f32 rows take the per-row pipeline. Host arithmetic only (sizes the workspace).
bool coarse_gemm_ok(const hisa_index_desc *d) {
    return d->L >= 4 && n_rows(d) >= 256 && d->q_dtype == HISA_BF16 && d->means_rows > 0 &&
           score_gemm_supported(d->H_i, d->D_i, 1, 1, d->B, d->L);
}

// Number of split-K ranges for the combine: about one item per SM (a split item re-reads its
// row's q and writes a partial as large as the row's output, which the merge reads back, so
// more splits than SMs cost more than they spread), never fewer rows per split than one chunk.
// `list_len` bounds the attended rows per query. Host arithmetic only (sizes the workspace).
int pick_nsplit(int64_t queries, int64_t list_len, int64_t *rows_per_split) {
    const int chunk = attend_chunk_rows();
    const int64_t chunks = (list_len + chunk - 1) / chunk;
    int64_t ns = kSmTarget / queries;
    if (ns > chunks) ns = chunks;
    if (ns < 1) ns = 1;
    if (ns > 64) ns = 64;
    const int64_t per = ((chunks + ns - 1) / ns) * chunk;
    *rows_per_split = per > 0 ? per : chunk;
    if (list_len > 0) ns = (list_len + *rows_per_split - 1) / *rows_per_split;
    return (int)(ns < 1 ? 1 : ns);
}

// Upper bound of the attended rows of one query row: the visible local window plus
// the pooled rows (all of them for the dense branch).
int64_t attn_list_len(const hisa_attn_desc *d, bool dense) {
    const int64_t local = d->W_max < d->window ? d->W_max : d->window;
    return local + (dense ? d->Np_max : (int64_t)d->k);
}

size_t attn_part_bytes(const hisa_attn_desc *d, bool dense) {
    int64_t per = 0;
    const int ns = pick_nsplit((int64_t)d->B * d->L, attn_list_len(d, dense), &per);
    if (ns <= 1) return 0;
    return (size_t)d->B * d->L * ns * d->H * (d->Dh + 2) * sizeof(float);
}

uint32_t *status_of(void *ws) { return reinterpret_cast<uint32_t *>(ws); }

float *scratch_of(void *ws) {
    return reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + kStatusBytes);
}

hisa_status check_ws(void *ws, size_t have, size_t need) {
    if (!ws || !aligned(ws, kAlign)) return HISA_EWORKSPACE;
    if (have < need) return HISA_EWORKSPACE;
    return HISA_OK;
}

hisa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? HISA_OK : HISA_ECUDA; }

ScoreParams score_params(const hisa_index_desc *d, int mode, const void *q, const float *w,
                         const void *rows, int rows_bf16, const int64_t *key_off,
                         const int32_t *t0, float *out, int64_t ld, void *ws) {
    ScoreParams p{};
    p.mode = mode;
    p.B = d->B; p.L = d->L; p.H_i = d->H_i; p.D_i = d->D_i; p.r = d->r;
    p.b = d->index_block; p.keep = d->index_keep;
    p.causal = d->L > 1;
    p.q = q; p.q_bf16 = d->q_dtype == HISA_BF16;
    p.w = w;
    p.head_scale = (float)(1.0 / std::sqrt((double)d->H_i * (double)d->D_i));
    p.rows = rows; p.rows_bf16 = rows_bf16;
    p.key_off = key_off; p.t0 = t0;
    p.out = out; p.ld_out = ld;
    p.Np_max = d->Np_max;
    p.keys_rows = d->keys_rows;
    p.means_rows = d->means_rows;
    p.status = status_of(ws);
    p.chained = (d->flags & HISA_FLAG_CHAINED) != 0;
    return p;
}

// A few long coarse / fine rows (a single long-context query): one CTA per row would leave
// most SMs idle, so each row's tiles are split over CTAs and a separate select follows.
// (Splitting shorter rows, or more of them, measured slower than one CTA per row: the
// separate select and the scores' round trip cost more than the idle SMs.) Coarse rows
// longer than the persistent pipeline takes (over 4096 blocks, 1M+ tokens) are split
// whatever their number.
bool split_rows(const hisa_index_desc *d, int mode, int64_t n) {
    const int sms = device_sm_count();
    const bool few_long = n >= 2048 && n_rows(d) * 8 <= sms;
    const bool past_pipe = mode == kCoarse && n > (int64_t)kCoarseChunk * kCoarseMaxChunks;
    return sms > 0 && (few_long || past_pipe) &&
           score_tc_split_ok(mode, d->H_i, d->D_i, mode == kFine ? d->k_dtype == HISA_BF16 : 0,
                             d->index_block);
}

// Coarse rows of more than kCoarseChunk blocks run in chunks whose (id, score) selections
// go to `scratch` (the workspace's score area, which holds far more than the pairs).
void set_coarse_chunks(ScoreTcParams *t, void *scratch) {
    t->chunks = 1;
    if (t->s.mode != kCoarse || t->s.n_max <= kCoarseChunk || !scratch) return;
    const int64_t rows = (int64_t)t->s.B * t->s.L;
    t->chunks = (int)((t->s.n_max + kCoarseChunk - 1) / kCoarseChunk);
    t->chunk_ids = reinterpret_cast<int32_t *>(scratch);
    t->chunk_sc = reinterpret_cast<float *>(t->chunk_ids + rows * t->chunks * t->k_sel);
}

// Runs one scoring pass: for the V4 indexer shape the persistent tcgen05 pipeline (coarse
// and fine, which also select) or the per-query tcgen05 kernel, else CUDA cores. With
// `sel` the tensor-core coarse / fine kernels also select (returns true in *fused); with
// `split` the rows' tiles are spread over CTAs and the scores go to p.out.
cudaError_t run_scores(const ScoreParams &p, int32_t *sel, int k_sel, bool *fused,
                       cudaStream_t s, bool split = false, void *scratch = nullptr) {
    *fused = false;
    if (split) {
        ScoreTcParams t{};
        t.s = p;
        return launch_score_tc(t, s);
    }
    if (sel && p.mode != kFlat &&
        score_pipe_supported(p.mode, p.H_i, p.D_i, p.rows_bf16, p.n_max, p.b, p.keep) &&
        (p.mode == kCoarse ? p.means_rows > 0 : p.keys_rows > 0)) {
        ScoreTcParams t{};
        t.s = p;
        t.sel = sel;
        t.k_sel = k_sel;
        set_coarse_chunks(&t, scratch);
        *fused = true;
        return launch_score_pipe(t, s);
    }
    if (p.mode == kFlat && p.out && p.keys_rows > 0 &&
        score_gemm_supported(p.H_i, p.D_i, p.q_bf16, p.rows_bf16, p.B, p.L))
        return launch_score_gemm(p, s);
    if (score_tc_supported(p.mode, p.H_i, p.D_i, p.rows_bf16, p.n_max, p.b) &&
        (p.mode == kCoarse || p.keys_rows > 0)) {
        ScoreTcParams t{};
        t.s = p;
        t.sel = sel;
        t.k_sel = k_sel;
        *fused = p.mode != kFlat;
        return launch_score_tc(t, s);
    }
    return launch_scores_simt(p, s);
}

}  // namespace

int hisa::device_sm_count() {
    static std::atomic<int> counts[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int c = counts[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev].store(c, std::memory_order_relaxed);
    }
    return c;
}

extern "C" {

const char *hisa_status_string(int32_t status) {
    switch (status) {
        case HISA_OK: return "HISA_OK";
        case HISA_EINVAL: return "HISA_EINVAL: invalid argument";
        case HISA_EDTYPE: return "HISA_EDTYPE: unsupported dtype or shape";
        case HISA_EWORKSPACE: return "HISA_EWORKSPACE: workspace missing, misaligned or too small";
        case HISA_ECUDA: return "HISA_ECUDA: CUDA call or launch failed";
        case HISA_EDEVICE: return "HISA_EDEVICE: a kernel flagged bad data";
        default: return "unknown hisa_status";
    }
}

size_t hisa_workspace_bytes(int32_t op, const void *desc) {
    if (!desc) return 0;
    if (op == HISA_OP_COMPRESS)
        return check_compress_desc(static_cast<const hisa_compress_desc *>(desc)) == HISA_OK
                   ? kStatusBytes : 0;
    if (op == HISA_OP_SPARSE_ATTEND) {
        const hisa_attn_desc *d = static_cast<const hisa_attn_desc *>(desc);
        if (check_attn_desc(d) != HISA_OK) return 0;
        const size_t a = attn_part_bytes(d, false), b = attn_part_bytes(d, true);
        return kStatusBytes + round_up(a > b ? a : b);
    }
    const hisa_index_desc *d = static_cast<const hisa_index_desc *>(desc);
    if (check_index_desc(d) != HISA_OK) return 0;
    switch (op) {
        case HISA_OP_INDEX_SCORES:
        case HISA_OP_BLOCK_MEANS:
            return kStatusBytes;
        case HISA_OP_BLOCK_FILTER: {
            if (check_hisa_gate(d) != HISA_OK) return 0;
            const int64_t nb_max = d->Np_max / d->index_block;
            return kStatusBytes + round_up((size_t)n_rows(d) * nb_max * sizeof(float)) +
                   (coarse_gemm_ok(d) ? round_up(coarse_gemm_planes_bytes(d->means_rows)) : 0);
        }
        case HISA_OP_SELECT_TOPK: {
            if (check_hisa_gate(d) != HISA_OK) return 0;
            const int64_t C = (int64_t)d->index_block * d->index_keep;
            return kStatusBytes + round_up((size_t)n_rows(d) * C * sizeof(float));
        }
        case HISA_OP_FLAT_TOPK:
            return kStatusBytes + round_up((size_t)n_rows(d) * d->Np_max * sizeof(float));
        default:
            return 0;
    }
}

hisa_status hisa_workspace_init(void *ws, size_t ws_bytes, hisa_stream_t stream) {
    hisa_status st = check_ws(ws, ws_bytes, kStatusBytes);
    if (st != HISA_OK) return st;
    return from_cuda(cudaMemsetAsync(ws, 0, kStatusBytes, reinterpret_cast<cudaStream_t>(stream)));
}

hisa_status hisa_device_status(const void *ws, hisa_stream_t stream, uint32_t *flags) {
    if (!ws || !flags || !aligned(ws, kAlign)) return HISA_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return HISA_ECUDA;
    *flags = v;
    return v ? HISA_EDEVICE : HISA_OK;
}

hisa_status hisa_index_scores(const hisa_index_desc *d, const void *q, const float *w,
                              const void *keys, const int64_t *key_off, const int32_t *t0,
                              float *scores, int64_t ld_scores, void *ws, size_t ws_bytes,
                              hisa_stream_t stream) {
    hisa_status st = check_index_desc(d);
    if (st != HISA_OK) return st;
    if (!q || !w || !keys || !key_off || !t0 || !scores) return HISA_EINVAL;
    if (!aligned(q, 16) || !aligned(keys, 16) || !aligned(w, 4) || !aligned(scores, 4))
        return HISA_EINVAL;
    if (ld_scores < d->Np_max || ld_scores < 1) return HISA_EINVAL;
    if ((st = check_ws(ws, ws_bytes, hisa_workspace_bytes(HISA_OP_INDEX_SCORES, d))) != HISA_OK)
        return st;
    ScoreParams p = score_params(d, kFlat, q, w, keys, d->k_dtype == HISA_BF16, key_off, t0,
                                 scores, ld_scores, ws);
    p.n_max = d->Np_max;
    bool fused = false;
    return from_cuda(run_scores(p, nullptr, 0, &fused, reinterpret_cast<cudaStream_t>(stream)));
}

hisa_status hisa_block_means(const hisa_index_desc *d, const void *keys, const int64_t *key_off,
                             const int64_t *means_off, const int32_t *first_block, float *means,
                             void *ws, size_t ws_bytes, hisa_stream_t stream) {
    hisa_status st = check_index_desc(d);
    if (st != HISA_OK) return st;
    if (d->index_block < 1) return HISA_EINVAL;
    if (!keys || !key_off || !means_off || !means) return HISA_EINVAL;
    if (!aligned(keys, 16) || !aligned(means, 4)) return HISA_EINVAL;
    if ((st = check_ws(ws, ws_bytes, hisa_workspace_bytes(HISA_OP_BLOCK_MEANS, d))) != HISA_OK)
        return st;
    MeansParams p{};
    p.B = d->B; p.D_i = d->D_i; p.b = d->index_block;
    p.keys = keys; p.keys_bf16 = d->k_dtype == HISA_BF16;
    p.key_off = key_off; p.means_off = means_off; p.first_block = first_block;
    p.means = means; p.Np_max = d->Np_max; p.keys_rows = d->keys_rows;
    p.means_rows = d->means_rows; p.status = status_of(ws);
    p.chained = (d->flags & HISA_FLAG_CHAINED) != 0;
    return from_cuda(launch_block_means(p, d->Np_max / d->index_block,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

hisa_status hisa_block_filter(const hisa_index_desc *d, const void *q, const float *w,
                              const float *means, const int64_t *means_off,
                              const int64_t *key_off, const int32_t *t0, int32_t *top_blk,
                              float *cscores, int64_t ld_cscores, void *ws, size_t ws_bytes,
                              hisa_stream_t stream) {
    hisa_status st = check_index_desc(d);
    if (st != HISA_OK) return st;
    if ((st = check_hisa_gate(d)) != HISA_OK) return st;
    if (!q || !w || !means || !means_off || !key_off || !t0 || !top_blk) return HISA_EINVAL;
    if (!aligned(q, 16) || !aligned(means, 16) || !aligned(w, 4)) return HISA_EINVAL;
    const int64_t nb_max = d->Np_max / d->index_block;
    if (cscores && ld_cscores < nb_max) return HISA_EINVAL;
    if ((st = check_ws(ws, ws_bytes, hisa_workspace_bytes(HISA_OP_BLOCK_FILTER, d))) != HISA_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool gemm = coarse_gemm_ok(d) && nb_max > 0;
    const bool split = !gemm && split_rows(d, kCoarse, nb_max);
    const bool tc = !gemm && !split && score_tc_supported(kCoarse, d->H_i, d->D_i, 0, nb_max, d->index_block);
    float *buf = cscores ? cscores : (tc ? nullptr : scratch_of(ws));
    const int64_t ld = cscores ? ld_cscores : (nb_max > 0 ? nb_max : 1);
    ScoreParams p = score_params(d, kCoarse, q, w, means, 0, key_off, t0, buf, ld, ws);
    p.means_off = means_off;
    p.n_max = nb_max;
    bool fused = false;
    cudaError_t e;
    if (gemm) {
        void *planes = reinterpret_cast<char *>(ws) + kStatusBytes +
                       round_up((size_t)n_rows(d) * nb_max * sizeof(float));
        e = launch_coarse_gemm(p, planes, s);
    } else {
        e = run_scores(p, top_blk, d->index_keep, &fused, s, split, scratch_of(ws));
    }
    if (e != cudaSuccess) return HISA_ECUDA;
    if (fused) return HISA_OK;
    SelectParams sp{};
    sp.mode = kCoarse; sp.B = d->B; sp.L = d->L; sp.b = d->index_block; sp.keep = d->index_keep;
    sp.k = d->index_keep;
    sp.scores = buf; sp.ld = ld; sp.key_off = key_off; sp.out = top_blk;
    sp.Np_max = d->Np_max; sp.keys_rows = d->keys_rows; sp.status = status_of(ws);
    return from_cuda(launch_select(sp, nb_max, s));
}

hisa_status hisa_block_filter_append(const hisa_index_desc *d, const void *q, const float *w,
                                     const void *keys, const int64_t *key_off, float *means,
                                     const int64_t *means_off, const int32_t *first_block,
                                     const int32_t *t0, int32_t *top_blk, float *cscores,
                                     int64_t ld_cscores, void *ws, size_t ws_bytes,
                                     hisa_stream_t stream) {
    hisa_status st = check_index_desc(d);
    if (st != HISA_OK) return st;
    if ((st = check_hisa_gate(d)) != HISA_OK) return st;
    if (!q || !w || !keys || !means || !means_off || !key_off || !t0 || !top_blk) return HISA_EINVAL;
    if (!aligned(q, 16) || !aligned(keys, 16) || !aligned(means, 16) || !aligned(w, 4))
        return HISA_EINVAL;
    const int64_t nb_max = d->Np_max / d->index_block;
    if (cscores && ld_cscores < nb_max) return HISA_EINVAL;
    if ((st = check_ws(ws, ws_bytes, hisa_workspace_bytes(HISA_OP_BLOCK_FILTER, d))) != HISA_OK)
        return st;
    const bool fused = d->L == 1 && d->k_dtype == HISA_BF16 && d->index_block == 64 && d->D_i == 128 &&
                       d->means_rows > 0 && d->keys_rows > 0 && !split_rows(d, kCoarse, nb_max) &&
                       score_pipe_supported(kCoarse, d->H_i, d->D_i, 0, nb_max, d->index_block,
                                            d->index_keep);
    if (!fused) {
        st = hisa_block_means(d, keys, key_off, means_off, first_block, means, ws, ws_bytes, stream);
        if (st != HISA_OK) return st;
        return hisa_block_filter(d, q, w, means, means_off, key_off, t0, top_blk, cscores,
                                 ld_cscores, ws, ws_bytes, stream);
    }
    ScoreParams p = score_params(d, kCoarse, q, w, means, 0, key_off, t0, cscores,
                                 cscores ? ld_cscores : 0, ws);
    p.means_off = means_off;
    p.n_max = nb_max;
    ScoreTcParams t{};
    t.s = p;
    t.sel = top_blk;
    t.k_sel = d->index_keep;
    t.append_keys = keys;
    t.first_block = first_block;
    set_coarse_chunks(&t, scratch_of(ws));
    return from_cuda(launch_score_pipe(t, reinterpret_cast<cudaStream_t>(stream)));
}

hisa_status hisa_select_topk(const hisa_index_desc *d, const void *q, const float *w,
                             const void *keys, const int64_t *key_off, const int32_t *t0,
                             const int32_t *top_blk, int32_t *I, float *fscores, void *ws,
                             size_t ws_bytes, hisa_stream_t stream) {
    hisa_status st = check_index_desc(d);
    if (st != HISA_OK) return st;
    if ((st = check_hisa_gate(d)) != HISA_OK) return st;
    if (!q || !w || !keys || !key_off || !t0 || !top_blk || !I) return HISA_EINVAL;
    if (!aligned(q, 16) || !aligned(keys, 16) || !aligned(w, 4)) return HISA_EINVAL;
    if ((st = check_ws(ws, ws_bytes, hisa_workspace_bytes(HISA_OP_SELECT_TOPK, d))) != HISA_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t C = (int64_t)d->index_block * d->index_keep;
    const bool split = split_rows(d, kFine, C) && d->keys_rows > 0;
    const bool tc = !split && score_tc_supported(kFine, d->H_i, d->D_i, d->k_dtype == HISA_BF16, C,
                                                 d->index_block) && d->keys_rows > 0;
    float *buf = fscores ? fscores : (tc ? nullptr : scratch_of(ws));
    ScoreParams p = score_params(d, kFine, q, w, keys, d->k_dtype == HISA_BF16, key_off, t0, buf,
                                 C, ws);
    p.top_blk = top_blk;
    p.n_max = C;
    bool fused = false;
    cudaError_t e = run_scores(p, I, d->index_topk, &fused, s, split);
    if (e != cudaSuccess) return HISA_ECUDA;
    if (fused) return HISA_OK;
    SelectParams sp{};
    sp.mode = kFine; sp.B = d->B; sp.L = d->L; sp.b = d->index_block; sp.keep = d->index_keep;
    sp.k = d->index_topk;
    sp.scores = buf; sp.ld = C; sp.key_off = key_off; sp.top_blk = top_blk; sp.out = I;
    sp.Np_max = d->Np_max; sp.keys_rows = d->keys_rows; sp.status = status_of(ws);
    return from_cuda(launch_select(sp, C, s));
}

hisa_status hisa_flat_topk(const hisa_index_desc *d, const void *q, const float *w,
                           const void *keys, const int64_t *key_off, const int32_t *t0,
                           int32_t *I, void *ws, size_t ws_bytes, hisa_stream_t stream) {
    hisa_status st = check_index_desc(d);
    if (st != HISA_OK) return st;
    if (!q || !w || !keys || !key_off || !t0 || !I) return HISA_EINVAL;
    if (!aligned(q, 16) || !aligned(keys, 16) || !aligned(w, 4)) return HISA_EINVAL;
    if ((st = check_ws(ws, ws_bytes, hisa_workspace_bytes(HISA_OP_FLAT_TOPK, d))) != HISA_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t ld = d->Np_max > 0 ? d->Np_max : 1;
    float *buf = scratch_of(ws);
    ScoreParams p = score_params(d, kFlat, q, w, keys, d->k_dtype == HISA_BF16, key_off, t0, buf,
                                 ld, ws);
    p.n_max = d->Np_max;
    bool fused = false;
    cudaError_t e = run_scores(p, nullptr, 0, &fused, s);
    if (e != cudaSuccess) return HISA_ECUDA;
    SelectParams sp{};
    sp.mode = kFlat; sp.B = d->B; sp.L = d->L; sp.b = d->index_block; sp.keep = d->index_keep;
    sp.k = d->index_topk;
    sp.scores = buf; sp.ld = ld; sp.key_off = key_off; sp.out = I;
    sp.Np_max = d->Np_max; sp.keys_rows = d->keys_rows; sp.status = status_of(ws);
    sp.work = buf;                       // the scores are scratch: long rows reduce in place
    return from_cuda(launch_select(sp, d->Np_max, s));
}

hisa_status hisa_compress_append(const hisa_compress_desc *d, const float *kv, const float *gate,
                                 const int64_t *tok_off, const int32_t *p_first,
                                 const int32_t *n_new, const float *ape, const float *norm_w,
                                 void *keys, const int64_t *key_off, float *means,
                                 const int64_t *means_off, void *ws, size_t ws_bytes,
                                 hisa_stream_t stream) {
    hisa_status st = check_compress_desc(d);
    if (st != HISA_OK) return st;
    if (!kv || !gate || !tok_off || !p_first || !n_new || !ape || !norm_w || !keys || !key_off)
        return HISA_EINVAL;
    if (means && !means_off) return HISA_EINVAL;
    if (!aligned(kv, 4) || !aligned(gate, 4) || !aligned(ape, 4) || !aligned(norm_w, 4) ||
        !aligned(keys, d->k_dtype == HISA_BF16 ? 2 : 4) || (means && !aligned(means, 4)))
        return HISA_EINVAL;
    if ((st = check_ws(ws, ws_bytes, hisa_workspace_bytes(HISA_OP_COMPRESS, d))) != HISA_OK)
        return st;
    CompressParams p{};
    p.B = d->B; p.D = d->D_i; p.C = d->overlap ? 2 * d->D_i : d->D_i; p.r = d->r;
    p.overlap = d->overlap; p.rope_dims = d->rope_dims; p.b = d->index_block;
    p.n_new_max = d->n_new_max; p.k_bf16 = d->k_dtype == HISA_BF16; p.eps = d->eps;
    p.log_theta = std::log((double)d->rope_theta);
    p.kv = kv; p.gate = gate; p.ape = ape; p.norm_w = norm_w;
    p.tok_off = tok_off; p.p_first = p_first; p.n_new = n_new;
    p.keys = keys; p.key_off = key_off;
    p.means = d->index_block > 0 ? means : nullptr; p.means_off = means_off;
    p.tok_rows = d->tok_rows; p.keys_rows = d->keys_rows; p.means_rows = d->means_rows;
    p.status = status_of(ws);
    p.chained = (d->flags & HISA_FLAG_CHAINED) != 0;
    return from_cuda(launch_compress(p, reinterpret_cast<cudaStream_t>(stream)));
}

hisa_status hisa_sparse_attend(const hisa_attn_desc *d, const void *q, const void *local_kv,
                               const int32_t *local_len, const int32_t *local_pos0,
                               const void *pooled_kv, const int64_t *kv_off, const int32_t *I,
                               const float *sinks, const int32_t *t0, void *out, void *ws,
                               size_t ws_bytes, hisa_stream_t stream) {
    hisa_status st = check_attn_desc(d);
    if (st != HISA_OK) return st;
    if (!q || !local_len || !local_pos0 || !kv_off || !sinks || !t0 || !out) return HISA_EINVAL;
    if (d->W_max > 0 && !local_kv) return HISA_EINVAL;
    if (d->Np_max > 0 && !pooled_kv) return HISA_EINVAL;
    if (I && d->k < 1) return HISA_EINVAL;
    if (!aligned(q, 16) || !aligned(local_kv, 16) || !aligned(pooled_kv, 16) || !aligned(out, 16))
        return HISA_EINVAL;
    if ((st = check_ws(ws, ws_bytes, hisa_workspace_bytes(HISA_OP_SPARSE_ATTEND, d))) != HISA_OK)
        return st;
    const bool dense = I == nullptr;
    AttnParams p{};
    p.B = d->B; p.L = d->L; p.H = d->H; p.Dh = d->Dh; p.window = d->window; p.W_max = d->W_max;
    p.r = d->r; p.k = dense ? 0 : d->k;
    p.causal = d->L > 1;
    p.Np_max = d->Np_max;
    p.kv_rows = d->kv_rows;
    p.scale = d->scale > 0.f ? d->scale : (float)(1.0 / std::sqrt((double)d->Dh));
    p.q = q; p.local_kv = local_kv; p.local_len = local_len; p.local_pos0 = local_pos0;
    p.pooled_kv = pooled_kv; p.kv_off = kv_off; p.I = I; p.sinks = sinks; p.t0 = t0;
    p.out = out;
    p.out_bf16 = d->out_dtype == HISA_BF16;
    p.part = scratch_of(ws);
    int64_t per = 0;
    p.nsplit = pick_nsplit((int64_t)d->B * d->L, attn_list_len(d, dense), &per);
    p.rows_per_split = (int)per;
    p.kv_bf16 = d->kv_dtype == HISA_BF16;
    p.status = status_of(ws);
    p.chained = (d->flags & HISA_FLAG_CHAINED) != 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (attend_tc_supported(d->H, d->Dh, p.kv_bf16)) return from_cuda(launch_attend_tc(p, s));
    return from_cuda(launch_attend_simt(p, s));
}

}  // extern "C"
