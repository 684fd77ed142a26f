// Per-query top-k of a row of scores held in global memory ([HiSA issue] "Conventions":
// argpartition returns an unordered top-k set; the flat, coarse and fine stages all take
// one). One CTA owns one query row; the selection itself is block_topk.
#include "select_core.cuh"

namespace hisa {

// Rows of at most kSmemSel scores are selected from shared memory (the short form); longer
// flat rows in chunks of kChunk when the caller provides candidate space.
constexpr int kSmemSel = 8192;
constexpr int kChunk = 8192;
constexpr size_t kMergeSmem = 200 * 1024;                 // candidate scores + ids of one row

template <int NT>
__global__ void __launch_bounds__(NT) k_select(SelectParams p) {
    __shared__ SelectShared<NT> sh;
    __shared__ int s_raw[64], s_blk[64];
    __shared__ int s_bad;
    grid_dep_wait();                                 // the scores are the previous grid's

    const int row = blockIdx.x;
    const int bq = row / p.L;
    const int tid = threadIdx.x;
    int32_t *out = p.out + (int64_t)row * p.k;

    const int64_t k0 = p.key_off[bq];
    const int64_t Np = p.key_off[bq + 1] - k0;
    bool ok = seq_ok(p.key_off, bq, p.Np_max, p.keys_rows);
    int64_t n = 0;
    if (!ok) {
        if (tid == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
    } else if (p.mode == kFlat) {
        n = Np;
    } else if (Np < (int64_t)p.b * p.keep) {
        ok = false;
        if (tid == 0) flag(p.status, HISA_DEV_GATE);
    } else {
        n = (p.mode == kCoarse) ? Np / p.b : (int64_t)p.keep * p.b;
    }
    if (ok && p.mode == kFine) {
        // the kept blocks in ascending order (candidates in ascending pos): all are loaded at
        // once, then thread s places block s by its rank, ties by index
        if (tid < p.keep) s_raw[tid] = p.top_blk[(int64_t)row * p.keep + tid];
        if (tid == 0) s_bad = 0;
        __syncthreads();
        if (tid < p.keep) {
            const int v = s_raw[tid];
            int rank = 0;
            for (int u = 0; u < p.keep; ++u) {
                const int o = s_raw[u];
                rank += (o < v || (o == v && u < tid)) ? 1 : 0;
            }
            s_blk[rank] = v;
            if (v < 0 || (int64_t)v >= Np / p.b) s_bad = 1;
        }
        __syncthreads();
        if (tid == 0 && s_bad) flag(p.status, HISA_DEV_BAD_BLOCK);
        ok = !s_bad;
    }
    if (!ok) {
        for (int e = tid; e < p.k; e += NT) out[e] = -1;
        return;
    }
    const float *sc = p.scores + (int64_t)row * p.ld;
    const int64_t kout = n < (int64_t)p.k ? n : (int64_t)p.k;
    extern __shared__ __align__(16) float s_sc[];
    if (n <= p.smem_n) {
        // the row in shared memory, then the short-form select (short rows are the common case)
        for (int64_t e = tid; e < n; e += NT) s_sc[e] = sc[e];
        __syncthreads();
        if (p.mode == kFine) {
            const int b = p.b;
            small_topk<NT, 0, 0>(s_sc, (int)n, (int)kout, out,
                                 [&](int64_t i) { return (int32_t)((int64_t)s_blk[i / b] * b + (i % b)); },
                                 sh, p.status);
        } else {
            small_topk<NT, 0, 0>(s_sc, (int)n, (int)kout, out, [](int64_t i) { return (int32_t)i; }, sh,
                                 p.status);
        }
    } else if (p.mode == kFine) {
        const int b = p.b;
        block_topk<NT>(sc, n, kout, out,
                       [&](int64_t i) { return (int32_t)((int64_t)s_blk[i / b] * b + (i % b)); },
                       sh, p.status);
    } else {
        block_topk<NT>(sc, n, kout, out, [](int64_t i) { return (int32_t)i; }, sh, p.status);
    }
    for (int64_t e = kout + tid; e < p.k; e += NT) out[e] = -1;
}

// Chunked flat select, first level. CTA (row, c) owns scores [c kChunk, c kChunk + len).
// A chunk longer than 2k is reduced in place: its top k, as (score, id) pairs in
// ascending id order, overwrite its first 2k floats (the chunk is in shared memory by
// then, and no other CTA touches it). Shorter chunks are left as they are. The global top
// k lies in the union of the chunks' top k, ties included, since every chunk keeps its
// equal scores by ascending id.
template <int NT>
__global__ void __launch_bounds__(NT) k_select_chunks(SelectParams p) {
    __shared__ SelectShared<NT> sh;
    __shared__ int32_t s_col[kMaxTopk];
    extern __shared__ __align__(16) float s_sc[];
    grid_dep_wait();
    const int row = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
    const int bq = row / p.L;
    if (!seq_ok(p.key_off, bq, p.Np_max, p.keys_rows)) return;   // the merge flags it
    const int64_t Np = p.key_off[bq + 1] - p.key_off[bq];
    int64_t len = Np - (int64_t)c * kChunk;
    len = len > kChunk ? kChunk : len;
    if (len <= 2 * (int64_t)p.k) return;
    float *w = p.work + (int64_t)row * p.ld + (int64_t)c * kChunk;
    for (int64_t e = tid; e < len; e += NT) s_sc[e] = w[e];
    __syncthreads();
    small_topk<NT, 0, 0>(s_sc, (int)len, p.k, s_col, [](int64_t i) { return (int32_t)i; }, sh, p.status);
    __syncthreads();
    for (int e = tid; e < p.k; e += NT) {
        w[2 * e] = s_sc[s_col[e]];
        w[2 * e + 1] = __int_as_float(c * kChunk + s_col[e]);
    }
}

// Second level: one CTA per row gathers every chunk's candidates in chunk order (so ids
// ascend), selects the top k among them and writes their ids; bad rows are all -1.
template <int NT>
__global__ void __launch_bounds__(NT) k_select_merge(SelectParams p, int cap) {
    __shared__ SelectShared<NT> sh;
    extern __shared__ __align__(16) float s_sc[];
    int32_t *s_id = reinterpret_cast<int32_t *>(s_sc + cap);
    grid_dep_wait();
    const int row = blockIdx.x, tid = threadIdx.x;
    const int bq = row / p.L;
    int32_t *out = p.out + (int64_t)row * p.k;
    int64_t n = 0;
    if (!seq_ok(p.key_off, bq, p.Np_max, p.keys_rows)) {
        if (tid == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
    } else {
        n = p.key_off[bq + 1] - p.key_off[bq];
    }
    const int64_t kout = n < (int64_t)p.k ? n : (int64_t)p.k;
    const float *w = p.work + (int64_t)row * p.ld;
    // every chunk but the last is longer than 2k (k <= 2048 < kChunk / 2) and holds k
    // candidates, so candidate i of the row (chunk order) is entry i % k of chunk i / k,
    // or of the last chunk past them: all loads go out at once
    const int64_t nchunk = (n + kChunk - 1) / kChunk;
    const int64_t last = n - (nchunk - 1) * kChunk;               // length of the last chunk
    const bool last_reduced = last > 2 * (int64_t)p.k;
    const int m = n > 0 ? (int)((nchunk - 1) * p.k + (last_reduced ? p.k : last)) : 0;
#pragma unroll 4
    for (int i = tid; i < m; i += NT) {
        int64_t c = i / p.k;
        if (c > nchunk - 1) c = nchunk - 1;
        const int e = (int)(i - c * p.k);
        const float *wc = w + c * kChunk;
        if (c < nchunk - 1 || last_reduced) {
            s_sc[i] = wc[2 * e];
            s_id[i] = __float_as_int(wc[2 * e + 1]);
        } else {
            s_sc[i] = wc[e];
            s_id[i] = (int32_t)(c * kChunk + e);
        }
    }
    __syncthreads();
    const auto ids = [&](int64_t i) { return s_id[i]; };
    if (kout > 0 && m <= 8 * NT)
        small_topk<NT, 0, 0>(s_sc, m, (int)kout, out, ids, sh, p.status);
    else if (kout > 0)                               // the usual case: the binned form, inlined
        small_topk_binned_body<NT, 0, 0>(s_sc, m, (int)kout, out, ids, sh, p.status);
    for (int64_t e = kout + tid; e < p.k; e += NT) out[e] = -1;
}

// Candidates of a row of at most ld scores after the first level.
int64_t chunked_candidates(int64_t ld, int k) {
    const int64_t nchunk = (ld + kChunk - 1) / kChunk;
    return (nchunk - 1) * (int64_t)k + 2 * (int64_t)k;
}

cudaError_t launch_select(const SelectParams &p, int64_t n_max, cudaStream_t s) {
    const unsigned rows = (unsigned)(p.B * p.L);
    if (rows == 0) return cudaSuccess;
    if (p.mode == kFlat && p.work && chunked_select_fits(p.ld, p.k) && n_max > kSmemSel) {
        const int64_t nchunk = (p.ld + kChunk - 1) / kChunk;
        const int cap = (int)chunked_candidates(p.ld, p.k);
        const cudaError_t a1 = smem_attr_once<k_select_chunks<1024>>(kChunk * 4);
        const cudaError_t a2 = smem_attr_once<k_select_merge<1024>>((int)kMergeSmem);
        if (a1 != cudaSuccess) return a1;
        if (a2 != cudaSuccess) return a2;
        // every select kernel waits before its first global access, so each may be launched
        // as a programmatic dependent of the kernel before it (the scoring kernel, or the
        // first level)
        cudaError_t e = launch_pdl(k_select_chunks<1024>, dim3(rows, (unsigned)nchunk), dim3(1024),
                                   (size_t)kChunk * 4, s, 1, p);
        if (e != cudaSuccess) return e;
        return launch_pdl(k_select_merge<1024>, dim3(rows), dim3(1024), (size_t)cap * 8, s, 1, p, cap);
    }
    SelectParams q = p;
    q.smem_n = n_max <= kSmemSel ? (int)n_max : 0;
    const size_t smem = (size_t)q.smem_n * 4;
    // short rows (the coarse stage of many prefill rows): four warps, four columns a thread,
    // so that sixteen CTAs share an SM
    if (n_max <= 512) return launch_pdl(k_select<128>, dim3(rows), dim3(128), smem, s, 1, q);
    const cudaError_t a = smem_attr_once<k_select<1024>>(kSmemSel * 4);
    if (a != cudaSuccess) return a;
    return launch_pdl(k_select<1024>, dim3(rows), dim3(1024), smem, s, 1, q);
}

bool chunked_select_fits(int64_t ld, int k) {
    if (ld <= kSmemSel || k < 1 || 2 * k > kChunk || k > kMaxTopk) return false;
    const int64_t cap = chunked_candidates(ld, k);
    return cap <= kSmallMax && (size_t)cap * 8 <= kMergeSmem;
}

}  // namespace hisa
