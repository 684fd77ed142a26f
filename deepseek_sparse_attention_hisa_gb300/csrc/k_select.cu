// Per-query top-k of a row of scores held in global memory ([HiSA issue] "Conventions":
// argpartition returns an unordered top-k set; the flat, coarse and fine stages all take
// one). One CTA owns one query row; the selection itself is block_topk.
#include "select_core.cuh"

namespace hisa {

template <int NT>
__global__ void __launch_bounds__(NT) k_select(SelectParams p) {
    __shared__ SelectShared<NT> sh;
    __shared__ int s_blk[64];
    __shared__ int s_bad;

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
        if (tid == 0) {
            const int32_t *tb = p.top_blk + (int64_t)row * p.keep;
            int bad = 0;
            for (int s = 0; s < p.keep; ++s) {  // insertion sort: candidates in ascending pos
                int v = tb[s], u = s;
                if (v < 0 || (int64_t)v >= Np / p.b) bad = 1;
                while (u > 0 && s_blk[u - 1] > v) { s_blk[u] = s_blk[u - 1]; --u; }
                s_blk[u] = v;
            }
            s_bad = bad;
            if (bad) flag(p.status, HISA_DEV_BAD_BLOCK);
        }
        __syncthreads();
        ok = !s_bad;
    }
    if (!ok) {
        for (int e = tid; e < p.k; e += NT) out[e] = -1;
        return;
    }
    const float *sc = p.scores + (int64_t)row * p.ld;
    const int64_t kout = n < (int64_t)p.k ? n : (int64_t)p.k;
    if (p.mode == kFine) {
        const int b = p.b;
        block_topk<NT>(sc, n, kout, out,
                       [&](int64_t i) { return (int32_t)((int64_t)s_blk[i / b] * b + (i % b)); },
                       sh, p.status);
    } else {
        block_topk<NT>(sc, n, kout, out, [](int64_t i) { return (int32_t)i; }, sh, p.status);
    }
    for (int64_t e = kout + tid; e < p.k; e += NT) out[e] = -1;
}

cudaError_t launch_select(const SelectParams &p, int64_t n_max, cudaStream_t s) {
    const unsigned rows = (unsigned)(p.B * p.L);
    if (n_max <= 256)
        k_select<256><<<rows, 256, 0, s>>>(p);
    else
        k_select<1024><<<rows, 1024, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace hisa
