// Indexer scoring on CUDA cores (any supported shape, f32 or bf16 inputs), and the
// block-mean representatives.
//
// score = sum_h relu(q_h . row) * scale * w_h, accumulated in f32
// ([HiSA issue] "Flat selection (baseline path)"; the coarse stage applies the same
// head combine to block means, the fine stage to the candidate rows, "HiSA decode
// path"). One thread owns one scored row: it holds the row in registers and walks
// the heads, with q broadcast from shared memory.
#include "hisa_internal.cuh"

namespace hisa {

template <int D, typename T>
__device__ __forceinline__ void load_row(const T *src, float (&v)[D]);

template <int D>
__device__ __forceinline__ void load_row(const float *src, float (&v)[D]) {
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
    for (int i = 0; i < D / 4; ++i) {
        float4 x = __ldg(s4 + i);
        v[4 * i + 0] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
    }
}

template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *src, float (&v)[D]) {
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        uint4 x = __ldg(s4 + i);
        const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&x);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float2 f = __bfloat1622float2(h2[e]);
            v[8 * i + 2 * e] = f.x;
            v[8 * i + 2 * e + 1] = f.y;
        }
    }
}

template <int D, typename QT, typename KT>
__global__ void __launch_bounds__(256) k_scores_simt(ScoreParams p) {
    extern __shared__ __align__(16) float smem[];
    float *sq = smem;                      // [H_i][D] f32
    float *sw = sq + p.H_i * D;            // [H_i] scaled weights
    int *sblk = reinterpret_cast<int *>(sw + p.H_i);  // [keep] kept blocks, ascending
    int *sraw = sblk + 64;                             // [keep] kept blocks as read

    const int row = blockIdx.x;            // b * L + j
    const int bq = row / p.L;
    const int j = row - bq * p.L;
    const int64_t k0 = p.key_off[bq];
    const int64_t Np = p.key_off[bq + 1] - k0;
    if (!seq_ok(p.key_off, bq, p.Np_max, p.keys_rows)) {
        if (threadIdx.x == 0 && blockIdx.y == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
        return;
    }
    int64_t n;
    if (p.mode == kFlat) {
        n = Np;
    } else {
        if (Np < (int64_t)p.b * p.keep) {  // HiSA gate, per sequence
            if (threadIdx.x == 0 && blockIdx.y == 0) flag(p.status, HISA_DEV_GATE);
            return;
        }
        n = (p.mode == kCoarse) ? Np / p.b : (int64_t)p.keep * p.b;
        if (p.mode == kCoarse && !means_ok(p.means_off, bq, n, p.means_rows)) {
            if (threadIdx.x == 0 && blockIdx.y == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
            return;
        }
    }
    const int64_t i0 = (int64_t)blockIdx.y * blockDim.x;
    if (i0 >= n) return;

    const QT *qrow = reinterpret_cast<const QT *>(p.q) + (int64_t)row * p.H_i * D;
    for (int e = threadIdx.x; e < p.H_i * D; e += blockDim.x) sq[e] = to_f32(qrow[e]);
    for (int h = threadIdx.x; h < p.H_i; h += blockDim.x)
        sw[h] = p.w[(int64_t)row * p.H_i + h] * p.head_scale;
    if (p.mode == kFine && (int)threadIdx.x < p.keep)
        sraw[threadIdx.x] = p.top_blk[(int64_t)row * p.keep + threadIdx.x];
    __syncthreads();
    if (p.mode == kFine && (int)threadIdx.x < p.keep) {
        // candidates in ascending pos: thread s places kept block s by its rank, ties by index
        const int v = sraw[threadIdx.x];
        int rank = 0;
        for (int u = 0; u < p.keep; ++u) {
            const int o = sraw[u];
            rank += (o < v || (o == v && u < (int)threadIdx.x)) ? 1 : 0;
        }
        sblk[rank] = v;
    }
    __syncthreads();

    const int64_t i = i0 + threadIdx.x;
    if (i >= n) return;
    const int64_t V = p.causal ? visible_len((int64_t)p.t0[bq] + j, p.r, Np) : Np;
    int64_t pos, src;
    if (p.mode == kFlat) {
        pos = i;
        src = k0 + i;
    } else if (p.mode == kCoarse) {
        pos = i * p.b;                     // a block is eligible iff its first row is visible
        src = p.means_off[bq] + i;
    } else {
        const int blk = sblk[i / p.b];
        if (blk < 0 || (int64_t)blk >= Np / p.b) {
            flag(p.status, HISA_DEV_BAD_BLOCK);
            p.out[(int64_t)row * p.ld_out + i] = kNeg;
            return;
        }
        pos = (int64_t)blk * p.b + (i % p.b);
        src = k0 + pos;
    }
    float result = kNeg;
    if (pos < V) {
        float kv[D];
        load_row<D>(reinterpret_cast<const KT *>(p.rows) + src * D, kv);
        float acc = 0.f;
        for (int h = 0; h < p.H_i; ++h) {
            const float4 *qh = reinterpret_cast<const float4 *>(sq + h * D);
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int d = 0; d < D / 4; ++d) {
                float4 qv = qh[d];
                a0 = fmaf(qv.x, kv[4 * d + 0], a0);
                a1 = fmaf(qv.y, kv[4 * d + 1], a1);
                a2 = fmaf(qv.z, kv[4 * d + 2], a2);
                a3 = fmaf(qv.w, kv[4 * d + 3], a3);
            }
            const float dot = (a0 + a1) + (a2 + a3);
            acc = fmaf(sw[h], fmaxf(dot, 0.f), acc);
        }
        result = acc;
    }
    p.out[(int64_t)row * p.ld_out + i] = result;
}

template <int D, typename QT, typename KT>
static cudaError_t launch_scores_t(const ScoreParams &p, cudaStream_t s) {
    const size_t smem = (size_t)p.H_i * D * 4 + (size_t)p.H_i * 4 + 2 * 64 * 4;
    const cudaError_t attr = smem_attr_once<k_scores_simt<D, QT, KT>>(128 * 128 * 4 + 1024);
    if (attr != cudaSuccess) return attr;
    const int64_t tiles = (p.n_max + 255) / 256;
    if (tiles == 0) return cudaSuccess;
    dim3 grid((unsigned)(p.B * p.L), (unsigned)tiles);
    k_scores_simt<D, QT, KT><<<grid, 256, smem, s>>>(p);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_scores_d(const ScoreParams &p, cudaStream_t s) {
    if (p.q_bf16) {
        if (p.rows_bf16) return launch_scores_t<D, __nv_bfloat16, __nv_bfloat16>(p, s);
        return launch_scores_t<D, __nv_bfloat16, float>(p, s);
    }
    if (p.rows_bf16) return launch_scores_t<D, float, __nv_bfloat16>(p, s);
    return launch_scores_t<D, float, float>(p, s);
}

cudaError_t launch_scores_simt(const ScoreParams &p, cudaStream_t s) {
    switch (p.D_i) {
        case 32: return launch_scores_d<32>(p, s);
        case 64: return launch_scores_d<64>(p, s);
        case 128: return launch_scores_d<128>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------
// block means ([HiSA issue] "HiSA decode path": rep = mean of the b rows of a block)
// ---------------------------------------------------------------------------
template <typename KT>
__global__ void k_block_means(MeansParams p) {
    const int bq = blockIdx.y;
    const int64_t k0 = p.key_off[bq];
    const int64_t Np = p.key_off[bq + 1] - k0;
    if (!seq_ok(p.key_off, bq, p.Np_max, p.keys_rows)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
        return;
    }
    const int64_t nb = Np / p.b;
    const int64_t m0 = p.means_off[bq];
    if (!means_ok(p.means_off, bq, nb, p.means_rows)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
        return;
    }
    int64_t fb = p.first_block ? (int64_t)p.first_block[bq] : 0;
    if (fb < 0) fb = 0;
    const KT *keys = reinterpret_cast<const KT *>(p.keys);
    const float inv_div = (float)p.b;
    for (int64_t beta = fb + blockIdx.x; beta < nb; beta += gridDim.x) {
        for (int d = threadIdx.x; d < p.D_i; d += blockDim.x) {
            const KT *src = keys + (k0 + beta * p.b) * p.D_i + d;
            // f32 sum in row order; loads are issued 16 rows at a time
            float s = 0.f;
            int i = 0;
            for (; i + 16 <= p.b; i += 16) {
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = to_f32(src[(int64_t)(i + u) * p.D_i]);
#pragma unroll
                for (int u = 0; u < 16; ++u) s += v[u];
            }
            for (; i < p.b; ++i) s += to_f32(src[(int64_t)i * p.D_i]);
            p.means[(m0 + beta) * p.D_i + d] = s / inv_div;
        }
    }
}

// The same means, one block per pass with all of its b * D_i keys in flight at once: the
// block is one contiguous run of keys, copied with 16-byte loads into shared memory as
// f32, then each thread sums one dimension: eight partial sums over the rows i = k (mod 8)
// in row order, combined by a fixed pairwise tree (the order the coarse kernel's append
// path uses too, so a block mean has the same bits whichever kernel wrote it).
constexpr int kMeansThreads = 256;
constexpr int kMeansStage = 8192;                      // f32 elements staged per block

template <typename KT>
__global__ void __launch_bounds__(kMeansThreads) k_block_means_staged(MeansParams p) {
    __shared__ float stage[kMeansStage];
    grid_dep_wait();
    const int bq = blockIdx.y;
    const int64_t k0 = p.key_off[bq];
    const int64_t Np = p.key_off[bq + 1] - k0;
    if (!seq_ok(p.key_off, bq, p.Np_max, p.keys_rows)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
        return;
    }
    const int64_t nb = Np / p.b;
    const int64_t m0 = p.means_off[bq];
    if (!means_ok(p.means_off, bq, nb, p.means_rows)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
        return;
    }
    int64_t fb = p.first_block ? (int64_t)p.first_block[bq] : 0;
    if (fb < 0) fb = 0;
    constexpr int kPer = 16 / (int)sizeof(KT);          // keys per 16-byte load
    const int n = p.b * p.D_i;                          // keys of one block
    const KT *keys = reinterpret_cast<const KT *>(p.keys);
    const float inv_div = (float)p.b;
    // a block that one round of loads covers (bf16 64 x 128): the next block's loads are
    // issued before this one is summed, so a CTA keeps a block in flight throughout
    const bool one_round = n / kPer <= 4 * kMeansThreads;
    uint4 nxt[4];
    auto load_block = [&](int64_t beta, uint4 *u) {
        const uint4 *src = reinterpret_cast<const uint4 *>(keys + (k0 + beta * p.b) * p.D_i);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int vv = (int)threadIdx.x + m * kMeansThreads;
            if (vv < n / kPer) u[m] = __ldg(src + vv);
        }
    };
    if (one_round && fb + blockIdx.x < nb) load_block(fb + blockIdx.x, nxt);
    for (int64_t beta = fb + blockIdx.x; beta < nb; beta += gridDim.x) {
        for (int v = threadIdx.x; v < n / kPer; v += 4 * kMeansThreads) {
            uint4 u[4];
            if (one_round) {
#pragma unroll
                for (int m = 0; m < 4; ++m) u[m] = nxt[m];
            } else {
                const uint4 *src = reinterpret_cast<const uint4 *>(keys + (k0 + beta * p.b) * p.D_i);
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    if (v + m * kMeansThreads < n / kPer) u[m] = __ldg(src + v + m * kMeansThreads);
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int vv = v + m * kMeansThreads;
                if (vv < n / kPer) {
                    const KT *x = reinterpret_cast<const KT *>(&u[m]);
#pragma unroll
                    for (int e = 0; e < kPer; ++e) stage[vv * kPer + e] = to_f32(x[e]);
                }
            }
        }
        if (one_round && beta + gridDim.x < nb) load_block(beta + gridDim.x, nxt);
        __syncthreads();
        for (int d = threadIdx.x; d < p.D_i; d += kMeansThreads) {
            // partial sums over the rows i = k (mod 8), each in row order, then the fixed
            // pairwise tree ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7))
            float ps[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float a = 0.f;
                for (int i = k; i < p.b; i += 8) a += stage[i * p.D_i + d];
                ps[k] = a;
            }
            const float s = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            p.means[(m0 + beta) * p.D_i + d] = s / inv_div;
        }
        __syncthreads();
    }
}

// bf16 keys, D_i and b multiples of 8, b <= 64: the same sums without staging. Thread
// (k, g) of a D_i-thread CTA loads rows k, k + 8, ... of the block, dims 8 g .. 8 g + 7, one
// 16-byte load per row (a warp reads two whole adjacent rows per load), and adds them in row
// order into the block's partial sums k of those dims; only the eight partial sums per dim
// pass through shared memory, to the same pairwise tree.
__global__ void __launch_bounds__(128, 8) k_block_means_rows(MeansParams p) {
    __shared__ float part[8][128];
    grid_dep_wait();
    const int bq = blockIdx.y;
    const int64_t k0 = p.key_off[bq];
    const int64_t Np = p.key_off[bq + 1] - k0;
    if (!seq_ok(p.key_off, bq, p.Np_max, p.keys_rows)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
        return;
    }
    const int64_t nb = Np / p.b;
    const int64_t m0 = p.means_off[bq];
    if (!means_ok(p.means_off, bq, nb, p.means_rows)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
        return;
    }
    int64_t fb = p.first_block ? (int64_t)p.first_block[bq] : 0;
    if (fb < 0) fb = 0;
    const int groups = p.D_i / 8, t = (int)threadIdx.x;
    const int k = t / groups, g = t - k * groups;           // residue class, dim group
    const int per = p.b / 8;                                  // rows of a class in a block
    const __nv_bfloat16 *keys = static_cast<const __nv_bfloat16 *>(p.keys);
    for (int64_t beta = fb + blockIdx.x; beta < nb; beta += gridDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(keys + (k0 + beta * p.b + k) * p.D_i + g * 8);
        const int64_t step = p.D_i;                           // uint4s from row i to row i + 8
        uint4 u[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < per) u[j] = __ldg(src + j * step);
        float ps[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) ps[e] = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < per) {
                const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(&u[j]);
#pragma unroll
                for (int e = 0; e < 8; ++e) ps[e] += __bfloat162float(x[e]);
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) part[k][g * 8 + e] = ps[e];
        __syncthreads();
        if (t < p.D_i) {
            const float s = ((part[0][t] + part[1][t]) + (part[2][t] + part[3][t])) +
                            ((part[4][t] + part[5][t]) + (part[6][t] + part[7][t]));
            p.means[(m0 + beta) * p.D_i + t] = s / (float)p.b;
        }
        __syncthreads();
    }
}

cudaError_t launch_block_means(const MeansParams &p, int64_t nb_max, cudaStream_t s) {
    if (nb_max <= 0) return cudaSuccess;
    // Blocks [first_block, nb) are walked grid-stride. An incremental update (first_block
    // given: few new blocks per sequence) sizes the grid from the batch, so that few CTAs
    // idle; a full build (no first_block) takes six CTAs per SM (as many as fit at once
    // with 32 KiB of staging each: one wave), each keeping a 64-row block in flight, which
    // the DRAM latency needs (two per SM ran at ~2.3 TB/s).
    const bool rows = p.keys_bf16 && p.D_i % 8 == 0 && p.D_i <= 128 && p.b % 8 == 0 && p.b <= 64;
    // the register form runs eight 128-thread CTAs per SM, each with a block in flight
    const int64_t target = p.first_block ? kTargetCtas : (rows ? 8 : 6) * (int64_t)kSmTarget;
    int64_t per_seq = (target + p.B - 1) / p.B;
    if (per_seq > nb_max) per_seq = nb_max;
    const unsigned gx = (unsigned)(per_seq < 1 ? 1 : per_seq);
    dim3 grid(gx, (unsigned)p.B);
    if (rows) return launch_pdl(k_block_means_rows, grid, dim3(p.D_i), 0, s, p.chained, p);
    if ((int64_t)p.b * p.D_i <= kMeansStage) {
        if (p.keys_bf16)
            return launch_pdl(k_block_means_staged<__nv_bfloat16>, grid, dim3(kMeansThreads), 0, s, p.chained,
                              p);
        return launch_pdl(k_block_means_staged<float>, grid, dim3(kMeansThreads), 0, s, p.chained, p);
    }
    const int threads = p.D_i;
    if (p.keys_bf16)
        k_block_means<__nv_bfloat16><<<grid, threads, 0, s>>>(p);
    else
        k_block_means<float><<<grid, threads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace hisa
