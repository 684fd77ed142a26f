// Sparse combine on CUDA cores ([HiSA issue] "Consuming the selection: sparse combine").
//
// For query row (b, j) the attended rows form one list: the local rows first, then the
// pooled rows named by I (or all Np_b rows for the dense branch). The list is split
// into `nsplit` ranges, one CTA each; a CTA walks its range in chunks of kChunk rows
// with an online softmax, all H query heads sharing every gathered row (one shared
// KV head, K = V). Invisible rows (sliding window, causal pooled re-mask, -1 padding)
// get zero weight. The sink joins the normaliser and carries no value; it is folded
// in by the last step: in-kernel when nsplit == 1, else by k_attend_combine over the
// split partials (m, l, acc).
#include "hisa_internal.cuh"

namespace hisa {

constexpr int kChunk = 32;
constexpr int kAttnThreads = 512;

__device__ __forceinline__ void unpack8(const uint4 &x, float (&v)[8], const __nv_bfloat16 *) {
    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&x);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float2 f = __bfloat1622float2(h2[e]);
        v[2 * e] = f.x;
        v[2 * e + 1] = f.y;
    }
}

// f32 rows are handled as two 16-byte halves of 4 values; see load8 below.
template <typename T>
__device__ __forceinline__ void load8(const T *src, float (&v)[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *src, float (&v)[8]) {
    uint4 x = *reinterpret_cast<const uint4 *>(src);
    unpack8(x, v, src);
}

template <>
__device__ __forceinline__ void load8<float>(const float *src, float (&v)[8]) {
    float4 a = reinterpret_cast<const float4 *>(src)[0];
    float4 b = reinterpret_cast<const float4 *>(src)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <int H, int DH, typename T>
struct AttnSmem {
    static constexpr int kPad = 16 / (int)sizeof(T);     // 16-byte row pad
    static constexpr int kStride = DH + kPad;             // elements per staged row
    static constexpr size_t kQ = (size_t)H * DH * sizeof(T);
    static constexpr size_t kKV = (size_t)kChunk * kStride * sizeof(T);
    static constexpr size_t kP = (size_t)H * kChunk * sizeof(float);
    static constexpr size_t bytes = kQ + kKV + kP + 3 * H * sizeof(float);
};

template <int H, int DH, typename T>
__global__ void __launch_bounds__(kAttnThreads) k_attend_simt(AttnParams p) {
    using S = AttnSmem<H, DH, T>;
    constexpr int DG = DH / 8;                                    // 8-wide dim groups
    constexpr int ITEMS = (H * DG + kAttnThreads - 1) / kAttnThreads;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T *sq = reinterpret_cast<T *>(smem_raw);
    T *skv = reinterpret_cast<T *>(smem_raw + S::kQ);
    float *sp = reinterpret_cast<float *>(smem_raw + S::kQ + S::kKV);
    float *sm = sp + H * kChunk;
    float *sl = sm + H;
    float *sa = sl + H;
    __shared__ const T *s_rowptr[kChunk];

    const int tid = threadIdx.x;
    const int row = blockIdx.x, split = blockIdx.y;
    const int bq = row / p.L, j = row - bq * p.L;
    const int64_t t = (int64_t)p.t0[bq] + j;
    const int64_t k0 = p.kv_off[bq];
    int64_t Np = p.kv_off[bq + 1] - k0;
    if (!seq_ok(p.kv_off, bq, p.Np_max, p.kv_rows)) {
        if (tid == 0 && split == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
        Np = 0;
    }
    int64_t nl = p.local_len[bq];
    nl = nl < 0 ? 0 : (nl > p.W_max ? p.W_max : nl);
    const int64_t pos0 = p.local_pos0[bq];
    // only the visible local window [lo, hi) enters the list
    int64_t lo = t - p.window + 1 - pos0, hi = t - pos0 + 1;
    lo = lo < 0 ? 0 : lo;
    hi = hi > nl ? nl : hi;
    const int64_t nloc = hi > lo ? hi - lo : 0;
    const int64_t npool = p.I ? (int64_t)p.k : Np;
    const int64_t ntot = nloc + npool;
    const int64_t e0 = (int64_t)split * p.rows_per_split;
    int64_t e1 = e0 + p.rows_per_split;
    if (e1 > ntot) e1 = ntot;
    const int64_t V = p.causal ? visible_len(t, p.r, Np) : Np;
    const T *local = reinterpret_cast<const T *>(p.local_kv) + ((int64_t)bq * p.W_max + lo) * DH;
    const T *pooled = reinterpret_cast<const T *>(p.pooled_kv) + k0 * DH;
    const int32_t *Irow = p.I ? p.I + (int64_t)row * p.k : nullptr;

    // stage q (H x DH) in its input type
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.q) +
                                                           (int64_t)row * H * DH);
        uint4 *dst = reinterpret_cast<uint4 *>(sq);
        for (int u = tid; u < (int)(S::kQ / 16); u += kAttnThreads) dst[u] = src[u];
    }
    for (int h = tid; h < H; h += kAttnThreads) { sm[h] = -INFINITY; sl[h] = 0.f; }
    float acc[ITEMS][8];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[it][e] = 0.f;
    __syncthreads();

    for (int64_t c0 = e0; c0 < e1; c0 += kChunk) {
        if (tid < kChunk) {
            const int64_t e = c0 + tid;
            const T *ptr = nullptr;
            if (e < e1) {
                if (e < nloc) {
                    ptr = local + e * DH;
                } else {
                    const int64_t kk = e - nloc;
                    const int64_t id = Irow ? (int64_t)Irow[kk] : kk;
                    if (id >= Np || id < -1) {
                        flag(p.status, HISA_DEV_BAD_ID);
                    } else if (id >= 0 && id < V) {
                        ptr = pooled + id * DH;
                    }
                }
            }
            s_rowptr[tid] = ptr;
        }
        __syncthreads();
        constexpr int UPR = DH * (int)sizeof(T) / 16;              // 16-byte units per row
        for (int u = tid; u < kChunk * UPR; u += kAttnThreads) {
            const int r = u / UPR, c = u - r * UPR;
            const T *ptr = s_rowptr[r];
            uint4 v = ptr ? reinterpret_cast<const uint4 *>(ptr)[c] : make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4 *>(skv + r * S::kStride)[c] = v;
        }
        __syncthreads();
        // scores s[h][r] = scale * q_h . kv_r
        for (int it = tid; it < H * kChunk; it += kAttnThreads) {
            const int r = it % kChunk, h = it / kChunk;
            float s = -INFINITY;
            if (s_rowptr[r]) {
                const T *qh = sq + h * DH;
                const T *kr = skv + r * S::kStride;
                float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
                for (int d = 0; d < DH; d += 8) {
                    float qv[8], kv[8];
                    load8<T>(qh + d, qv);
                    load8<T>(kr + d, kv);
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        a0 = fmaf(qv[e], kv[e], a0);
                        a1 = fmaf(qv[e + 1], kv[e + 1], a1);
                    }
                }
                s = (a0 + a1) * p.scale;
            }
            sp[h * kChunk + r] = s;
        }
        __syncthreads();
        // online softmax update per head
        for (int h = tid; h < H; h += kAttnThreads) {
            const float mold = sm[h];
            float mx = mold;
            for (int r = 0; r < kChunk; ++r) mx = fmaxf(mx, sp[h * kChunk + r]);
            const float alpha = (mx == -INFINITY) ? 1.f : expf(mold - mx);
            float sum = 0.f;
            for (int r = 0; r < kChunk; ++r) {
                const float v = sp[h * kChunk + r];
                const float pr = (v == -INFINITY) ? 0.f : expf(v - mx);
                sp[h * kChunk + r] = pr;
                sum += pr;
            }
            sm[h] = mx;
            sl[h] = sl[h] * alpha + sum;
            sa[h] = alpha;
        }
        __syncthreads();
        // acc[h][d] = alpha_h * acc + sum_r p[h][r] * kv_r[d]
#pragma unroll
        for (int it = 0; it < ITEMS; ++it) {
            const int item = tid + it * kAttnThreads;
            if (item < H * DG) {
                const int h = item / DG, dg = item - h * DG;
                const float alpha = sa[h];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[it][e] *= alpha;
                for (int r = 0; r < kChunk; ++r) {
                    const float pr = sp[h * kChunk + r];
                    float kv[8];
                    load8<T>(skv + r * S::kStride + dg * 8, kv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[it][e] = fmaf(pr, kv[e], acc[it][e]);
                }
            }
        }
        __syncthreads();
    }

#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int item = tid + it * kAttnThreads;
        if (item >= H * DG) continue;
        const int h = item / DG, dg = item - h * DG;
        if (p.nsplit == 1) {
            const float sink = p.sinks[h];
            const float mh = sm[h];
            const float M = fmaxf(mh, sink);
            const float wm = (mh == -INFINITY) ? 0.f : expf(mh - M);
            const float denom = sl[h] * wm + expf(sink - M);
            const float f = wm / denom;
            const int64_t at = ((int64_t)row * H + h) * DH + dg * 8;
            if (p.out_bf16) {
                uint4 v;
                uint32_t *w = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[it][2 * e] * f, acc[it][2 * e + 1] * f);
                    w[e] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + at) = v;
            } else {
                float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + at);
                dst[0] = make_float4(acc[it][0] * f, acc[it][1] * f, acc[it][2] * f, acc[it][3] * f);
                dst[1] = make_float4(acc[it][4] * f, acc[it][5] * f, acc[it][6] * f, acc[it][7] * f);
            }
        } else {
            float *base = p.part + (((int64_t)row * p.nsplit + split) * H + h) * (DH + 2);
            if (dg == 0) { base[0] = sm[h]; base[1] = sl[h]; }
#pragma unroll
            for (int e = 0; e < 8; ++e) base[2 + dg * 8 + e] = acc[it][e];
        }
    }
}

// Merge the split partials and fold in the sink: M = max(max_s m_s, sink),
// n = sum_s l_s e^{m_s - M} + e^{sink - M}, out = sum_s acc_s e^{m_s - M} / n.
template <int DH>
__global__ void k_attend_combine(AttnParams p) {
    grid_dep_wait();                                 // the partials are the previous grid's
    const int row = blockIdx.x, h = blockIdx.y;
    const int H = p.H;
    const float sink = p.sinks[h];
    const size_t stride = (size_t)H * (DH + 2);
    const float *base = p.part + ((int64_t)row * p.nsplit * H + h) * (DH + 2);
    float M = sink;
    for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, base[s * stride]);
    float denom = expf(sink - M);
    for (int s = 0; s < p.nsplit; ++s) {
        const float m = base[s * stride];
        if (m != -INFINITY) denom += base[s * stride + 1] * expf(m - M);
    }
    for (int d = threadIdx.x; d < DH; d += blockDim.x) {
        float o = 0.f;
        for (int s = 0; s < p.nsplit; ++s) {
            const float m = base[s * stride];
            if (m != -INFINITY) o += base[s * stride + 2 + d] * expf(m - M);
        }
        const int64_t at = ((int64_t)row * H + h) * DH + d;
        if (p.out_bf16)
            static_cast<__nv_bfloat16 *>(p.out)[at] = __float2bfloat16_rn(o / denom);
        else
            static_cast<float *>(p.out)[at] = o / denom;
    }
}

cudaError_t launch_attend_combine(const AttnParams &p, cudaStream_t s) {
    dim3 g2((unsigned)(p.B * p.L), (unsigned)p.H);
    switch (p.Dh) {
        // waits before its first global access, so it may always be launched as a
        // programmatic dependent of the kernel that writes the partials
        case 64: return launch_pdl(k_attend_combine<64>, g2, dim3(64), 0, s, 1, p);
        case 128: return launch_pdl(k_attend_combine<128>, g2, dim3(128), 0, s, 1, p);
        case 512: return launch_pdl(k_attend_combine<512>, g2, dim3(256), 0, s, 1, p);
        default: return cudaErrorInvalidValue;
    }
}

template <int H, int DH, typename T>
static cudaError_t launch_attend_t(const AttnParams &p, cudaStream_t s) {
    using S = AttnSmem<H, DH, T>;
    const cudaError_t attr = smem_attr_once<k_attend_simt<H, DH, T>>((int)S::bytes);
    if (attr != cudaSuccess) return attr;
    dim3 grid((unsigned)(p.B * p.L), (unsigned)p.nsplit);
    k_attend_simt<H, DH, T><<<grid, kAttnThreads, S::bytes, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.nsplit == 1) return e;
    return launch_attend_combine(p, s);
}

int attend_simt_supported(int H, int Dh) {
    return (H == 8 && Dh == 64) || (H == 16 && Dh == 128) || (H == 64 && Dh == 512);
}

// Split ranges are cut in multiples of 64 rows: one tensor-core tile, two CUDA-core chunks.
int attend_chunk_rows() { return 64; }

cudaError_t launch_attend_simt(const AttnParams &p, cudaStream_t s) {
    const bool bf = p.kv_bf16 != 0;
    if (p.H == 8 && p.Dh == 64)
        return bf ? launch_attend_t<8, 64, __nv_bfloat16>(p, s) : launch_attend_t<8, 64, float>(p, s);
    if (p.H == 16 && p.Dh == 128)
        return bf ? launch_attend_t<16, 128, __nv_bfloat16>(p, s)
                  : launch_attend_t<16, 128, float>(p, s);
    if (p.H == 64 && p.Dh == 512)
        return bf ? launch_attend_t<64, 512, __nv_bfloat16>(p, s)
                  : launch_attend_t<64, 512, float>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace hisa
