// The indexer's compressor ([HiSA issue] "The pooled stream and positions",
// "Configuration": compressor.{wkv, wgate, ape, norm}): each new pooled row is the gated
// pooling of its r-token window (and, in the overlap variant, of the window before it),
// RMS-normalised and rotated on its trailing rope_dims dims at position p r, then written
// to the pooled key cache; the means of the index_block-row blocks that the new rows
// complete are appended to the block-mean cache in the same call.
//
// One CTA per (sequence, block of index_block pooled rows that the new rows touch), one
// thread per output dim. A pooled row costs 2 r token rows of kv and gate (coalesced:
// thread d reads column d of each) and one block reduction for the RMS; the pair partner
// of a rotated dim is the neighbouring lane. The block mean reads the block's b stored
// rows back (the CTA's own rows are visible after __syncthreads) and sums each dim in
// the order of hisa_block_means (eight partial sums over rows = k mod 8, in row order,
// then a fixed pairwise tree), so both write the same bits.
#include <math.h>

#include "hisa_internal.cuh"

namespace hisa {

namespace {

constexpr int kRowsPerUnitFlat = 64;     // rows per CTA when no block means are kept (b == 0)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void k_compress(CompressParams p) {
    __shared__ float red[4];
    grid_dep_wait();
    const int sq = blockIdx.y;
    const int d = threadIdx.x;                       // output dim; blockDim.x == D
    const int D = p.D;
    const int64_t p0 = p.p_first[sq];
    const int64_t nn = p.n_new[sq];
    if (nn <= 0) return;
    // sequence sq's token rows, key rows and (when kept) block-mean rows must fit
    const int64_t t0 = p.tok_off[sq], t1 = p.tok_off[sq + 1];
    const int64_t k0 = p.key_off[sq], k1 = p.key_off[sq + 1];
    bool ok = p0 >= 0 && nn <= p.n_new_max && t0 >= 0 && t1 - t0 == (nn + 1) * p.r &&
              t1 <= p.tok_rows && k0 >= 0 && k0 + p0 + nn <= k1 && k1 <= p.keys_rows;
    const int64_t np_after = p0 + nn;
    if (ok && p.b > 0 && p.means) {
        const int64_t nb = np_after / p.b;
        ok = means_ok(p.means_off, sq, nb, p.means_rows);
    }
    if (!ok) {
        if (d == 0 && blockIdx.x == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
        return;
    }
    // the rows of this unit
    int64_t r_lo, r_hi, beta = -1;
    if (p.b > 0) {
        beta = p0 / p.b + blockIdx.x;
        r_lo = beta * p.b > p0 ? beta * p.b : p0;
        r_hi = (beta + 1) * p.b < np_after ? (beta + 1) * p.b : np_after;
    } else {
        r_lo = p0 + (int64_t)blockIdx.x * kRowsPerUnitFlat;
        r_hi = r_lo + kRowsPerUnitFlat < np_after ? r_lo + kRowsPerUnitFlat : np_after;
    }
    if (r_lo >= r_hi) return;

    const int C = p.C;
    const int cur = p.overlap ? D : 0;               // channel offset of the current window
    const float nw = p.norm_w[d];
    // rotation of this dim's pair: trailing rope_dims dims, pairs (2m, 2m + 1)
    const int first_rot = D - p.rope_dims;
    const bool rot = d >= first_rot;
    double freq = 0.0;
    if (rot) {
        const int i = (d - first_rot) >> 1;          // rotated pair index
        freq = exp(-2.0 * (double)i / (double)p.rope_dims * p.log_theta);
    }
    const float *ape = p.ape;
    for (int64_t row = r_lo; row < r_hi; ++row) {
        const int64_t tw = t0 + (row - p0 + 1) * p.r;       // first token of its window
        // online softmax over the entries of this dim
        float m = -INFINITY, l = 0.f, acc = 0.f;
        auto take = [&](float z, float v) {
            if (z > m) {
                const float a = expf(m - z);                // m = -inf: 0
                l *= a;
                acc *= a;
                m = z;
            }
            const float e = expf(z - m);
            l += e;
            acc += e * v;
        };
        if (p.overlap && row > 0) {
            for (int i = 0; i < p.r; ++i) {
                const int64_t t = tw - p.r + i;
                take(p.gate[t * C + d] + ape[i * C + d], p.kv[t * C + d]);
            }
        }
        for (int i = 0; i < p.r; ++i) {
            const int64_t t = tw + i;
            take(p.gate[t * C + cur + d] + ape[i * C + cur + d], p.kv[t * C + cur + d]);
        }
        float y = acc / l;
        // RMSNorm over the D dims
        float ss = warp_sum(y * y);
        if ((d & 31) == 0) red[d >> 5] = ss;
        __syncthreads();
        ss = 0.f;
        for (int w = 0; w < (D >> 5); ++w) ss += red[w];
        __syncthreads();
        y = y / sqrtf(ss / (float)D + p.eps) * nw;
        // RoPE at position row * r; the angle is reduced modulo 2 pi in double
        const float partner = __shfl_xor_sync(0xffffffffu, y, 1);
        if (rot) {
            double ang = (double)(row * p.r) * freq;
            ang -= 6.283185307179586 * floor(ang / 6.283185307179586);
            float sn, cs;
            sincosf((float)ang, &sn, &cs);
            y = (d & 1) ? partner * sn + y * cs : y * cs - partner * sn;
        }
        const int64_t dst = (k0 + row) * D + d;
        if (p.k_bf16)
            reinterpret_cast<__nv_bfloat16 *>(p.keys)[dst] = __float2bfloat16_rn(y);
        else
            reinterpret_cast<float *>(p.keys)[dst] = y;
    }
    // the mean of a block the new rows complete
    if (p.b > 0 && p.means && (beta + 1) * p.b <= np_after) {
        __syncthreads();                             // this CTA's rows are visible to it
        const int64_t base = (k0 + beta * p.b) * D + d;
        float ps[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float a = 0.f;
            for (int i = k; i < p.b; i += 8) {
                const int64_t at = base + (int64_t)i * D;
                a += p.k_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.keys)[at])
                              : reinterpret_cast<const float *>(p.keys)[at];
            }
            ps[k] = a;
        }
        const float s = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        p.means[(p.means_off[sq] + beta) * D + d] = s / (float)p.b;
    }
}

}  // namespace

cudaError_t launch_compress(const CompressParams &p, cudaStream_t s) {
    if (p.B == 0 || p.n_new_max == 0) return cudaSuccess;
    const int64_t per = p.b > 0 ? (int64_t)p.n_new_max / p.b + 2
                                : ((int64_t)p.n_new_max + kRowsPerUnitFlat - 1) / kRowsPerUnitFlat;
    dim3 grid((unsigned)per, (unsigned)p.B);
    return launch_pdl(k_compress, grid, dim3(p.D), 0, s, p.chained, p);
}

}  // namespace hisa
