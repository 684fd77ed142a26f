// The indexer's compressor ([HiSA issue] "The pooled stream and positions",
// "Configuration": compressor.{wkv, wgate, ape, norm}): each new pooled row is the gated
// pooling of its r-token window (and, in the overlap variant, of the window before it),
// RMS-normalised and rotated on its trailing rope_dims dims at position p r, then written
// to the pooled key cache; the means of the index_block-row blocks that the new rows
// complete are appended to the block-mean cache in the same call.
//
// One CTA per (sequence, block of index_block pooled rows that the new rows touch), D x L
// threads (L = 1, 4 or 8 row lanes: 8 for a few long appends, fewer when many CTAs share
// the SMs): thread (d, k) owns output dim d of the block's rows i = k, k + L, ... (i counted
// from the block's first row), which it takes in row order. A pooled row costs 2 r token
// rows of kv and gate (coalesced: thread d reads column d of each) and one reduction over
// the row's D threads for the RMS (a named barrier per row lane, so the eight lanes do not
// wait on one another); the pair partner of a rotated dim is the neighbouring lane. Each
// thread sums the values of its rows as stored (new rows as written, older rows of the block
// read back) into the partial sums of hisa_block_means it owns (sum j over rows = j mod 8,
// in row order: j = k, k + L, ...); the block mean then combines the eight partial sums in
// that function's fixed pairwise tree, so both write the same bits.
#include <math.h>

#include "hisa_internal.cuh"

namespace hisa {

namespace {

constexpr int kRowsPerUnitFlat = 64;     // rows per CTA when no block means are kept (b == 0)
constexpr int kSums = 8;                 // partial sums of a block mean (rows = j mod 8)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void lane_sync(int lane, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(lane + 1), "r"(threads) : "memory");
}

template <int L>
__global__ void __launch_bounds__(128 * L, 8 / L) k_compress(CompressParams p) {
    constexpr int J = kSums / L;                     // partial sums per thread
    __shared__ float red[L][4];
    __shared__ float part[kSums][128];
    grid_dep_wait();
    const int sq = blockIdx.y;
    const int d = threadIdx.x;                       // output dim; blockDim.x == D
    const int lk = threadIdx.y;                      // row lane
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
        if (d == 0 && lk == 0 && blockIdx.x == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
        return;
    }
    // the rows of this unit; `origin` is the row that lane 0 starts from
    int64_t r_lo, r_hi, beta = -1, origin;
    if (p.b > 0) {
        beta = p0 / p.b + blockIdx.x;
        r_lo = beta * p.b > p0 ? beta * p.b : p0;
        r_hi = (beta + 1) * p.b < np_after ? (beta + 1) * p.b : np_after;
        origin = beta * p.b;
    } else {
        r_lo = p0 + (int64_t)blockIdx.x * kRowsPerUnitFlat;
        r_hi = r_lo + kRowsPerUnitFlat < np_after ? r_lo + kRowsPerUnitFlat : np_after;
        origin = r_lo;
    }
    if (r_lo >= r_hi) return;
    // a block the new rows complete gets its mean: its older rows are read back as stored
    const bool mean = p.b > 0 && p.means && (beta + 1) * p.b <= np_after;

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
    // this lane's rows are origin + lk + t L, t = 0, 1, ...; row t adds to partial sum t mod J
    float ps[J];                                     // partial sums lk, lk + L, ... of the block mean
#pragma unroll
    for (int j = 0; j < J; ++j) ps[j] = 0.f;
    if (mean) {
        // the block's older rows, as stored, eight loads in flight per round
        for (int64_t g = origin + lk; g < r_lo; g += kSums * L) {
            float v[kSums];
#pragma unroll
            for (int u = 0; u < kSums; ++u) {
                const int64_t at = (k0 + g + u * L) * D + d;
                v[u] = g + u * L >= r_lo ? 0.f
                       : p.k_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.keys)[at])
                                  : reinterpret_cast<const float *>(p.keys)[at];
            }
#pragma unroll
            for (int u = 0; u < kSums; ++u)
                if (g + u * L < r_lo) ps[u % J] += v[u];
        }
    }
    // the new rows, from the first group of J of this lane's rows that reaches r_lo
    int64_t g0 = origin + lk;
    if (r_lo > g0) g0 += (r_lo - g0) / kSums * kSums;
    for (int64_t g = g0; g < r_hi; g += kSums) {
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int64_t row = g + j * L;               // block row lk + j L (mod 8)
        if (row >= r_hi) break;
        if (row < r_lo) continue;                    // read above
        const int64_t dst = (k0 + row) * D + d;
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
        // RMSNorm over the D dims of this row (its lane's D threads)
        float ss = warp_sum(y * y);
        if ((d & 31) == 0) red[lk][d >> 5] = ss;
        lane_sync(lk, D);
        ss = 0.f;
        for (int w = 0; w < (D >> 5); ++w) ss += red[lk][w];
        lane_sync(lk, D);
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
        if (p.k_bf16) {
            const __nv_bfloat16 h = __float2bfloat16_rn(y);
            reinterpret_cast<__nv_bfloat16 *>(p.keys)[dst] = h;
            ps[j] += __bfloat162float(h);
        } else {
            reinterpret_cast<float *>(p.keys)[dst] = y;
            ps[j] += y;
        }
      }
    }
    if (!mean) return;
#pragma unroll
    for (int j = 0; j < J; ++j) part[lk + j * L][d] = ps[j];
    __syncthreads();
    if (lk == 0) {
        const float(*q)[128] = part;
        const float s = ((q[0][d] + q[1][d]) + (q[2][d] + q[3][d])) + ((q[4][d] + q[5][d]) + (q[6][d] + q[7][d]));
        p.means[(p.means_off[sq] + beta) * D + d] = s / (float)p.b;
    }
}

}  // namespace

cudaError_t launch_compress(const CompressParams &p, cudaStream_t s) {
    if (p.B == 0 || p.n_new_max == 0) return cudaSuccess;
    // blocks that n_new_max rows can touch: (n + b - 2) / b + 1 (rows p0 .. p0 + n - 1 from
    // the last row of a block)
    const int64_t per = p.b > 0 ? ((int64_t)p.n_new_max + p.b - 2) / p.b + 1
                                : ((int64_t)p.n_new_max + kRowsPerUnitFlat - 1) / kRowsPerUnitFlat;
    if (p.D % 32 || p.D > 128) return cudaErrorInvalidValue;
    dim3 grid((unsigned)per, (unsigned)p.B);
    // row lanes: up to one CTA per SM (a prefill append) spreads its rows over 8 lanes; up to
    // two per SM (a decode append of one row per sequence, mostly older rows read back for
    // the mean) over 4; more CTAs than that take one lane
    const int64_t ctas = per * (int64_t)p.B;
    const int sms = device_sm_count();
    if (sms > 0 && ctas <= sms)
        return launch_pdl(k_compress<8>, grid, dim3(p.D, 8), 0, s, p.chained, p);
    if (sms > 0 && ctas <= 2 * (int64_t)sms)
        return launch_pdl(k_compress<4>, grid, dim3(p.D, 4), 0, s, p.chained, p);
    return launch_pdl(k_compress<1>, grid, dim3(p.D, 1), 0, s, p.chained, p);
}

}  // namespace hisa
