// Per-query top-k as a set, by radix select over 32-bit orderable score keys
// ([HiSA issue] "Conventions": argpartition returns an unordered top-k set; the flat,
// coarse and fine stages all take one).
//
// One CTA owns one query row. Four 8-bit passes (most significant digit first) find
// the k-th largest key T and how many of the elements equal to T are still needed;
// a final pass emits, in ascending column order, every element above T plus the
// lowest-indexed elements equal to T. No global sort, no inter-CTA traffic.
#include "hisa_internal.cuh"

namespace hisa {

template <int NT>
__global__ void __launch_bounds__(NT) k_select(SelectParams p) {
    constexpr int NW = NT / 32;
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_prefix, s_kk;
    __shared__ uint32_t s_wg[NW], s_we[NW];
    __shared__ uint32_t s_tg, s_te;
    __shared__ int s_blk[64];
    __shared__ int s_bad, s_nonfinite;

    const int row = blockIdx.x;
    const int bq = row / p.L;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t *out = p.out + (int64_t)row * p.k;

    const int64_t k0 = p.key_off[bq];
    const int64_t Np = p.key_off[bq + 1] - k0;
    bool ok = Np >= 0 && Np <= p.Np_max;
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
            for (int s = 0; s < p.keep; ++s) {
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
    if (tid == 0) s_nonfinite = 0;

    uint32_t prefix = 0u, mask = 0u, kk = (uint32_t)kout;
    if (kout > 0) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int e = tid; e < 256; e += NT) hist[e] = 0u;
            __syncthreads();
            for (int64_t i = tid; i < n; i += NT) {
                const float v = sc[i];
                if (shift == 24 && !isfinite(v)) s_nonfinite = 1;
                const uint32_t key = order_key(v);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                // lane l owns bins 255-8l .. 248-8l (descending); scan counts over lanes
                uint32_t c[8], tot = 0u;
#pragma unroll
                for (int t = 0; t < 8; ++t) { c[t] = hist[255 - 8 * lane - t]; tot += c[t]; }
                uint32_t incl = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                const uint32_t excl = incl - tot;
                if (excl < kk && kk <= incl) {
                    uint32_t cum = excl;
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        if (cum + c[t] >= kk) {
                            const uint32_t digit = 255u - 8u * lane - t;
                            s_prefix = prefix | (digit << shift);
                            s_kk = kk - cum;
                            break;
                        }
                        cum += c[t];
                    }
                }
            }
            __syncthreads();
            prefix = s_prefix;
            kk = s_kk;
            mask |= 255u << shift;
            __syncthreads();
        }
        if (tid == 0 && s_nonfinite) flag(p.status, HISA_DEV_NONFINITE);

        // emit: elements > T, plus the first kk (by column) equal to T, in column order
        const uint32_t T = prefix;
        const uint32_t lt = (1u << lane) - 1u;
        uint32_t base_g = 0u, base_e = 0u;
        for (int64_t start = 0; start < n; start += NT) {
            const int64_t i = start + tid;
            uint32_t key = 0u;
            const bool valid = i < n;
            if (valid) key = order_key(sc[i]);
            const bool g = valid && key > T;
            const bool e = valid && key == T;
            const uint32_t bg = __ballot_sync(0xffffffffu, g);
            const uint32_t be = __ballot_sync(0xffffffffu, e);
            if (lane == 0) { s_wg[warp] = __popc(bg); s_we[warp] = __popc(be); }
            __syncthreads();
            if (warp == 0) {
                const uint32_t vg = lane < NW ? s_wg[lane] : 0u;
                const uint32_t ve = lane < NW ? s_we[lane] : 0u;
                uint32_t ig = vg, ie = ve;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t a = __shfl_up_sync(0xffffffffu, ig, o);
                    const uint32_t b = __shfl_up_sync(0xffffffffu, ie, o);
                    if (lane >= o) { ig += a; ie += b; }
                }
                if (lane < NW) { s_wg[lane] = ig - vg; s_we[lane] = ie - ve; }
                if (lane == 31) { s_tg = ig; s_te = ie; }
            }
            __syncthreads();
            const uint32_t pg = base_g + s_wg[warp] + __popc(bg & lt);
            const uint32_t pe = base_e + s_we[warp] + __popc(be & lt);
            if (g || (e && pe < kk)) {
                int32_t id;
                if (p.mode == kFine)
                    id = (int32_t)((int64_t)s_blk[i / p.b] * p.b + (i % p.b));
                else
                    id = (int32_t)i;
                out[pg + (pe < kk ? pe : kk)] = id;
            }
            base_g += s_tg;
            base_e += s_te;
            __syncthreads();
        }
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
