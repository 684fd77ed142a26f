// Block-wide top-k of one row of f32 scores, as a set, by radix select over orderable
// 32-bit keys ([HiSA issue] "Conventions": argpartition returns an unordered top-k set).
//
// Four 8-bit passes (most significant digit first) find the k-th largest key T and how
// many elements equal to T are still needed; a final pass emits, in ascending column
// order, every element above T plus the lowest-indexed elements equal to T. Equal
// scores therefore fall to the lower column; -0.0 equals +0.0. All NT threads of the
// CTA take part; `sc` may point to global or shared memory.
#pragma once

#include "hisa_internal.cuh"

namespace hisa {

template <int NT>
struct SelectShared {
    uint32_t hist[256];
    uint32_t wg[NT / 32], we[NT / 32];
    uint32_t prefix, kk, tg, te;
    int nonfinite;
};

// Writes the kout selected columns, mapped through map(i), to out[0..kout) in ascending
// column order. Caller guarantees 0 <= kout <= n. Contains __syncthreads(): every thread
// of the CTA must call it with the same arguments.
template <int NT, typename Map>
__device__ void block_topk(const float *sc, int64_t n, int64_t kout, int32_t *out, Map map,
                           SelectShared<NT> &sh, uint32_t *status) {
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (kout <= 0) return;
    if (tid == 0) sh.nonfinite = 0;
    uint32_t prefix = 0u, mask = 0u, kk = (uint32_t)kout;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int e = tid; e < 256; e += NT) sh.hist[e] = 0u;
        __syncthreads();
        for (int64_t i = tid; i < n; i += NT) {
            const float v = sc[i];
            if (shift == 24 && !isfinite(v)) sh.nonfinite = 1;
            const uint32_t key = order_key(v);
            if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns bins 255-8l .. 248-8l (descending); scan counts over lanes
            uint32_t c[8], tot = 0u;
#pragma unroll
            for (int t = 0; t < 8; ++t) { c[t] = sh.hist[255 - 8 * lane - t]; tot += c[t]; }
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
                        sh.prefix = prefix | ((255u - 8u * lane - t) << shift);
                        sh.kk = kk - cum;
                        break;
                    }
                    cum += c[t];
                }
            }
        }
        __syncthreads();
        prefix = sh.prefix;
        kk = sh.kk;
        mask |= 255u << shift;
        __syncthreads();
    }
    if (tid == 0 && sh.nonfinite) flag(status, HISA_DEV_NONFINITE);

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
        if (lane == 0) { sh.wg[warp] = __popc(bg); sh.we[warp] = __popc(be); }
        __syncthreads();
        if (warp == 0) {
            const uint32_t vg = lane < NW ? sh.wg[lane] : 0u;
            const uint32_t ve = lane < NW ? sh.we[lane] : 0u;
            uint32_t ig = vg, ie = ve;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t a = __shfl_up_sync(0xffffffffu, ig, o);
                const uint32_t b = __shfl_up_sync(0xffffffffu, ie, o);
                if (lane >= o) { ig += a; ie += b; }
            }
            if (lane < NW) { sh.wg[lane] = ig - vg; sh.we[lane] = ie - ve; }
            if (lane == 31) { sh.tg = ig; sh.te = ie; }
        }
        __syncthreads();
        const uint32_t pg = base_g + sh.wg[warp] + __popc(bg & lt);
        const uint32_t pe = base_e + sh.we[warp] + __popc(be & lt);
        if (g || (e && pe < kk)) out[pg + (pe < kk ? pe : kk)] = map(i);
        base_g += sh.tg;
        base_e += sh.te;
        __syncthreads();
    }
}

}  // namespace hisa
