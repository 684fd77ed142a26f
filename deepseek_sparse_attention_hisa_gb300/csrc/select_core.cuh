// Block-wide top-k of one row of f32 scores, as a set, by radix select over orderable
// 32-bit keys ([HiSA issue] "Conventions": argpartition returns an unordered top-k set).
//
// Scores of one row cluster in value, so their float bits share most high bits and a
// digit of the raw bits would put nearly every score in one bin. Instead, pass 1 bins
// the unmasked scores linearly in value over their [min, max] (256 bins; the binning is
// non-decreasing, so a higher bin holds strictly larger scores and equal scores share a
// bin; one shared atomic per distinct bin per warp), finds the bin of the k-th largest
// score, compacts that bin's elements and resolves them exactly by one warp: up to 32 by
// direct ranking, more by a radix select over their keys. When the k-th score is masked
// or the range degenerates, a block-wide four-pass radix select over the keys is used.
// The final pass emits, in ascending column order, every element above the k-th key T
// plus the lowest-indexed elements equal to T: each warp owns a contiguous segment of
// columns, so one block-wide prefix over warps fixes every output position. Equal
// scores therefore fall to the lower column; -0.0 equals +0.0. `sc` may point to global
// or shared memory.
#pragma once

#include "hisa_internal.cuh"

namespace hisa {

constexpr int kCand = 1024;

// Barrier of the selecting threads: the whole CTA (BAR == 0) or the NT threads of named
// barrier BAR (a group of whole warps that selects while the other warps keep working).
template <int NT, int BAR>
__device__ __forceinline__ void group_sync() {
    if (BAR == 0)
        __syncthreads();
    else
        asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT) : "memory");
}

template <int NT>
struct alignas(16) SelectShared {
    uint32_t hist[256];
    uint32_t wg[NT / 32], we[NT / 32];
    uint32_t prefix, kk, ncand;
    int nonfinite;
    alignas(16) int32_t cand[kCand];
};

// One warp: find the digit (at `shift`) of the kk-th largest key among the keys counted
// in hist; writes the extended prefix and the remaining rank to *prefix_out / *kk_out.
__device__ __forceinline__ void warp_find_digit(const uint32_t *hist, uint32_t prefix,
                                                uint32_t kk, int shift, uint32_t *prefix_out,
                                                uint32_t *kk_out) {
    const int lane = threadIdx.x & 31;
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
                *prefix_out = prefix | ((255u - 8u * lane - t) << shift);
                *kk_out = kk - cum;
                break;
            }
            cum += c[t];
        }
    }
}

// hist[digit] += 1 for every lane of the warp with valid == true, one atomic per distinct
// digit per warp (scores cluster, so many lanes share a bin).
__device__ __forceinline__ void warp_hist_add(uint32_t *hist, bool valid, uint32_t digit) {
    const uint32_t active = __ballot_sync(0xffffffffu, valid);
    if (valid) {
        const uint32_t peers = __match_any_sync(active, digit);
        if ((threadIdx.x & 31) == (uint32_t)(__ffs(peers) - 1)) atomicAdd(&hist[digit], __popc(peers));
    }
}

__device__ __forceinline__ float key_to_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Scores at or below this are selection masks (NEG = -1e30), kept out of the value range.
constexpr float kMaskedBelow = -1e29f;

// Block-wide radix select over the full keys: four 8-bit passes; resolves any input.
// Leaves the k-th key in sh.prefix and the count of its equals to take in sh.kk.
// The selecting threads are threadIdx.x in [TID0, TID0 + NT) (TID0 a multiple of 32).
// The general paths below are rare (non-finite or heavily tied scores, long rows): they
// are kept out of line so that the selecting kernels' hot code stays small.
template <int NT, int BAR = 0, int TID0 = 0>
__device__ __noinline__ void block_radix_threshold(const float *sc, int64_t n, uint32_t kout,
                                      SelectShared<NT> &sh) {
    const int tid = (int)threadIdx.x - TID0, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0u, mask = 0u, kk = kout;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int e = tid; e < 256; e += NT) sh.hist[e] = 0u;
        group_sync<NT, BAR>();
        for (int64_t base = (int64_t)warp * 32; base < n; base += NT) {
            const int64_t i = base + lane;
            const uint32_t key = i < n ? order_key(sc[i]) : 0u;
            warp_hist_add(sh.hist, i < n && (key & mask) == prefix, (key >> shift) & 255u);
        }
        group_sync<NT, BAR>();
        if (warp == 0) warp_find_digit(sh.hist, prefix, kk, shift, &sh.prefix, &sh.kk);
        group_sync<NT, BAR>();
        prefix = sh.prefix;
        kk = sh.kk;
        mask |= 255u << shift;
        group_sync<NT, BAR>();
    }
}

// Writes the kout selected columns, mapped through map(i), to out[0..kout) in ascending
// column order. Caller guarantees 0 <= kout <= n. Contains barriers (group_sync<NT, BAR>):
// every selecting thread (threadIdx.x in [TID0, TID0 + NT)) must call it with the same
// arguments.
template <int NT, int BAR = 0, int TID0 = 0, typename Map>
__device__ __noinline__ void block_topk(const float *sc, int64_t n, int64_t kout, int32_t *out, Map map,
                           SelectShared<NT> &sh, uint32_t *status) {
    constexpr int NW = NT / 32;
    const int tid = (int)threadIdx.x - TID0, lane = tid & 31, warp = tid >> 5;
    if (kout <= 0) return;

    // ---- range of the unmasked finite scores (as keys: integer min / max) ----
    uint32_t kmin = 0xffffffffu, kmax = 0u, nfree = 0u;
    int nonfinite = 0;
    for (int64_t i = tid; i < n; i += NT) {
        const float v = sc[i];
        const bool fin = isfinite(v);
        nonfinite |= !fin;
        if (fin && v > kMaskedBelow) {
            const uint32_t key = order_key(v);
            kmin = key < kmin ? key : kmin;
            kmax = key > kmax ? key : kmax;
            ++nfree;
        }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    nfree = __reduce_add_sync(0xffffffffu, nfree);
    nonfinite = __reduce_or_sync(0xffffffffu, nonfinite);
    if (lane == 0) { sh.wg[warp] = kmin; sh.we[warp] = kmax; sh.cand[warp] = (int32_t)nfree; }
    if (tid == 0) { sh.nonfinite = 0; sh.ncand = 0u; }
    for (int e = tid; e < 256; e += NT) sh.hist[e] = 0u;
    group_sync<NT, BAR>();
    if (lane == 0 && nonfinite) sh.nonfinite = 1;
    kmin = 0xffffffffu;
    kmax = 0u;
    nfree = 0u;
    for (int w = 0; w < NW; ++w) {
        kmin = sh.wg[w] < kmin ? sh.wg[w] : kmin;
        kmax = sh.we[w] > kmax ? sh.we[w] : kmax;
        nfree += (uint32_t)sh.cand[w];
    }
    group_sync<NT, BAR>();
    const float smin = key_to_float(kmin), smax = key_to_float(kmax);
    const float scale = 255.0f / (smax - smin);
    if (nfree < (uint64_t)kout || !(smax > smin) || !isfinite(scale)) {
        // the k-th score is masked, or the unmasked scores are (nearly) all equal
        block_radix_threshold<NT, BAR, TID0>(sc, n, (uint32_t)kout, sh);
    } else {
        // value bins: bin(s) is non-decreasing in s, so a higher bin holds strictly
        // larger scores and equal scores share a bin
        auto bin_of = [&](float v) -> uint32_t {
            if (!(v >= smin)) return 0u;
            if (!(v < smax)) return 255u;
            const int b = (int)((v - smin) * scale);
            return (uint32_t)(b < 0 ? 0 : (b > 254 ? 254 : b));
        };
        for (int64_t base = (int64_t)warp * 32; base < n; base += NT) {
            const int64_t i = base + lane;
            const float v = i < n ? sc[i] : 0.f;
            warp_hist_add(sh.hist, i < n, bin_of(v));
        }
        group_sync<NT, BAR>();
        // the bin of the k-th largest score; sh.kk = its rank inside that bin
        if (warp == 0) warp_find_digit(sh.hist, 0u, (uint32_t)kout, 0, &sh.prefix, &sh.kk);
        group_sync<NT, BAR>();
        const uint32_t dbin = sh.prefix;
        uint32_t kk = sh.kk;
        for (int64_t base = (int64_t)warp * 32; base < n; base += NT) {
            const int64_t i = base + lane;
            const bool c = i < n && bin_of(sc[i]) == dbin;
            const uint32_t bal = __ballot_sync(0xffffffffu, c);
            uint32_t at = 0u;
            if (lane == 0 && bal) at = atomicAdd(&sh.ncand, (uint32_t)__popc(bal));
            at = __shfl_sync(0xffffffffu, at, 0) + __popc(bal & ((1u << lane) - 1u));
            if (c && at < (uint32_t)kCand) sh.cand[at] = (int32_t)i;
        }
        group_sync<NT, BAR>();
        const uint32_t m = sh.ncand;
        if (m <= 32u) {
            if (warp == 0) {                   // few candidates: rank them directly
                const bool have = (uint32_t)lane < m;
                const int32_t idx = have ? sh.cand[lane] : 0x7fffffff;
                const uint32_t key = have ? order_key(sc[idx]) : 0u;
                uint32_t rank = 0u;            // candidates ahead in (key desc, column asc)
                for (int j = 0; j < 32; ++j) {
                    const uint32_t kj = __shfl_sync(0xffffffffu, key, j);
                    const int32_t ij = __shfl_sync(0xffffffffu, idx, j);
                    rank += ((uint32_t)j < m && (kj > key || (kj == key && ij < idx))) ? 1u : 0u;
                }
                if (have && rank == kk - 1u) sh.prefix = key;   // the last one selected
                __syncwarp();
                const uint32_t t = sh.prefix;
                const uint32_t above = __popc(__ballot_sync(0xffffffffu, have && key > t));
                if (lane == 0) sh.kk = kk - above;
            }
        } else if (m <= (uint32_t)kCand) {
            if (warp == 0) {                   // radix over the candidates' keys, one warp
                uint32_t prefix = 0u, mask = 0u;
                for (int sft = 24; sft >= 0; sft -= 8) {
                    for (int e = lane; e < 256; e += 32) sh.hist[e] = 0u;
                    __syncwarp();
                    for (uint32_t c = lane; c < m; c += 32) {
                        const uint32_t key = order_key(sc[sh.cand[c]]);
                        if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> sft) & 255u], 1u);
                    }
                    __syncwarp();
                    warp_find_digit(sh.hist, prefix, kk, sft, &sh.prefix, &sh.kk);
                    __syncwarp();
                    prefix = sh.prefix;
                    kk = sh.kk;
                    mask |= 255u << sft;
                    __syncwarp();
                }
            }
        } else {
            block_radix_threshold<NT, BAR, TID0>(sc, n, (uint32_t)kout, sh);
        }
    }
    group_sync<NT, BAR>();
    if (tid == 0 && sh.nonfinite) flag(status, HISA_DEV_NONFINITE);
    const uint32_t T = sh.prefix;
    const uint32_t kk = sh.kk;

    // ---- emit: warp w owns columns [lo, hi) ----
    const uint32_t lt = (1u << lane) - 1u;
    const int64_t seg = (n + NW - 1) / NW;
    const int64_t lo = warp * seg, hi = lo + seg < n ? lo + seg : n;
    uint32_t cg = 0u, ce = 0u;
    for (int64_t start = lo; start < hi; start += 32) {
        const int64_t i = start + lane;
        const uint32_t key = i < hi ? order_key(sc[i]) : 0u;
        cg += __popc(__ballot_sync(0xffffffffu, i < hi && key > T));
        ce += __popc(__ballot_sync(0xffffffffu, i < hi && key == T));
    }
    if (lane == 0) { sh.wg[warp] = cg; sh.we[warp] = ce; }
    group_sync<NT, BAR>();
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
    }
    group_sync<NT, BAR>();
    uint32_t base_g = sh.wg[warp], base_e = sh.we[warp];
    for (int64_t start = lo; start < hi; start += 32) {
        const int64_t i = start + lane;
        const uint32_t key = i < hi ? order_key(sc[i]) : 0u;
        const bool g = i < hi && key > T;
        const bool e = i < hi && key == T;
        const uint32_t bg = __ballot_sync(0xffffffffu, g);
        const uint32_t be = __ballot_sync(0xffffffffu, e);
        const uint32_t pg = base_g + __popc(bg & lt);
        const uint32_t pe = base_e + __popc(be & lt);
        const uint32_t at = pg + (pe < kk ? pe : kk);
        // at < kout for finite scores; the guard keeps non-finite input (flagged) in bounds
        if ((g || (e && pe < kk)) && at < (uint64_t)kout) out[at] = map(i);
        base_g += __popc(bg);
        base_e += __popc(be);
    }
    group_sync<NT, BAR>();
}

}  // namespace hisa

namespace hisa {

// Capacity of the threshold bin that small_topk resolves itself.
constexpr int kSmallCand = 128;

// Top kout of n <= E * NT scores in shared memory, short form. Thread t holds the E
// contiguous columns [t E, t E + E) in registers for the whole call. The selecting warps
// share the SM's shared-memory and shuffle pipes, so every step keeps those instructions
// few (one warp scans the histogram; no warp repeats another's reads):
//   1. per-warp range (integer min / max of the unmasked keys) and counts;
//   2. a 512-bin histogram of the unmasked scores over their value range; warp 0 finds
//      the bin tb of the kout-th largest score and the rank kk that the selection takes
//      inside tb;
//   3. the threshold-bin candidates (column, key) appended to a list; each owner ranks its
//      own candidates against the list by (key desc, column asc) and keeps those below kk;
//   4. a block scan of the per-thread selected counts gives each thread its output slots,
//      so the selection is written in ascending column order.
// Returns false, before writing anything and after a barrier that ends every use of sh,
// when the input needs the general select: a non-finite score, fewer than kout unmasked
// scores, (nearly) equal unmasked scores, or more than kSmallCand scores in the threshold
// bin. The result is block_topk's.
template <int NT, int BAR, int TID0, int E, typename Map>
__device__ bool fast_topk(const float *sc, int n, int kout, int32_t *out, Map map,
                          SelectShared<NT> &sh) {
    constexpr int NW = NT / 32, kBins = 512;
    static_assert(E == 4 || E == 8, "columns per thread");
    static_assert(kBins + 2 * kSmallCand <= kCand && NW <= 32 && 4 * NW <= 256 && E * 32 < 0x10000, "scratch");
    const int tid = (int)threadIdx.x - TID0, lane = tid & 31, warp = tid >> 5;
    uint32_t *hist = reinterpret_cast<uint32_t *>(sh.cand);             // kBins counts
    uint2 *cand = reinterpret_cast<uint2 *>(sh.cand + kBins);             // (column, key)
    uint2 *part = reinterpret_cast<uint2 *>(sh.hist);                     // per warp (min, max)
    uint32_t *pcnt = sh.hist + 2 * NW, *wtot = sh.hist + 3 * NW;          // per warp
    const int c0 = tid * E;
    const int dwarps = (n + 32 * E - 1) / (32 * E);                       // warps with columns
    const bool dw = warp < dwarps;
    float x[E];
    uint32_t key[E];
    uint32_t fr = 0u;                                  // bit e: column c0 + e is unmasked
    if (dw) {
        if (c0 + E <= n && (reinterpret_cast<uintptr_t>(sc) & 15u) == 0u) {
#pragma unroll
            for (int v = 0; v < E / 4; ++v) {
                const float4 f = reinterpret_cast<const float4 *>(sc + c0)[v];
                x[4 * v] = f.x; x[4 * v + 1] = f.y; x[4 * v + 2] = f.z; x[4 * v + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) x[e] = c0 + e < n ? sc[c0 + e] : kNeg;
        }
        uint32_t kmin = 0xffffffffu, kmax = 0u;
        bool bad = false;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            key[e] = order_key(x[e]);
            const bool fin = isfinite(x[e]);
            bad |= c0 + e < n && !fin;
            if (c0 + e < n && fin && x[e] > kMaskedBelow) {
                fr |= 1u << e;
                kmin = key[e] < kmin ? key[e] : kmin;
                kmax = key[e] > kmax ? key[e] : kmax;
            }
        }
        // count of unmasked columns (< 2^16 per warp) and a non-finite flag in one word
        const uint32_t cw = (uint32_t)__popc(fr) + (bad ? 0x10000u : 0u);
        kmin = __reduce_min_sync(0xffffffffu, kmin);
        kmax = __reduce_max_sync(0xffffffffu, kmax);
        const uint32_t cs = __reduce_add_sync(0xffffffffu, cw);
        if (lane == 0) part[warp] = make_uint2(kmin, kmax), pcnt[warp] = cs;
    }
    for (int e = tid; e < kBins / 4; e += NT) reinterpret_cast<uint4 *>(hist)[e] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) sh.ncand = 0u;
    group_sync<NT, BAR>();                                                  // 1
    float smin, scale;
    uint32_t nfree, anybad;
    {
        const uint2 pw = lane < dwarps ? part[lane] : make_uint2(0xffffffffu, 0u);
        const uint32_t pc = lane < dwarps ? pcnt[lane] : 0u;
        const uint32_t kmin = __reduce_min_sync(0xffffffffu, pw.x);
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, pw.y);
        const uint32_t csum = __reduce_add_sync(0xffffffffu, pc);  // nfree <= n < 2^16
        nfree = csum & 0xffffu;
        anybad = csum >> 16;
        smin = key_to_float(kmin);
        const float smax = key_to_float(kmax);
        scale = (float)(kBins - 1) / (smax - smin);
        anybad |= !(smax > smin) || !isfinite(scale);   // (nearly) all equal: general select
    }
    if (anybad || nfree < (uint32_t)kout) {
        group_sync<NT, BAR>();
        return false;
    }
    // value bins: non-decreasing in the score, equal scores share a bin
    uint32_t bin[E];
    if (dw) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int bi = (int)((x[e] - smin) * scale);
            bin[e] = (uint32_t)(bi < 0 ? 0 : (bi > kBins - 1 ? kBins - 1 : bi));
            if ((fr >> e) & 1u) atomicAdd(&hist[bin[e]], 1u);
        }
    }
    group_sync<NT, BAR>();                                                  // 2
    if (warp == 0) {
        // lane l scans bins 511 - 16 l down to 496 - 16 l
        uint32_t pre[16];                              // inclusive prefix, descending bins
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 h = reinterpret_cast<const uint4 *>(hist + kBins - 16 * (lane + 1))[v];
            pre[15 - 4 * v] = h.x; pre[14 - 4 * v] = h.y; pre[13 - 4 * v] = h.z; pre[12 - 4 * v] = h.w;
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1)
#pragma unroll
            for (int t = 15; t >= o; --t) pre[t] += pre[t - o];
        const uint32_t tot = pre[15];
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const uint32_t excl = incl - tot;
        if (excl < (uint32_t)kout && (uint32_t)kout <= incl) {
            // the first t whose inclusive count reaches kout: the count of those below it
            const uint32_t need = (uint32_t)kout - excl;
            uint32_t t0 = 0u, before = 0u;
#pragma unroll
            for (int t = 0; t < 16; ++t) t0 += pre[t] < need ? 1u : 0u;
#pragma unroll
            for (int t = 1; t < 16; ++t) before = (uint32_t)t == t0 ? pre[t - 1] : before;
            sh.prefix = (uint32_t)(kBins - 1 - 16 * lane) - t0;
            sh.kk = need - before;
        }
    }
    group_sync<NT, BAR>();                                                  // 3
    const uint32_t tb = sh.prefix, kk = sh.kk;
    uint32_t sel = 0u, mine = 0u;                      // bit e: selected / a tb candidate
    if (dw) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const bool f = (fr >> e) & 1u;
            if (f && bin[e] > tb) sel |= 1u << e;
            if (f && bin[e] == tb) mine |= 1u << e;
        }
        if (mine) {
            uint32_t at = atomicAdd(&sh.ncand, (uint32_t)__popc(mine));
#pragma unroll
            for (int e = 0; e < E; ++e)
                if ((mine >> e) & 1u) {
                    if (at < (uint32_t)kSmallCand) cand[at] = make_uint2((uint32_t)(c0 + e), key[e]);
                    ++at;
                }
        }
    }
    group_sync<NT, BAR>();                                                  // 4
    const uint32_t m = sh.ncand;
    if (m > (uint32_t)kSmallCand) {
        group_sync<NT, BAR>();
        return false;
    }
    if (mine) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if ((mine >> e) & 1u) {
                const uint32_t k0 = key[e], col = (uint32_t)(c0 + e);
                uint32_t r = 0u;
#pragma unroll 4
                for (uint32_t d = 0; d < m; ++d) {
                    const uint2 o = cand[d];
                    r += (o.y > k0 || (o.y == k0 && o.x < col)) ? 1u : 0u;
                }
                if (r < kk) sel |= 1u << e;
            }
        }
    }
    const uint32_t cnt_t = (uint32_t)__popc(sel);
    uint32_t excl = 0u;                                // selected columns of lower lanes
    if (dw) {
        const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
        for (int bit = 0; (1 << bit) <= E; ++bit)
            excl += (uint32_t)__popc(__ballot_sync(0xffffffffu, (cnt_t >> bit) & 1u) & lt) << bit;
        if (lane == 31) wtot[warp] = excl + cnt_t;
    }
    group_sync<NT, BAR>();                                                  // 5
    if (dw) {
        // this warp's first slot: the selected counts of the warps before it
        const uint32_t v = lane < warp ? wtot[lane] : 0u;
        uint32_t pos = __reduce_add_sync(0xffffffffu, v) + excl;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if ((sel >> e) & 1u) {
                if (pos < (uint32_t)kout) out[pos] = map((int64_t)(c0 + e));
                ++pos;
            }
        }
    }
    return true;
}

// Top kout of n <= kSmallMax scores held in shared memory, for the common case: finite
// scores, at least kout unmasked, a non-degenerate range and at most kSmallCand scores in
// the k-th score's bin; anything else goes to block_topk. Warp w owns columns
// [w * seg, (w + 1) * seg). Four passes over the scores: range; value-bin histogram (the
// bins of block_topk); threshold-bin candidates plus per-warp counts above the bin; and
// the emission. The candidates are ranked once, exactly, by (key desc, column asc) into a
// bitmap of selected columns. The selection is written in ascending column order and
// equals block_topk's. Each lane handles four columns per step, so that their shared-
// memory loads overlap (a selecting warp may be the only warp of its SM sub-partition).
// Caller guarantees 0 <= kout <= n <= kSmallMax. Contains group_sync<NT, BAR>().
constexpr int kSmallMax = (kCand - 2 * kSmallCand) * 32;
template <int NT, int BAR, int TID0, typename Map>
__device__ __noinline__ void small_topk_binned(const float *sc, int n, int kout, int32_t *out, Map map,
                                               SelectShared<NT> &sh, uint32_t *status);
template <int NT, int BAR, int TID0, typename Map>
__device__ __forceinline__ void small_topk_binned_body(const float *sc, int n, int kout, int32_t *out, Map map,
                                                       SelectShared<NT> &sh, uint32_t *status);

template <int NT, int BAR, int TID0, typename Map>
__device__ void small_topk(const float *sc, int n, int kout, int32_t *out, Map map,
                           SelectShared<NT> &sh, uint32_t *status) {
    if (kout <= 0) return;
    if (n <= 4 * NT) {
        if (fast_topk<NT, BAR, TID0, 4>(sc, n, kout, out, map, sh)) return;
    } else if (n <= 8 * NT) {
        if (fast_topk<NT, BAR, TID0, 8>(sc, n, kout, out, map, sh)) return;
    }
    small_topk_binned<NT, BAR, TID0>(sc, n, kout, out, map, sh, status);
}

// small_topk's general form (see above): value bins over the range, the threshold bin's
// candidates ranked exactly, block_topk for anything it does not resolve. Out of line for
// the kernels whose hot path is fast_topk (their code stays small); a kernel whose main
// work it is calls the inlined body, where the compiler sees that sc, out's map and sh are
// shared memory (through a generic pointer each pass ran two to three times slower).
template <int NT, int BAR, int TID0, typename Map>
__device__ __noinline__ void small_topk_binned(const float *sc, int n, int kout, int32_t *out, Map map,
                                               SelectShared<NT> &sh, uint32_t *status) {
    small_topk_binned_body<NT, BAR, TID0>(sc, n, kout, out, map, sh, status);
}

template <int NT, int BAR, int TID0, typename Map>
__device__ __forceinline__ void small_topk_binned_body(const float *sc, int n, int kout, int32_t *out, Map map,
                                                       SelectShared<NT> &sh, uint32_t *status) {
    constexpr int NW = NT / 32, U = 4;
    const int tid = (int)threadIdx.x - TID0, lane = tid & 31, warp = tid >> 5;
    const int seg = ((n + NW * 32 * U - 1) / (NW * 32 * U)) * (32 * U);
    const int lo = warp * seg, hi = lo + seg < n ? lo + seg : n;
    uint32_t *bits = reinterpret_cast<uint32_t *>(sh.cand + 2 * kSmallCand);   // selected columns
    uint32_t kmin = 0xffffffffu, kmax = 0u, nfree = 0u;
    int nonfinite = 0;
    for (int base = lo + lane; base < hi; base += 32 * U) {
        float x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = base + 32 * u < hi ? sc[base + 32 * u] : kNeg;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool fin = isfinite(x[u]);
            nonfinite |= !fin;
            if (fin && x[u] > kMaskedBelow) {
                const uint32_t key = order_key(x[u]);
                kmin = key < kmin ? key : kmin;
                kmax = key > kmax ? key : kmax;
                ++nfree;
            }
        }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    nfree = __reduce_add_sync(0xffffffffu, nfree);
    nonfinite = __reduce_or_sync(0xffffffffu, nonfinite);
    if (lane == 0) {
        sh.wg[warp] = kmin;
        sh.we[warp] = kmax;
        sh.cand[warp] = (int32_t)nfree;
        sh.cand[NW + warp] = nonfinite;
    }
    for (int e = tid; e < 256; e += NT) sh.hist[e] = 0u;
    for (int e = tid; e < (n + 31) / 32; e += NT) bits[e] = 0u;
    if (tid == 0) sh.ncand = 0u;
    group_sync<NT, BAR>();
    kmin = 0xffffffffu;
    kmax = 0u;
    nfree = 0u;
    nonfinite = 0;
    for (int w = 0; w < NW; ++w) {
        kmin = sh.wg[w] < kmin ? sh.wg[w] : kmin;
        kmax = sh.we[w] > kmax ? sh.we[w] : kmax;
        nfree += (uint32_t)sh.cand[w];
        nonfinite |= sh.cand[NW + w];
    }
    const float smin = key_to_float(kmin), smax = key_to_float(kmax);
    const float scale = 255.0f / (smax - smin);
    if (nonfinite || nfree < (uint32_t)kout || !(smax > smin) || !isfinite(scale)) {
        group_sync<NT, BAR>();                       // everyone has read sh before it is reused
        block_topk<NT, BAR, TID0>(sc, n, kout, out, map, sh, status);
        return;
    }
    auto bin_of = [&](float x) -> int {
        if (!(x >= smin)) return 0;
        if (!(x < smax)) return 255;
        const int b = (int)((x - smin) * scale);
        return b < 0 ? 0 : (b > 254 ? 254 : b);
    };
    for (int base = lo + lane; base < hi; base += 32 * U) {
        float x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = base + 32 * u < hi ? sc[base + 32 * u] : 0.f;
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + 32 * u < hi) atomicAdd(&sh.hist[bin_of(x[u])], 1u);
    }
    group_sync<NT, BAR>();
    if (warp == 0) warp_find_digit(sh.hist, 0u, (uint32_t)kout, 0, &sh.prefix, &sh.kk);
    if (tid < NW) sh.wg[tid] = 0u;                   // threshold-bin selections per warp
    group_sync<NT, BAR>();
    const int tb = (int)sh.prefix;
    const uint32_t kk = sh.kk;                       // taken from the threshold bin
    uint32_t above = 0u;
    for (int base = lo + lane; base < hi; base += 32 * U) {
        float x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = base + 32 * u < hi ? sc[base + 32 * u] : 0.f;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + 32 * u;
            if (i < hi) {
                const int b = bin_of(x[u]);
                above += b > tb ? 1u : 0u;
                if (b == tb) {
                    const uint32_t slot = atomicAdd(&sh.ncand, 1u);
                    if (slot < (uint32_t)kSmallCand) {
                        sh.cand[2 * slot] = i;
                        sh.cand[2 * slot + 1] = (int32_t)order_key(x[u]);
                    }
                }
            }
        }
    }
    above = __reduce_add_sync(0xffffffffu, above);
    if (lane == 0) sh.we[warp] = above;
    group_sync<NT, BAR>();
    const uint32_t m = sh.ncand;
    if (m > (uint32_t)kSmallCand) {
        group_sync<NT, BAR>();
        block_topk<NT, BAR, TID0>(sc, n, kout, out, map, sh, status);
        return;
    }
    // rank every candidate once; the kk first in (key desc, column asc) are selected
    for (uint32_t c = tid; c < m; c += NT) {
        const int ic = sh.cand[2 * c];
        const uint32_t kc = (uint32_t)sh.cand[2 * c + 1];
        uint32_t r = 0u;
        for (uint32_t d = 0; d < m; ++d) {
            const uint32_t kd = (uint32_t)sh.cand[2 * d + 1];
            r += (kd > kc || (kd == kc && sh.cand[2 * d] < ic)) ? 1u : 0u;
        }
        if (r < kk) {
            atomicOr(&bits[ic >> 5], 1u << (ic & 31));
            atomicAdd(&sh.wg[ic / seg], 1u);
        }
    }
    group_sync<NT, BAR>();
    uint32_t pos = 0u;
    for (int w = 0; w < warp; ++w) pos += sh.we[w] + sh.wg[w];
    const uint32_t lt = (1u << lane) - 1u;
    for (int base = lo; base < hi; base += 32 * U) {
        float x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + 32 * u + lane;
            x[u] = i < hi ? sc[i] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + 32 * u + lane;
            bool s = false;
            if (i < hi) {
                const int b = bin_of(x[u]);
                s = b > tb || (b == tb && ((bits[i >> 5] >> (i & 31)) & 1u));
            }
            const uint32_t bal = __ballot_sync(0xffffffffu, s);
            const uint32_t at = pos + __popc(bal & lt);
            if (s && at < (uint32_t)kout) out[at] = map(i);
            pos += __popc(bal);
        }
    }
    group_sync<NT, BAR>();
}

}  // namespace hisa
