// Sparse combine on the sm_103a tensor cores for the DeepSeek-V4 shape (64 query heads
// sharing one 512-dim bf16 KV head), ([HiSA issue] "Consuming the selection: sparse
// combine").
//
// One CTA owns a range of one query row's attended-row list (the visible local window
// rows, then the gathered pooled rows). The list streams through shared memory in tiles
// of kTR = 32 rows (four slots); per tile:
//   S  = Q . K^T      tcgen05, M = 64 heads, N = kTR rows, K = 512   (TMEM, 2 buffers)
//   P  = exp2(S * scale*log2e - m) per head, in the thread that owns the head's TMEM lane
//   O^T += V^T . P^T  tcgen05, M = 128 dims x 4, N = 64 heads, K = kTR  (TMEM, f32)
// K = V, so the same staged tile is the B operand of the first product (K-major) and the
// A operand of the second (MN-major). The running max m is lazy: O^T and l are rescaled
// only when a tile's max exceeds m by more than 8 (log2 units), so p <= 256.
// Warp roles: 0-3 softmax + epilogue (warp w reads TMEM lanes 32w..32w+31; in the softmax
// the two halves of a warp split each head's tile rows), 4 S = Q.K^T issue, 7 O += V^T.P^T
// issue (two issuing warps, so that neither product waits behind the other), 4 MMA issue
// and TMEM owner, 5-6 producers (cp.async gather, 128-byte swizzle, zero-fill of rows
// that are invisible or past the list). Every mbarrier wait is bounded; a timeout sets
// HISA_DEV_TIMEOUT, raises a shared abort flag and the CTA drains and exits.
#include "hisa_internal.cuh"
#include "tc_ptx.cuh"

namespace hisa {
namespace {

using namespace tc;

constexpr int kH = 64, kDH = 512, kTR = 32, kSlots = 4;
constexpr int kRPL = kTR / 32;                        // tile rows per producer lane
constexpr int kSoftWarps = 4, kMmaWarp = 4, kProdWarp0 = 5, kProdWarps = 4;
constexpr int kPvWarp = kProdWarp0 + kProdWarps;
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kThreads = 32 * (kSoftWarps + 1 + kProdWarps + 1);
constexpr uint32_t kQBytes = kH * kDH * 2;            // 64 KiB, K-major, 8 chunks of 64 dims
constexpr uint32_t kSlotBytes = kTR * kDH * 2;        // 32 KiB per staged tile
constexpr uint32_t kPBytes = kH * 128;                // P^T: 64 heads x 64 rows bf16
constexpr int kPBufs = 3;                              // P tiles in flight (softmax ahead of PV)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kQBytes;
constexpr uint32_t kOffP = kOffKV + kSlots * kSlotBytes;
constexpr uint32_t kOffBar = kOffP + kPBufs * kPBytes;
// barriers: full[4] empty[4] s_full[2] s_free[2] p_full[2] p_free[2] q_full drain
constexpr int kBarFull = 0, kBarEmpty = 4, kBarSFull = 8, kBarSFree = 10, kBarPFull = 12,
              kBarPFree = kBarPFull + kPBufs, kBarQ = kBarPFree + kPBufs, kBarDrain = kBarQ + 1,
              kNumBars = kBarDrain + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kOffIds = kOffMisc + 1024;          // this CTA's slice of I (<= kMaxTopk)
constexpr uint32_t kSmemBytes = kOffIds + kMaxTopk * 4 + 1024;  // + 1 KiB alignment slack
constexpr uint32_t kTmemCols = 512;                   // S: cols [0,128), O^T: [128, 384)
constexpr uint32_t kColO = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;

struct Misc {
    uint32_t tmem;
    int abort;
    uint64_t mask[kSlots];
    float alpha[kH];
    float factor[kH];
};

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return mbar_wait_abortable(bar, parity, abort);
}

// A wait taken by a whole warp; the result is made warp-uniform.
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort));
}

// 2^x by the hardware approximation (ex2.approx.ftz: relative error <= 2^-22; -inf -> +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void named_sync_soft() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

__device__ __forceinline__ uint32_t named_or_soft(uint32_t v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(v) : "memory");
    return r;
}

__global__ void __launch_bounds__(kThreads, 1) k_attend_tc(AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    Misc *misc = reinterpret_cast<Misc *>(smem + kOffMisc);
    volatile int *abort = &misc->abort;

    grid_dep_wait();                                    // before the first global access
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = blockIdx.x, split = blockIdx.y;
    const int bq = row / p.L, j = row - bq * p.L;
    const int64_t t = (int64_t)p.t0[bq] + j;
    const int64_t k0 = p.kv_off[bq];
    int64_t Np = p.kv_off[bq + 1] - k0;
    const bool bad_off = !seq_ok(p.kv_off, bq, p.Np_max, p.kv_rows);
    if (bad_off) Np = 0;
    // visible local window rows [lo, hi) of this query row
    int64_t nl = p.local_len[bq];
    nl = nl < 0 ? 0 : (nl > p.W_max ? p.W_max : nl);
    const int64_t pos0 = p.local_pos0[bq];
    int64_t lo = t - p.window + 1 - pos0, hi = t - pos0 + 1;
    lo = lo < 0 ? 0 : lo;
    hi = hi > nl ? nl : hi;
    const int64_t nloc = hi > lo ? hi - lo : 0;
    const int64_t npool = p.I ? (int64_t)p.k : Np;
    const int64_t ntot = nloc + npool;
    const int64_t e0 = (int64_t)split * p.rows_per_split;
    int64_t e1 = e0 + p.rows_per_split;
    e1 = e1 > ntot ? ntot : e1;
    const int T = e1 > e0 ? (int)((e1 - e0 + kTR - 1) / kTR) : 0;
    const int64_t V = p.causal ? visible_len(t, p.r, Np) : Np;
    const __nv_bfloat16 *local =
        reinterpret_cast<const __nv_bfloat16 *>(p.local_kv) + ((int64_t)bq * p.W_max + lo) * kDH;
    const __nv_bfloat16 *pooled = reinterpret_cast<const __nv_bfloat16 *>(p.pooled_kv) + k0 * kDH;
    const int32_t *Irow = p.I ? p.I + (int64_t)row * p.k : nullptr;

    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) {
            uint32_t cnt = 1;
            if (b >= kBarFull && b < kBarFull + kSlots) cnt = kProdThreads + 1;
            if (b == kBarSFree || b == kBarSFree + 1 || (b >= kBarPFull && b < kBarPFull + kPBufs))
                cnt = kSoftWarps * 32;
            if (b == kBarQ) cnt = kProdThreads;
            if (b == kBarDrain) cnt = 2;                  // one commit from each issuing warp
            mbar_init(&bars[b], cnt);
        }
        mbar_fence_init();
        misc->abort = 0;
        if (bad_off && split == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&misc->tmem, kTmemCols);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = misc->tmem;

    if (warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps) {
        // ---------------- producers ----------------
        const int pt = tid - kProdWarp0 * 32;
        const int pu = pt & 63;                               // the 16-byte unit of a row it copies
        const int pr0 = pt >> 6;                              // first row; rows pr0, pr0 + kRowStep, ...
        constexpr int kRowStep = kProdThreads / 64;
        constexpr int kPre = 512 / kProdThreads;
        int32_t *ids = reinterpret_cast<int32_t *>(smem + kOffIds);
        const int64_t kk0 = e0 > nloc ? e0 - nloc : 0;
        const int64_t kk1 = e1 > nloc ? e1 - nloc : 0;
        // the first 512 selected ids of this CTA's range, fetched now, staged after the
        // local-window tiles are on their way
        int32_t pre[kPre];
#pragma unroll
        for (int m = 0; m < kPre; ++m) {
            const int64_t kk = kk0 + pt + kProdThreads * m;
            pre[m] = (Irow && kk < kk1) ? Irow[kk] : -1;
        }
        const uint32_t qb = sbase + kOffQ;
        const __nv_bfloat16 *qrow = reinterpret_cast<const __nv_bfloat16 *>(p.q) + (int64_t)row * kH * kDH;
        for (int h = pr0; h < kH; h += kRowStep)
            cp_async16(qb + (pu >> 3) * (kH * 128) + sw128_offset(h, (pu & 7) * 8),
                       qrow + h * kDH + pu * 8);
        cp_async_arrive(&bars[kBarQ]);
        // gathers tile i into slot i % kSlots (the slot must be free)
        auto issue_tile = [&](int i) {
            const int s = i % kSlots;
            // lane r resolves rows r, r + 32, ... of the tile
            const __nv_bfloat16 *src[kRPL];
            uint32_t valid[kRPL];
#pragma unroll
            for (int hlf = 0; hlf < kRPL; ++hlf) {
                src[hlf] = nullptr;
                const int64_t e = e0 + (int64_t)i * kTR + hlf * 32 + lane;
                if (e < e1) {
                    if (e < nloc) {
                        src[hlf] = local + e * kDH;
                    } else {
                        const int64_t kk = e - nloc;
                        const int64_t id = Irow ? (int64_t)ids[kk - kk0] : kk;
                        if (id >= Np || id < -1) {
                            if (pt < 32) flag(p.status, HISA_DEV_BAD_ID);
                        } else if (id >= 0 && id < V) {
                            src[hlf] = pooled + id * kDH;
                        }
                    }
                }
                valid[hlf] = __ballot_sync(0xffffffffu, src[hlf] != nullptr);
            }
            const uint32_t slot = sbase + kOffKV + s * kSlotBytes;
            const uint32_t dst0 = slot + (pu >> 3) * (kTR * 128);
#pragma unroll 4
            for (int r = pr0; r < kTR; r += kRowStep) {
                const __nv_bfloat16 *rs = reinterpret_cast<const __nv_bfloat16 *>(__shfl_sync(
                    0xffffffffu, reinterpret_cast<uintptr_t>(src[r >> 5]), r & 31));
                const bool v = (valid[r >> 5] >> (r & 31)) & 1u;
                cp_async16_zfill(dst0 + sw128_offset(r, (pu & 7) * 8),
                                 v ? static_cast<const void *>(rs + pu * 8) : p.q, v);
            }
            if (pt == 0) {
                uint64_t m = 0;
#pragma unroll
                for (int hlf = 0; hlf < kRPL; ++hlf) m |= (uint64_t)valid[hlf] << (32 * hlf);
                misc->mask[s] = m;
            }
            cp_async_arrive(&bars[kBarFull + s]);
            if (pt == 0) mbar_arrive(&bars[kBarFull + s]);
        };
        // leading tiles with local rows only go out before the ids are staged
        int n_pre = 0;
        while (n_pre < T && n_pre < kSlots) {
            const int64_t end = e0 + (int64_t)(n_pre + 1) * kTR;
            if ((end < e1 ? end : e1) > nloc) break;
            issue_tile(n_pre++);
        }
        if (Irow) {
#pragma unroll
            for (int m = 0; m < kPre; ++m) {
                const int64_t kk = kk0 + pt + kProdThreads * m;
                if (kk < kk1) ids[kk - kk0] = pre[m];
            }
            for (int64_t base = kk0 + 512; base < kk1; base += 512) {
                int32_t v[kPre];
#pragma unroll
                for (int m = 0; m < kPre; ++m) {
                    const int64_t kk = base + pt + kProdThreads * m;
                    v[m] = kk < kk1 ? Irow[kk] : -1;
                }
#pragma unroll
                for (int m = 0; m < kPre; ++m) {
                    const int64_t kk = base + pt + kProdThreads * m;
                    if (kk < kk1) ids[kk - kk0] = v[m];
                }
            }
        }
        asm volatile("bar.sync 2, %0;" ::"n"(kProdThreads) : "memory");   // the producer warps
        bool ok = true;
        for (int i = n_pre; i < T; ++i) {
            const int s = i % kSlots;
            if (i >= kSlots && !wait_bar(&bars[kBarEmpty + s], ((i / kSlots) - 1) & 1, abort)) {
                ok = false;
                break;
            }
            issue_tile(i);
        }
        cp_async_wait_all();
        if (!ok) {
            *abort = 1;
            flag(p.status, HISA_DEV_TIMEOUT);
        }
    } else if (warp == kMmaWarp || warp == kPvWarp) {
        // ---------------- MMA issue (warp-uniform loops, one elected lane issues) ------
        if (T > 0) {
            const uint32_t id_s = idesc_bf16_f32(64, kTR, 0, 0);   // N = kTR rows
            const uint32_t id_o = idesc_bf16_f32(128, 64, 1, 0);
            const uint64_t qd = smem_desc_sw128(sbase + kOffQ, 16, 1024);
            bool ok = wait_bar_warp(&bars[kBarQ], 0, abort);
            auto issue_s = [&](int i) -> bool {
                const int s = i % kSlots, sb = i & 1;
                if (!wait_bar_warp(&bars[kBarFull + s], (i / kSlots) & 1, abort)) return false;
                if (i >= 2 && !wait_bar_warp(&bars[kBarSFree + sb], ((i >> 1) - 1) & 1, abort)) return false;
                fence_after_sync();
                const uint64_t bd = smem_desc_sw128(sbase + kOffKV + s * kSlotBytes, 16, 1024);
                const uint32_t d = tmem + sb * kTR;
#pragma unroll
                for (int ks = 0; ks < kDH / 16; ++ks) {
                    const uint32_t ko = (ks >> 2), kb = (ks & 3) * 32;
                    mma_bf16_warp(d, desc_add(qd, ko * (kH * 128) + kb),
                             desc_add(bd, ko * (kTR * 128) + kb), id_s, ks > 0);
                }
                mma_commit_warp(&bars[kBarSFull + sb]);
                return true;
            };
            auto issue_pv = [&](int i) -> bool {
                const int s = i % kSlots, pb = i % kPBufs;
                if (!wait_bar_warp(&bars[kBarPFull + pb], (i / kPBufs) & 1, abort)) return false;
                fence_after_sync();
                const uint64_t ad = smem_desc_sw128(sbase + kOffKV + s * kSlotBytes, kTR * 128, 1024);
                const uint64_t bd = smem_desc_sw128(sbase + kOffP + pb * kPBytes, 16, 1024);
                const uint32_t first = i > 0 ? 1u : 0u;
#pragma unroll
                for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                    for (int ks = 0; ks < kTR / 16; ++ks)
                        mma_bf16_warp(tmem + kColO + mt * 64, desc_add(ad, (2 * mt) * (kTR * 128) + ks * 2048),
                                 desc_add(bd, ks * 32), id_o, ks > 0 ? 1u : first);
                mma_commit_warp(&bars[kBarEmpty + s]);
                mma_commit_warp(&bars[kBarPFree + pb]);
                return true;
            };
            if (warp == kMmaWarp)
                for (int i = 0; i < T && ok; ++i) ok = issue_s(i);
            else
                for (int i = 0; i < T && ok; ++i) ok = issue_pv(i);
            if (!ok) {
                *abort = 1;
                flag(p.status, HISA_DEV_TIMEOUT);
            }
            // drain: every MMA issued by either warp has completed before TMEM is freed
            // (a bounded wait that an abort does not cut short)
            mma_commit_warp(&bars[kBarDrain]);
            __syncwarp();
            mbar_wait(&bars[kBarDrain], 0, 1u << 24);
            __syncwarp();
        }
    } else {
        // ---------------- softmax + epilogue (warps 0-3) ----------------
        // S rows (heads) live in TMEM lanes 0-15 of each quadrant (M = 64). Lane l of warp w
        // owns head 16 w + (l % 16) and the tile rows 16 (l / 16) .. + 15: the two lanes of a
        // head combine their max and sum with one shuffle.
        const bool lead = lane < 16;                    // writes the head's shared values
        const int h = warp * 16 + (lane & 15);
        const int half = lane >> 4;
        const float c2 = p.scale * kLog2e;
        const float sink2 = p.sinks[h] * kLog2e;
        float m2 = -INFINITY, l = 0.f;
        uint32_t pfree_seen[kPBufs] = {};
        bool ok = true;
        auto wait_pfree = [&](int buf, uint32_t phase) -> bool {   // PV of tile (kPBufs*phase + buf) done
            while (pfree_seen[buf] <= phase) {
                if (!wait_bar(&bars[kBarPFree + buf], pfree_seen[buf] & 1, abort)) return false;
                ++pfree_seen[buf];
            }
            return true;
        };
        constexpr int kHR = kTR / 2;                    // rows per lane
        for (int i = 0; i < T && ok; ++i) {
            const int s = i % kSlots, sb = i & 1;
            if (!wait_bar(&bars[kBarFull + s], (i / kSlots) & 1, abort) ||
                !wait_bar(&bars[kBarSFull + sb], (i >> 1) & 1, abort)) {
                ok = false;
                break;
            }
            fence_after_sync();
            const uint32_t mask = (uint32_t)(misc->mask[s] >> (kHR * half));
            float v[kHR];
            tmem_ld16_x2(tmem + ((uint32_t)(32 * warp) << 16) + sb * kTR, v);
            tmem_ld_wait();
            fence_before_sync();
            mbar_arrive(&bars[kBarSFree + sb]);
#pragma unroll
            for (int r = 0; r < kHR; ++r) v[r] = ((mask >> r) & 1u) ? v[r] * c2 : -INFINITY;
            float mx[kHR / 2];                              // pairwise tree: short dependency chains
#pragma unroll
            for (int r = 0; r < kHR / 2; ++r) mx[r] = fmaxf(v[2 * r], v[2 * r + 1]);
#pragma unroll
            for (int w = kHR / 4; w >= 1; w >>= 1)
#pragma unroll
                for (int r = 0; r < w; ++r) mx[r] = fmaxf(mx[r], mx[r + w]);
            const float tmax = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], 16));
            float alpha = 1.f;
            uint32_t resc = 0;
            if (tmax > m2 + kLazy) {
                if (m2 != -INFINITY) {
                    alpha = ex2_approx(m2 - tmax);
                    resc = 1;
                }
                m2 = tmax;
            }
            // exp2(-inf - m) = +0 in the hardware approximation; m2 is finite once any row
            // of this head was visible, and rows are only ever -inf when masked
            const float msub = m2 == -INFINITY ? 0.f : m2;
            float pr[kHR];
#pragma unroll
            for (int r = 0; r < kHR; ++r) pr[r] = ex2_approx(v[r] - msub);
            uint32_t packed[kHR / 2];
#pragma unroll
            for (int r = 0; r < kHR; r += 2) {
                __nv_bfloat162 b2 = __floats2bfloat162_rn(pr[r], pr[r + 1]);
                packed[r / 2] = *reinterpret_cast<uint32_t *>(&b2);
            }
#pragma unroll
            for (int w = kHR / 2; w >= 1; w >>= 1)
#pragma unroll
                for (int r = 0; r < w; ++r) pr[r] += pr[r + w];
            const float sum = pr[0] + __shfl_xor_sync(0xffffffffu, pr[0], 16);
            // P buffer i % kPBufs is free once PV(i - kPBufs) has completed
            if (i >= kPBufs && !wait_pfree(i % kPBufs, (uint32_t)(i / kPBufs - 1))) { ok = false; break; }
            l = l * alpha + sum;
            {
                uint8_t *pb = smem + kOffP + (i % kPBufs) * kPBytes;
#pragma unroll
                for (int u = 0; u < kHR / 8; ++u)
                    *reinterpret_cast<uint4 *>(pb + sw128_offset(h, (half * (kHR / 8) + u) * 8)) =
                        make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
            }
            if (named_or_soft(resc)) {
                // rescale O^T columns of the heads whose reference max moved up
                if (lead) misc->alpha[h] = alpha;
                named_sync_soft();
                if (!wait_pfree((i - 1) % kPBufs, (uint32_t)((i - 1) / kPBufs))) { ok = false; break; }
                fence_after_sync();
#pragma unroll 1
                for (int mt = 0; mt < 4; ++mt)
#pragma unroll 1
                    for (int c = 0; c < 64; c += 16) {
                        float o[16];
                        const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16) + kColO + mt * 64 + c;
                        tmem_ld16(ta, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 16; ++q) o[q] *= misc->alpha[c + q];
                        tmem_st16(ta, o);
                    }
                tmem_st_wait();
            }
            fence_async_smem();
            fence_before_sync();
            mbar_arrive(&bars[kBarPFull + (i % kPBufs)]);
        }
        // ---------------- epilogue ----------------
        if (ok && T > 0) ok = wait_pfree((T - 1) % kPBufs, (uint32_t)((T - 1) / kPBufs));
        if (!ok) {
            *abort = 1;
            flag(p.status, HISA_DEV_TIMEOUT);
        }
        fence_after_sync();
        const bool have_o = ok && T > 0;
        if (p.nsplit == 1) {
            if (lead) {
                const float M = fmaxf(m2, sink2);
                const float wm = (m2 == -INFINITY) ? 0.f : exp2f(m2 - M);
                misc->factor[h] = wm / (l * wm + exp2f(sink2 - M));
            }
            named_sync_soft();
            float *out = p.out + (int64_t)row * kH * kDH;
            for (int mt = 0; mt < 4; ++mt) {
                const int d = mt * 128 + warp * 32 + lane;
                for (int c = 0; c < 64; c += 16) {
                    float o[16];
                    if (have_o) {
                        tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + kColO + mt * 64 + c, o);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q) o[q] = 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q) out[(c + q) * kDH + d] = o[q] * misc->factor[c + q];
                }
            }
        } else {
            float *base = p.part + ((int64_t)row * p.nsplit + split) * kH * (kDH + 2);
            if (lead) {
                base[h * (kDH + 2)] = (m2 == -INFINITY) ? -INFINITY : m2 / kLog2e;
                base[h * (kDH + 2) + 1] = l;
            }
            for (int mt = 0; mt < 4; ++mt) {
                const int d = mt * 128 + warp * 32 + lane;
                for (int c = 0; c < 64; c += 16) {
                    float o[16];
                    if (have_o) {
                        tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + kColO + mt * 64 + c, o);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q) o[q] = 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q) base[(c + q) * (kDH + 2) + 2 + d] = o[q];
                }
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int attend_tc_supported(int H, int Dh, int kv_bf16) { return H == kH && Dh == kDH && kv_bf16; }

cudaError_t launch_attend_tc(const AttnParams &p, cudaStream_t s) {
    static const cudaError_t attr = cudaFuncSetAttribute(
        k_attend_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (attr != cudaSuccess) return attr;
    dim3 grid((unsigned)(p.B * p.L), (unsigned)p.nsplit);
    cudaError_t e = launch_pdl(k_attend_tc, grid, dim3(kThreads), kSmemBytes, s, p);
    if (e != cudaSuccess || p.nsplit == 1) return e;
    return launch_attend_combine(p, s);
}

}  // namespace hisa
