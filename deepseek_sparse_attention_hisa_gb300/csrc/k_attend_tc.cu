// Sparse combine on the sm_103a tensor cores for the DeepSeek-V4 shape (64 query heads
// sharing one 512-dim bf16 KV head), ([HiSA issue] "Consuming the selection: sparse
// combine").
//
// A work item is a range of one query row's attended-row list (the visible local window
// rows, then the gathered pooled rows). One CTA per SM walks the items blockIdx.x,
// blockIdx.x + gridDim.x, ...; the list tiles of consecutive items stream through the
// same kSlots = 5 ring slots, so an item's start (q, first tiles) and end (the epilogue) overlap its
// neighbours' streaming. The list streams in tiles of kTR = 32 rows; per tile:
//   S  = Q . K^T      tcgen05, M = 64 heads, N = kTR rows, K = 512   (TMEM, 2 buffers)
//   P  = exp2(S * scale*log2e - m) per head, in the thread that owns the head's TMEM lane
//   O^T += V^T . P^T  tcgen05, M = 128 dims x 4, N = 64 heads, K = kTR  (TMEM, f32)
// K = V, so the same staged tile is the B operand of the first product (K-major) and the
// A operand of the second (MN-major). The running max m is lazy: O^T and l are rescaled
// only when a tile's max exceeds m by more than 8 (log2 units), so p <= 256.
// Warp roles: 0-3 softmax (warp w reads TMEM lanes 32w..32w+31; the two halves of a warp
// split each head's tile rows), 4 S = Q.K^T issue and TMEM owner, 5-8 producers (cp.async
// gather, 128-byte swizzle, zero-fill of rows that are invisible or past the list), 9
// O += V^T.P^T issue (two issuing warps, so that neither product waits behind the other),
// 10-13 epilogue (each item's q dims 0-255 from its ring slot into TMEM, the next item's
// as soon as this item's S products are done, then O^T -> out while the other warps
// start the next item). Every mbarrier
// wait is bounded; a timeout sets HISA_DEV_TIMEOUT, raises a shared abort flag and the CTA
// drains and exits.
#include "hisa_internal.cuh"
#include "tc_ptx.cuh"

namespace hisa {
namespace {

using namespace tc;

constexpr int kH = 64, kDH = 512, kTR = 32, kSlots = 5;
constexpr int kRPL = kTR / 32;                        // tile rows per producer lane
constexpr int kSoftWarps = 4, kMmaWarp = 4, kProdWarp0 = 5, kProdWarps = 4;
constexpr int kPvWarp = kProdWarp0 + kProdWarps;
constexpr int kEpiWarp0 = kPvWarp + 1, kEpiWarps = 4;
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kBarSoft = 1, kBarProd = 2, kBarEpi = 3; // named barriers (0 = __syncthreads)
// q: dims [0, kQT) are the A operand of the S products from TMEM (copied there through a
// ring slot at the start of each item), dims [kQT, 512) from shared memory
constexpr int kQT = 256;
constexpr uint32_t kQChunk = kH * 128;                // one 64-dim chunk of q, 8 KiB
constexpr uint32_t kQBytes = (kDH - kQT) / 64 * kQChunk;   // 32 KiB in shared memory
constexpr uint32_t kSlotBytes = kTR * kDH * 2;        // 32 KiB per staged tile
constexpr uint32_t kPBytes = kH * 128;                // P^T: 64 heads x 64 rows bf16
constexpr int kPBufs = 3;                              // P tiles in flight (softmax ahead of PV)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kQBytes;
constexpr uint32_t kOffP = kOffKV + kSlots * kSlotBytes;
constexpr uint32_t kOffBar = kOffP + kPBufs * kPBytes;
// barriers: full[5] empty[5] s_full[2] s_free[2] p_full[3] p_free[3]; per item: q_full
// (q's shared-memory dims landed), q_tmem (its TMEM dims written), q_free (the item's S
// products are done), o_full (its PV products are done), o_free (the epilogue has read
// O^T), stat (the softmax wrote the item's per-head statistics); drain
constexpr int kBarFull = 0, kBarEmpty = kSlots, kBarSFull = 2 * kSlots, kBarSFree = kBarSFull + 2,
              kBarPFull = kBarSFree + 2, kBarPFree = kBarPFull + kPBufs, kBarQ = kBarPFree + kPBufs,
              kBarQT = kBarQ + 1, kBarQFree = kBarQT + 1,
              kBarOFull = kBarQFree + 1, kBarOFree = kBarOFull + 1, kBarStat = kBarOFree + 1,
              kBarDrain = kBarStat + 1, kNumBars = kBarDrain + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kOffIds = kOffMisc + 1536;          // an item's slice of I (<= kMaxTopk)
constexpr uint32_t kSmemBytes = kOffIds + kMaxTopk * 4 + 1024;  // + 1 KiB alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
constexpr uint32_t kTmemCols = 512;                   // S: [0, 64), O^T: [64, 320), q: [320, 448)
constexpr uint32_t kColO = 64;
constexpr uint32_t kColQ = 320;
static_assert(kColO + 256 <= kColQ && kColQ + kQT / 2 <= kTmemCols, "TMEM columns");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;

struct Misc {
    uint32_t tmem;
    int abort;
    uint64_t mask[kSlots];
    float alpha[kH];
    float factor[kH];                                 // nsplit = 1: out scale of each head
    float stat_m[kH], stat_l[kH];                     // nsplit > 1: running max and sum
};
static_assert(sizeof(Misc) <= 1536, "misc block");

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


__device__ __forceinline__ uint32_t named_or_soft(uint32_t v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(v) : "memory");
    return r;
}

// What every role derives for one work item (a query row, or one split of its list).
struct Item {
    int row, split, bq;
    int64_t t, k0, Np, V;
    int64_t lo, nloc, e0, e1;      // visible local window [lo, lo + nloc); list range [e0, e1)
    int T;                         // tiles of kTR list entries
    bool bad_off;
};

__device__ __forceinline__ Item item_of(const AttnParams &p, int id) {
    Item x;
    x.row = id / p.nsplit;
    x.split = id - x.row * p.nsplit;
    x.bq = x.row / p.L;
    const int j = x.row - x.bq * p.L;
    x.t = (int64_t)p.t0[x.bq] + j;
    x.k0 = p.kv_off[x.bq];
    x.Np = p.kv_off[x.bq + 1] - x.k0;
    x.bad_off = !seq_ok(p.kv_off, x.bq, p.Np_max, p.kv_rows);
    if (x.bad_off) x.Np = 0;
    int64_t nl = p.local_len[x.bq];
    nl = nl < 0 ? 0 : (nl > p.W_max ? p.W_max : nl);
    const int64_t pos0 = p.local_pos0[x.bq];
    int64_t lo = x.t - p.window + 1 - pos0, hi = x.t - pos0 + 1;
    lo = lo < 0 ? 0 : lo;
    hi = hi > nl ? nl : hi;
    x.lo = lo;
    x.nloc = hi > lo ? hi - lo : 0;
    const int64_t npool = p.I ? (int64_t)p.k : x.Np;
    const int64_t ntot = x.nloc + npool;
    x.e0 = (int64_t)x.split * p.rows_per_split;
    x.e1 = x.e0 + p.rows_per_split;
    x.e1 = x.e1 > ntot ? ntot : x.e1;
    x.T = x.e1 > x.e0 ? (int)((x.e1 - x.e0 + kTR - 1) / kTR) : 0;
    x.V = p.causal ? visible_len(x.t, p.r, x.Np) : x.Np;
    return x;
}

// True on every participating thread iff v is true on all of them (named barrier id).
__device__ __forceinline__ bool group_all(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0u;
}

__global__ void __launch_bounds__(kThreads, 1) k_attend_tc(AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    Misc *misc = reinterpret_cast<Misc *>(smem + kOffMisc);
    volatile int *abort = &misc->abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int items = p.B * p.L * p.nsplit;

    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) {
            uint32_t cnt = 1;
            if (b >= kBarFull && b < kBarFull + kSlots) cnt = kProdThreads + 1;
            if (b == kBarSFree || b == kBarSFree + 1 || (b >= kBarPFull && b < kBarPFull + kPBufs) ||
                b == kBarStat)
                cnt = kSoftWarps * 32;
            if (b == kBarQ) cnt = kProdThreads;
            if (b == kBarQT) cnt = kEpiWarps * 32;
            if (b == kBarOFree) cnt = kEpiWarps * 32;
            if (b == kBarDrain) cnt = 2;                  // one commit from each issuing warp
            mbar_init(&bars[b], cnt);
        }
        mbar_fence_init();
        misc->abort = 0;
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&misc->tmem, kTmemCols);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = misc->tmem;
    // no grid_dep_wait() here: the producers wait before their first selected id and the
    // epilogue before its first output write; the first item's q and local rows go first
    bool ok = true;
    auto fail = [&]() {
        ok = false;
        *abort = 1;
    };

    if (warp >= kProdWarp0 && warp < kProdWarp0 + kProdWarps) {
        // ---------------- producers: q and the list tiles of each item ----------------
        const int pt = tid - kProdWarp0 * 32;
        const int pu = pt & 63;                               // the 16-byte unit of a row it copies
        const int pr0 = pt >> 6;                              // first row; rows pr0, pr0 + kRowStep, ...
        constexpr int kRowStep = kProdThreads / 64;
        constexpr int kPre = 512 / kProdThreads;
        int32_t *ids = reinterpret_cast<int32_t *>(smem + kOffIds);
        uint32_t g = 0;                                       // list tiles issued (all items)
        int n = 0;
        bool waited = false;                                  // grid_dep_wait() done
        for (int id = blockIdx.x; id < items; id += gridDim.x, ++n) {
            const Item x = item_of(p, id);
            const __nv_bfloat16 *qrow = reinterpret_cast<const __nv_bfloat16 *>(p.q) + (int64_t)x.row * kH * kDH;
            // the item's q: dims [0, kQT) into the next ring slot (its Full barrier, like a
            // tile's; the epilogue warps move them into TMEM and free the slot), dims [kQT, 512)
            // into the q region once the previous item's S products are done with it
            auto issue_q = [&]() -> bool {
                const int s = g % kSlots;
                const bool w = g < (uint32_t)kSlots || wait_bar(&bars[kBarEmpty + s], ((g / kSlots) - 1) & 1, abort);
                if (!group_all(kBarProd, kProdThreads, w)) return false;
                const uint32_t slot = sbase + kOffKV + s * kSlotBytes;
                const int qu = pt & 31;                         // 16-byte unit of dims [0, kQT)
                for (int h = pt >> 5; h < kH; h += kProdThreads / 32)
                    cp_async16(slot + (qu >> 3) * kQChunk + sw128_offset(h, (qu & 7) * 8), qrow + h * kDH + qu * 8);
                cp_async_arrive(&bars[kBarFull + s]);
                if (pt == 0) mbar_arrive(&bars[kBarFull + s]);
                ++g;
                const bool wq = n < 1 || wait_bar(&bars[kBarQFree], (n - 1) & 1, abort);
                if (!group_all(kBarProd, kProdThreads, wq)) return false;
                const uint32_t qb = sbase + kOffQ;
                for (int h = pt >> 5; h < kH; h += kProdThreads / 32)
                    cp_async16(qb + (qu >> 3) * kQChunk + sw128_offset(h, (qu & 7) * 8),
                               qrow + h * kDH + kQT + qu * 8);
                cp_async_arrive(&bars[kBarQ]);
                return true;
            };
            // the first item's q depends on its row alone, so it goes out before anything waits
            // for the item's metadata loads (item_of): the kernel's start is shorter by one
            // dependent load
            if (n == 0 && !issue_q()) { fail(); break; }
            if (x.bad_off && x.split == 0 && pt == 0) flag(p.status, HISA_DEV_BAD_OFFSETS);
            const __nv_bfloat16 *local =
                reinterpret_cast<const __nv_bfloat16 *>(p.local_kv) + ((int64_t)x.bq * p.W_max + x.lo) * kDH;
            const __nv_bfloat16 *pooled = reinterpret_cast<const __nv_bfloat16 *>(p.pooled_kv) + x.k0 * kDH;
            const int32_t *Irow = p.I ? p.I + (int64_t)x.row * p.k : nullptr;
            const int64_t kk0 = x.e0 > x.nloc ? x.e0 - x.nloc : 0;
            const int64_t kk1 = x.e1 > x.nloc ? x.e1 - x.nloc : 0;
            // the first 512 selected ids of the item, fetched now (the first item: once its q
            // and local tiles are issued and the previous grid is done), staged after the local tiles
            int32_t pre[kPre];
            auto fetch_pre = [&]() {
#pragma unroll
                for (int m = 0; m < kPre; ++m) {
                    const int64_t kk = kk0 + pt + kProdThreads * m;
                    pre[m] = (Irow && kk < kk1) ? Irow[kk] : -1;
                }
            };
            if (waited) fetch_pre();
            if (n > 0 && !issue_q()) { fail(); break; }
            // gathers tile i of the item into slot g % kSlots, once that slot is free
            auto issue_tile = [&](int i) -> bool {
                const int s = g % kSlots;
                const bool w = g < (uint32_t)kSlots || wait_bar(&bars[kBarEmpty + s], ((g / kSlots) - 1) & 1, abort);
                if (!group_all(kBarProd, kProdThreads, w)) return false;
                // lane r resolves rows r, r + 32, ... of the tile
                const __nv_bfloat16 *src[kRPL];
                uint32_t valid[kRPL];
#pragma unroll
                for (int hlf = 0; hlf < kRPL; ++hlf) {
                    src[hlf] = nullptr;
                    const int64_t e = x.e0 + (int64_t)i * kTR + hlf * 32 + lane;
                    if (e < x.e1) {
                        if (e < x.nloc) {
                            src[hlf] = local + e * kDH;
                        } else {
                            const int64_t kk = e - x.nloc;
                            const int64_t idv = Irow ? (int64_t)ids[kk - kk0] : kk;
                            if (idv >= x.Np || idv < -1) {
                                if (pt < 32) flag(p.status, HISA_DEV_BAD_ID);
                            } else if (idv >= 0 && idv < x.V) {
                                src[hlf] = pooled + idv * kDH;
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
                ++g;
                return true;
            };
            // leading tiles with local rows only go out before the ids are staged
            int i = 0;
            bool good = true;
            while (good && i < x.T) {
                const int64_t end = x.e0 + (int64_t)(i + 1) * kTR;
                if ((end < x.e1 ? end : x.e1) > x.nloc) break;
                good = issue_tile(i++);
            }
            if (!good) { fail(); break; }
            if (!waited) {
                grid_dep_wait();
                waited = true;
                fetch_pre();
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
            asm volatile("bar.sync %0, %1;" ::"n"(kBarProd), "n"(kProdThreads) : "memory");
            for (; good && i < x.T; ++i) good = issue_tile(i);
            // the next item restages the ids: every tile of this one has read its own
            asm volatile("bar.sync %0, %1;" ::"n"(kBarProd), "n"(kProdThreads) : "memory");
            if (!good) { fail(); break; }
        }
        cp_async_wait_all();
    } else if (warp == kMmaWarp || warp == kPvWarp) {
        // ---------------- MMA issue (warp-uniform loops, one elected lane issues) ------
        const uint32_t id_s = idesc_bf16_f32(64, kTR, 0, 0);   // N = kTR rows
        const uint32_t id_o = idesc_bf16_f32(128, 64, 1, 0);
        const uint64_t qd = smem_desc_sw128(sbase + kOffQ, 16, 1024);
        uint32_t g = 0;                                   // ring entries (q slots and list tiles)
        uint32_t gt = 0;                                  // list tiles (all items)
        int n = 0;
        for (int id = blockIdx.x; id < items && ok; id += gridDim.x, ++n) {
            const Item x = item_of(p, id);
            ++g;                                          // the ring entry that carried q
            if (warp == kMmaWarp) {
                // S = Q . K^T of every tile of the item, then release q to the producers
                if (!wait_bar_warp(&bars[kBarQ], n & 1, abort) || !wait_bar_warp(&bars[kBarQT], n & 1, abort)) {
                    fail();
                    break;
                }
                fence_after_sync();
                for (int i = 0; i < x.T; ++i, ++g, ++gt) {
                    const int s = g % kSlots, sb = gt & 1;
                    if (!wait_bar_warp(&bars[kBarFull + s], (g / kSlots) & 1, abort) ||
                        (gt >= 2 && !wait_bar_warp(&bars[kBarSFree + sb], ((gt >> 1) - 1) & 1, abort))) {
                        fail();
                        break;
                    }
                    fence_after_sync();
                    const uint64_t bd = smem_desc_sw128(sbase + kOffKV + s * kSlotBytes, 16, 1024);
                    const uint32_t d = tmem + sb * kTR;
#pragma unroll
                    for (int ks = 0; ks < kQT / 16; ++ks) {        // q dims from TMEM
                        const uint32_t ko = (ks >> 2), kb = (ks & 3) * 32;
                        mma_bf16_tmem_a_warp(d, tmem + kColQ + ks * 8, desc_add(bd, ko * (kTR * 128) + kb), id_s,
                                             ks > 0);
                    }
#pragma unroll
                    for (int ks = kQT / 16; ks < kDH / 16; ++ks) { // q dims from shared memory
                        const uint32_t ko = (ks >> 2), kb = (ks & 3) * 32;
                        mma_bf16_warp(d, desc_add(qd, (ko - kQT / 64) * kQChunk + kb),
                                      desc_add(bd, ko * (kTR * 128) + kb), id_s, 1u);
                    }
                    mma_commit_warp(&bars[kBarSFull + sb]);
                }
                if (!ok) break;
                mma_commit_warp(&bars[kBarQFree]);
                // the CTA's last item has all its S products: a successor may launch during
                // its last PV products and epilogue (it waits for this grid)
                if (id + (int)gridDim.x >= items) grid_dep_trigger();
            } else {
                // O^T += V^T . P^T of every tile; O^T starts from zero once the previous item's
                // epilogue has read it, and is handed to the epilogue after the last tile
                if (n >= 1 && !wait_bar_warp(&bars[kBarOFree], (n - 1) & 1, abort)) { fail(); break; }
                fence_after_sync();
                for (int i = 0; i < x.T; ++i, ++g, ++gt) {
                    const int s = g % kSlots, pb = gt % kPBufs;
                    if (!wait_bar_warp(&bars[kBarPFull + pb], (gt / kPBufs) & 1, abort)) { fail(); break; }
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
                }
                if (!ok) break;
                mma_commit_warp(&bars[kBarOFull]);
            }
        }
        // drain: every MMA issued by either warp has completed before TMEM is freed
        // (a bounded wait that an abort does not cut short)
        mma_commit_warp(&bars[kBarDrain]);
        __syncwarp();
        mbar_wait(&bars[kBarDrain], 0, 1u << 24);
        __syncwarp();
    }
    else if (warp < kSoftWarps) {
        // ---------------- softmax (warps 0-3) ----------------
        // S rows (heads) live in TMEM lanes 0-15 of each quadrant (M = 64). Lane l of warp w
        // owns head 16 w + (l % 16) and the tile rows 16 (l / 16) .. + 15: the two lanes of a
        // head combine their max and sum with one shuffle.
        const bool lead = lane < 16;                    // writes the head's shared values
        const int h = warp * 16 + (lane & 15);
        const int half = lane >> 4;
        const float c2 = p.scale * kLog2e;
        const float sink2 = p.sinks[h] * kLog2e;
        uint32_t pfree_seen[kPBufs] = {};
        auto wait_pfree = [&](int buf, uint32_t phase) -> bool {   // PV of tile (kPBufs*phase + buf) done
            while (pfree_seen[buf] <= phase) {
                if (!wait_bar(&bars[kBarPFree + buf], pfree_seen[buf] & 1, abort)) return false;
                ++pfree_seen[buf];
            }
            return true;
        };
        constexpr int kHR = kTR / 2;                    // rows per lane
        uint32_t g = 0;                                 // ring entries (q slots and list tiles)
        uint32_t gt = 0;                                // list tiles (all items)
        int n = 0;
        for (int id = blockIdx.x; id < items; id += gridDim.x, ++n) {
            const Item x = item_of(p, id);
            float m2 = -INFINITY, l = 0.f;
            ++g;                                        // the ring entry that carried q (the epilogue's)
            for (int i = 0; i < x.T; ++i, ++g, ++gt) {
                const int s = g % kSlots, sb = gt & 1;
                const bool w = wait_bar(&bars[kBarFull + s], (g / kSlots) & 1, abort) &&
                               wait_bar(&bars[kBarSFull + sb], (gt >> 1) & 1, abort);
                if (!group_all(kBarSoft, kSoftWarps * 32, w)) { fail(); break; }
                fence_after_sync();
                const uint32_t mask = (uint32_t)(misc->mask[s] >> (kHR * half));
                float v[kHR];
                tmem_ld16_x2(tmem + ((uint32_t)(32 * warp) << 16) + sb * kTR, v);
                tmem_ld_wait();
                fence_before_sync();
                mbar_arrive(&bars[kBarSFree + sb]);
#pragma unroll
                for (int r = 0; r < kHR; ++r) v[r] = ((mask >> r) & 1u) ? v[r] * c2 : -INFINITY;
                float mx[kHR / 2];                          // pairwise tree: short dependency chains
#pragma unroll
                for (int r = 0; r < kHR / 2; ++r) mx[r] = fmaxf(v[2 * r], v[2 * r + 1]);
#pragma unroll
                for (int wd = kHR / 4; wd >= 1; wd >>= 1)
#pragma unroll
                    for (int r = 0; r < wd; ++r) mx[r] = fmaxf(mx[r], mx[r + wd]);
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
                for (int wd = kHR / 2; wd >= 1; wd >>= 1)
#pragma unroll
                    for (int r = 0; r < wd; ++r) pr[r] += pr[r + wd];
                const float sum = pr[0] + __shfl_xor_sync(0xffffffffu, pr[0], 16);
                // P buffer gt % kPBufs is free once PV(gt - kPBufs) has completed
                const bool wp = gt < (uint32_t)kPBufs || wait_pfree(gt % kPBufs, gt / kPBufs - 1);
                if (!group_all(kBarSoft, kSoftWarps * 32, wp)) { fail(); break; }
                l = l * alpha + sum;
                {
                    uint8_t *pbuf = smem + kOffP + (gt % kPBufs) * kPBytes;
#pragma unroll
                    for (int u = 0; u < kHR / 8; ++u)
                        *reinterpret_cast<uint4 *>(pbuf + sw128_offset(h, (half * (kHR / 8) + u) * 8)) =
                            make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
                }
                if (named_or_soft(resc)) {
                    // rescale O^T columns of the heads whose reference max moved up, once the
                    // previous tile's PV product (this item's) has landed
                    if (lead) misc->alpha[h] = alpha;
                    const bool wr = i < 1 || wait_pfree((gt - 1) % kPBufs, (gt - 1) / kPBufs);
                    if (!group_all(kBarSoft, kSoftWarps * 32, wr)) { fail(); break; }
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
                mbar_arrive(&bars[kBarPFull + (gt % kPBufs)]);
            }
            if (!ok) break;
            // the item's per-head statistics, for the epilogue warps: written once the epilogue
            // has released the previous item's O^T (and so has read its statistics)
            const bool wo = n < 1 || wait_bar(&bars[kBarOFree], (n - 1) & 1, abort);
            if (!group_all(kBarSoft, kSoftWarps * 32, wo)) { fail(); break; }
            if (lead) {
                if (p.nsplit == 1) {
                    const float M = fmaxf(m2, sink2);
                    const float wm = (m2 == -INFINITY) ? 0.f : exp2f(m2 - M);
                    misc->factor[h] = wm / (l * wm + exp2f(sink2 - M));
                } else {
                    misc->stat_m[h] = (m2 == -INFINITY) ? -INFINITY : m2 / kLog2e;
                    misc->stat_l[h] = l;
                }
            }
            mbar_arrive(&bars[kBarStat]);
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
        // ---------------- epilogue (warps 10-13): q -> TMEM, O^T -> out, beside the stream ------
        const int quad = warp & 3;                      // TMEM lanes 32 quad .. + 31 = dims
        const int et = tid - kEpiWarp0 * 32;
        // q dims [0, kQT) of an item, from the ring entry gq the producers filled, into TMEM:
        // lane l < 16 of the warp of lane quadrant c holds head 16 c + l, as the M = 64 A operand
        // wants; then the slot is free again
        auto copy_q = [&](uint32_t gq) -> bool {
            const int s = gq % kSlots;
            const bool wq = wait_bar(&bars[kBarFull + s], (gq / kSlots) & 1, abort);
            if (!group_all(kBarEpi, kEpiWarps * 32, wq)) return false;
            const uint8_t *qs = smem + kOffKV + s * kSlotBytes;
            const int hq = quad * 16 + (lane & 15);
#pragma unroll 2
            for (int c0 = 0; c0 < kQT / 2; c0 += 16) {   // 16 columns = 32 dims = 4 units
                float v[16];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4 w4 = make_uint4(0u, 0u, 0u, 0u);
                    if (lane < 16) {
                        const int qu = c0 / 4 + u;            // dims 8 qu .. + 7
                        w4 = *reinterpret_cast<const uint4 *>(qs + (qu >> 3) * kQChunk +
                                                              sw128_offset(hq, (qu & 7) * 8));
                    }
                    v[4 * u] = __uint_as_float(w4.x);
                    v[4 * u + 1] = __uint_as_float(w4.y);
                    v[4 * u + 2] = __uint_as_float(w4.z);
                    v[4 * u + 3] = __uint_as_float(w4.w);
                }
                tmem_st16(tmem + ((uint32_t)(32 * quad) << 16) + kColQ + c0, v);
            }
            tmem_st_wait();
            fence_before_sync();
            mbar_arrive(&bars[kBarQT]);
            asm volatile("bar.sync %0, %1;" ::"n"(kBarEpi), "n"(kEpiWarps * 32) : "memory");   // slot read
            if (et == 0) mbar_arrive(&bars[kBarEmpty + s]);
            return true;
        };
        uint32_t gq = 0;                                // ring entry of this item's q
        int n = 0;
        for (int id = blockIdx.x; id < items; id += gridDim.x, ++n) {
            const Item x = item_of(p, id);
            if (n == 0 && !copy_q(0)) { fail(); break; }
            // the next item's q, as soon as this item's S products no longer read the old one
            if (id + (int)gridDim.x < items) {
                const bool wf = wait_bar(&bars[kBarQFree], n & 1, abort);
                if (!group_all(kBarEpi, kEpiWarps * 32, wf)) { fail(); break; }
                fence_after_sync();
                gq += 1u + (uint32_t)x.T;
                if (!copy_q(gq)) { fail(); break; }
            }
            if (!wait_bar(&bars[kBarStat], n & 1, abort) || !wait_bar(&bars[kBarOFull], n & 1, abort)) {
                fail();
                break;
            }
            fence_after_sync();
            if (n == 0) grid_dep_wait();                // before the first output write
            const bool have_o = x.T > 0;
            if (p.nsplit == 1) {
                const int64_t out0 = (int64_t)x.row * kH * kDH;
                for (int mt = 0; mt < 4; ++mt) {
                    const int d = mt * 128 + quad * 32 + lane;
                    for (int c = 0; c < 64; c += 16) {
                        float o[16];
                        if (have_o) {
                            tmem_ld16(tmem + ((uint32_t)(32 * quad) << 16) + kColO + mt * 64 + c, o);
                            tmem_ld_wait();
                        } else {
#pragma unroll
                            for (int q = 0; q < 16; ++q) o[q] = 0.f;
                        }
                        if (p.out_bf16) {
                            __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) + out0;
#pragma unroll
                            for (int q = 0; q < 16; ++q)
                                out[(c + q) * kDH + d] = __float2bfloat16_rn(o[q] * misc->factor[c + q]);
                        } else {
                            float *out = static_cast<float *>(p.out) + out0;
#pragma unroll
                            for (int q = 0; q < 16; ++q) out[(c + q) * kDH + d] = o[q] * misc->factor[c + q];
                        }
                    }
                }
            } else {
                float *base = p.part + ((int64_t)x.row * p.nsplit + x.split) * kH * (kDH + 2);
                if (quad == 0) {
                    for (int hh = lane; hh < kH; hh += 32) {
                        base[hh * (kDH + 2)] = misc->stat_m[hh];
                        base[hh * (kDH + 2) + 1] = misc->stat_l[hh];
                    }
                }
                for (int mt = 0; mt < 4; ++mt) {
                    const int d = mt * 128 + quad * 32 + lane;
                    for (int c = 0; c < 64; c += 16) {
                        float o[16];
                        if (have_o) {
                            tmem_ld16(tmem + ((uint32_t)(32 * quad) << 16) + kColO + mt * 64 + c, o);
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
            fence_before_sync();
            mbar_arrive(&bars[kBarOFree]);
        }
    }
    if (!ok) flag(p.status, HISA_DEV_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    // this CTA is done: the next kernel may take over the SM once it exits (that kernel waits
    // for this grid before it reads what this grid writes)
    grid_dep_trigger();
    if (warp == kMmaWarp) {
        fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int attend_tc_supported(int H, int Dh, int kv_bf16) { return H == kH && Dh == kDH && kv_bf16; }

cudaError_t launch_attend_tc(const AttnParams &p, cudaStream_t s) {
    const cudaError_t attr = smem_attr_once<k_attend_tc>((int)kSmemBytes);
    if (attr != cudaSuccess) return attr;
    // persistent: one CTA per SM walks the items (query row, split)
    const int nsm = device_sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    const int64_t items = (int64_t)p.B * p.L * p.nsplit;
    if (items == 0) return cudaSuccess;
    dim3 grid((unsigned)(items < nsm ? items : nsm));
    cudaError_t e = launch_pdl(k_attend_tc, grid, dim3(kThreads), kSmemBytes, s, p.chained, p);
    if (e != cudaSuccess || p.nsplit == 1) return e;
    return launch_attend_combine(p, s);
}

}  // namespace hisa
