// prefill_tc.cu: varlen causal prefill with a paged prefix (pa_prefill_varlen) on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Source: "nano-vLLM Part 4", section 3 (prefill: packed prompts, variable-length attention with an
// optional prefix block table); smzdm nano-vLLM deep dive, "GPU执行优化" (cu_seqlens mark sequence
// boundaries) and "模型实现细节" (prefix cache used when cu_seqlens_k > cu_seqlens_q); "mini-vLLM"
// (prompts attending causally to themselves).
//
// Persistent: one CTA per SM takes work items (128 query rows of one sequence for two query heads
// of one GQA group, which share every K/V tile) from a counter until none is left, so the start-up
// of one item overlaps the end of the previous one. Head dim 64 or 128 (one or two 64-column halves
// per tile); a group of G query heads is cut into ceil(G / 2) pairs, and the pair that has one head
// (odd G) computes its second head on a zero Q tile whose output is dropped. Items go out in bands
// of prompts whose K/V fits in L2 (sized from max_seqlen_k), largest first within a band.
//
//   warp 3      scheduler: claims items, reads their lengths, checks the block table, drops items
//               without rows, writes zero rows + an error bit for bad ones, and queues the rest.
//   warp 0      producer: TMA loads of each item's two Q tiles and of 128-key K and V tiles
//               through the block table (or from the packed k, v), 128-byte swizzled, into a
//               3-slot ring in the order the MMAs consume them (K0, K1, V0, K2, V1, ...).
//   warps 1, 2  one MMA issuer per head (one thread each; warp 1 owns the 512 TMEM columns):
//                 S_h = Q_h K^T   as soon as the softmax has read S_h of the previous tile,
//                 O_h += P_h V    as soon as P_h is written.
//               Q, K and V come from shared memory, and P never shares columns with S, so S of the
//               next tile (or the next item's first tile) is computed while the softmax still works
//               on the current one.
//   warps 4-7   softmax of head A, warps 8-11 softmax of head B: thread = one query row = one
//               TMEM lane. S is read once into registers (then released), masked (causal bound
//               P + row, context end), row max, P = 2^(s - m) in bf16/fp16: at head dim 128
//               stored to shared memory in the swizzled layout the PV MMA reads, at head dim 64
//               written to TMEM columns of its own (the PV MMA's A operand; the row's P leaves the
//               shared-memory store port alone, 8 % faster there). O is rescaled in TMEM only when
//               the row max grew by more than 2^8 (the normaliser uses the same reference, so the
//               result is exact). The output rows leave through the warp's rows of the P buffer
//               as whole rows (D * 2 bytes).
//   TMEM columns: S_A 0-127, S_B 128-255, O_A from 256, O_B from 384 (D columns each); at head
//   dim 64 P_A 320-383 and P_B 448-511 (16-bit pairs, one row per lane).
// Every wait is bounded (PA_DEVERR_TIMEOUT); on a timeout every role drains what it started
// (TMA, MMAs) before the TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <atomic>

#include "pa_internal.h"

namespace pa {

namespace {

constexpr int BM = 128, BN = 128;
constexpr int kThreads = 384;
constexpr int kHalf = BM * 64 * 2;  // one 128-row x 64-column half tile: 16 KB
constexpr int kPTile = BM * BN * 2; // P (128 rows x 128 keys): 32 KB, also the output stage (the
                                    // output stage alone at head dim 64, where P is in TMEM)
constexpr int kRing = 3;            // K/V tile slots
// per-head barriers take index base + h (h = 0 for head A, 1 for head B)
enum {
    B_QFULL = 0,               // the item's two Q tiles landed (TMA transaction count)
    B_QEMPTY,                  // both heads issued the item's last QK (two commits)
    B_FULL,                    // + slot: a K/V tile landed
    B_EMPTY = B_FULL + kRing,  // + slot: both heads' MMAs are done with it (two commits)
    B_S = B_EMPTY + kRing,     // + h: S = Q K^T is in TMEM
    B_F = B_S + 2,             // + h: the softmax warps have read S (4 arrivals)
    B_P = B_F + 2,             // + h: P is written (4 arrivals)
    B_O = B_P + 2,             // + h: O += P V is done, so P's buffer is free again
    B_OFREE = B_O + 2,         // + h: the item's output has been read out of TMEM (4 arrivals)
    B_END = B_OFREE + 2,       // + h: every MMA of that head has completed
    B_VZ = B_END + 2,          // the last V tile's rows past the keys are zero
    B_VZACK,                   // head B has waited for that zeroing (so head A never runs two
                               // zeroings ahead of it: a parity wait cannot tell those apart)
    B_IFULL = B_VZACK + 1,     // + k: work item k of the queue is published
    B_IEMPTY = B_IFULL + 2,    // + k: every role has read it (kItemReaders arrivals)
    NBAR = B_IEMPTY + 2
};
constexpr int kItemReaders = 11;  // producer, two MMA issuers, eight softmax warps

// One work item: 128 query rows of sequence s for the query heads ha and hb (hb < 0: the pair has
// one head) of the GQA group of kv head g. nkv == 0 marks the end of the work.
struct ItemInfo {
    int s, q0, k0, kl, m0, mrows, P, n_end, nkv, ha, hb, g;
};
// shared-memory layout for head dim HD: Q tiles, P tiles, the K/V ring, barriers, the item queue
template <int HD>
struct TcLayout {
    static constexpr int kHalves = HD / 64;    // 64-column halves per tile row
    static constexpr int kQ = BM * HD * 2;     // one Q tile
    static constexpr int kKV = BN * HD * 2;    // one K or V tile
    static constexpr uint32_t kKVDesc = kKV >> 4;  // one ring slot further, in descriptor units
    static constexpr int OFF_QA = 0, OFF_QB = kQ, OFF_PA = 2 * kQ, OFF_PB = OFF_PA + kPTile,
                         OFF_RING = OFF_PB + kPTile, OFF_BAR = OFF_RING + kRing * kKV;
    static constexpr int OFF_ITEMS = OFF_BAR + NBAR * 8;
    static constexpr int OFF_MISC = OFF_ITEMS + 2 * static_cast<int>(sizeof(ItemInfo));  // tmem base, abort flag
    static constexpr int kSmem = OFF_MISC + 16 + 1024;                                   // + alignment slack
    static_assert(kSmem <= 232448, "shared memory per CTA");
};
constexpr unsigned kFull = 0xffffffffu;

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;  // q, out: [total_q, Hq, 128]; k, v: [rows, Hkv, 128]; boxes [.,1,64]
    const int32_t *cu_q, *cu_k, *block_tables;
    void *out;
    int32_t *err;
    unsigned long long *sched;  // [0]: next work item, [1]: CTAs finished (both 0 between launches)
    long long n_items;          // bands * band * pairs * row blocks
    int S, Hq, Hkv, G, max_blocks, num_blocks, causal, max_seqlen_q, box_rows, row_blocks;
    int pairs;                  // Hkv * ceil(G / 2)
    int band;                   // prompts per band of the item order
    BlockGeom geom;
    float scale_log2;
};

__device__ __forceinline__ bool tc_warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const bool ok = mbar_wait(bar, parity) && !*abort_flag;
    const bool all = __all_sync(kFull, ok);
    __syncwarp();
    return all;
}

// 4 consecutive 32-bit TMEM columns of this thread's lane (a 4-register operand: the 16-register
// form of the same store made the softmax spill at the 168-register limit)
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tc_abort(int32_t *err, volatile int *abort_flag) {
    raise_err(err, PA_DEVERR_TIMEOUT);
    *abort_flag = 1;
}

// Persistent: one CTA per SM takes work items from a counter until none is left.
//
// The K/V tiles of all the CTA's items go through the ring in the order the MMAs consume them:
// the next tile's QK is issued before the current tile's PV, across item boundaries too:
//   K0, K1, V0, K2, V1, ..., K(n-1), V(n-2), K0', V(n-1), K1', V0', ...
// Load i uses slot i % kRing; the producer and both MMA issuers count loads the same way.
template <class E, int HD>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
    using T = typename E::T;
    using Lay = TcLayout<HD>;
    constexpr int OFF_QA = Lay::OFF_QA, OFF_QB = Lay::OFF_QB, OFF_PA = Lay::OFF_PA, OFF_PB = Lay::OFF_PB,
                  OFF_RING = Lay::OFF_RING, OFF_BAR = Lay::OFF_BAR, OFF_ITEMS = Lay::OFF_ITEMS,
                  OFF_MISC = Lay::OFF_MISC;
    constexpr int kHalves = Lay::kHalves;
    // head dim 64: P has TMEM columns of its own (S 0-255, O_A 256-319, P_A 320-383, O_B 384-447,
    // P_B 448-511), so the softmax writes it with tcgen05.st and PV reads it as the A operand
    constexpr bool kPTmem = HD == 64;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + OFF_BAR;
    ItemInfo *items = reinterpret_cast<ItemInfo *>(smem + OFF_ITEMS);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    auto bar = [&](int i) { return bar0 + 8u * i; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    T *out = static_cast<T *>(p.out);

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) {
            uint32_t count = 1;
            if (i == B_QEMPTY || (i >= B_EMPTY && i < B_EMPTY + kRing)) count = 2;
            if ((i >= B_F && i < B_O) || (i >= B_OFREE && i < B_END)) count = 4;  // B_F, B_P, B_OFREE
            if (i >= B_IEMPTY) count = kItemReaders;
            mbar_init(bar(i), count);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // every role reads the work items in the same order: item n sits in queue entry n % 2
    auto read_item = [&](int n, ItemInfo &it) -> bool {
        if (!tc_warp_wait(bar(B_IFULL + (n & 1)), (n >> 1) & 1, abort_flag)) return false;
        it = items[n & 1];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_IEMPTY + (n & 1)));
        return true;
    };

    if (warp == 3) {
        // ================================== scheduler ==================================
        // Resolves items ahead of the other roles: lengths, table check; items that cover no
        // query rows are dropped, items with bad inputs get zero rows and an error bit.
        int published = 0;
        bool ok = true;
        unsigned long long nxt = lane == 0 ? atomicAdd(p.sched, 1ull) : 0ull;
        while (ok) {
            const long long idx = static_cast<long long>(__shfl_sync(kFull, nxt, 0));
            if (idx >= p.n_items) break;
            if (lane == 0) nxt = atomicAdd(p.sched, 1ull);  // in flight while this one is resolved
            // tickets by band of p.band prompts, then rank r of a row block counted from its
            // prompt's last one (the block with the most keys), then prompt, then pair: within a
            // band large items go first and the last ones are the first row blocks of long prompts,
            // the smallest; a band's K/V stays in L2 while its row blocks run
            const long long per_rank = static_cast<long long>(p.band) * p.pairs;
            const long long per_band = per_rank * p.row_blocks;
            const int bnd = static_cast<int>(idx / per_band);
            const long long rem0 = idx % per_band;
            const int r = static_cast<int>(rem0 / per_rank);
            const int rem = static_cast<int>(rem0 % per_rank);
            const int s = bnd * p.band + rem / p.pairs;
            const int pair = rem % p.pairs;
            if (s >= p.S) continue;
            // the pair's query heads: pairs of one group's heads, the last one alone for odd G
            const int ppg = (p.G + 1) / 2;
            const int g = pair / ppg, hk = 2 * (pair % ppg);
            const int ha = g * p.G + hk, hb = hk + 1 < p.G ? ha + 1 : -1;
            const int q0 = p.cu_q[s], ql = p.cu_q[s + 1] - q0;
            const int k0 = p.cu_k[s], kl = p.cu_k[s + 1] - k0;
            if (ql < 0 || ql > p.max_seqlen_q) {
                if (r == 0 && pair == 0 && lane == 0) raise_err(p.err, PA_DEVERR_LENGTH);
                continue;
            }
            const int mb = (ql + BM - 1) / BM - 1 - r;  // row block of this rank
            if (mb < 0) continue;
            const int m0 = mb * BM;
            const int mrows = min(BM, ql - m0);
            const int32_t *trow =
                p.block_tables ? p.block_tables + static_cast<size_t>(s) * p.max_blocks : nullptr;
            bool bad = kl < ql;
            if (trow && static_cast<long long>(kl) > static_cast<long long>(p.max_blocks) * p.geom.block_size)
                bad = true;
            const int P = kl - ql;
            const int n_end = bad ? 0 : (p.causal ? min(kl, P + m0 + mrows) : kl);
            int table_bad = 0;
            if (!bad && trow) {
                const int nblk = p.geom.block_of(n_end - 1) + 1;
                for (int i = lane; i < nblk; i += 32) {
                    const int id = trow[i];
                    if (id < 0 || id >= p.num_blocks) table_bad = 1;
                }
            }
            table_bad = __any_sync(kFull, table_bad);
            if (bad || table_bad) {  // the item is skipped: its rows are zero
                if (lane == 0) raise_err(p.err, bad ? PA_DEVERR_LENGTH : PA_DEVERR_TABLE);
                for (int i = lane; i < mrows * HD * 2; i += 32) {
                    const int r = i / (2 * HD), h = (i / HD) & 1, d = i % HD;
                    const int head = h ? hb : ha;
                    if (head >= 0) out[(static_cast<size_t>(q0 + m0 + r) * p.Hq + head) * HD + d] = T(0.f);
                }
                continue;
            }
            if (!(ok = tc_warp_wait(bar(B_IEMPTY + (published & 1)), ((published >> 1) & 1) ^ 1, abort_flag)))
                break;
            if (lane == 0) {
                ItemInfo it;
                it.s = s, it.q0 = q0, it.k0 = k0, it.kl = kl, it.m0 = m0, it.mrows = mrows, it.P = P;
                it.n_end = n_end, it.nkv = (n_end + BN - 1) / BN, it.ha = ha, it.hb = hb, it.g = g;
                items[published & 1] = it;
                mbar_arrive(bar(B_IFULL + (published & 1)));  // release: the entry is visible
            }
            __syncwarp();
            ++published;
        }
        // the end marker
        if (ok && (ok = tc_warp_wait(bar(B_IEMPTY + (published & 1)), ((published >> 1) & 1) ^ 1, abort_flag))) {
            if (lane == 0) {
                ItemInfo it{};
                items[published & 1] = it;
                mbar_arrive(bar(B_IFULL + (published & 1)));
            }
            __syncwarp();
        }
        if (!ok && lane == 0) tc_abort(p.err, abort_flag);
    } else if (warp == 0) {
        // =================================== producer ===================================
        prefetch_tmap(&p.tm_q);
        prefetch_tmap(&p.tm_k);
        prefetch_tmap(&p.tm_v);
        const int R = p.box_rows, nbox = BN / R;
        const uint32_t box_bytes = static_cast<uint32_t>(R) * 128;  // one half-row box
        long long L = 0;                                            // loads issued
        int n = 0;                                                  // items taken
        bool ok = true;
        // tile j of item `it` (K or V) into the next ring slot
        auto load_tile = [&](const ItemInfo &it, int j, bool is_v) -> bool {
            const int32_t *trow =
                p.block_tables ? p.block_tables + static_cast<size_t>(it.s) * p.max_blocks : nullptr;
            const int n0 = j * BN;
            int row = -1;  // this lane's box (lanes 0 .. nbox-1): its first key row, or -1
            if (lane < nbox && n0 + lane * R < it.n_end) {
                const int pos = n0 + lane * R;
                row = trow ? trow[p.geom.block_of(pos)] * p.geom.block_size + p.geom.offset_of(pos)
                           : it.k0 + pos;
            }
            const uint32_t bytes = __popc(__ballot_sync(kFull, row >= 0)) * box_bytes * kHalves;
            const int slot = static_cast<int>(L % kRing);
            if (!tc_warp_wait(bar(B_EMPTY + slot), static_cast<uint32_t>((L / kRing) & 1) ^ 1, abort_flag))
                return false;
            if (lane == 0) mbar_arrive_expect_tx(bar(B_FULL + slot), bytes);
            __syncwarp();
            if (row >= 0) {
                const uint32_t dst = sbase + OFF_RING + slot * Lay::kKV + lane * R * 128;
                for (int half = 0; half < kHalves; ++half)
                    tma_load_3d(dst + half * kHalf, is_v ? &p.tm_v : &p.tm_k, half * 64, it.g, row,
                                bar(B_FULL + slot));
            }
            ++L;
            return true;
        };
        ItemInfo prev{}, cur{};
        bool have_prev = false;
        while (ok) {
            if (!(ok = read_item(n, cur)) || cur.nkv == 0) break;
            ok = load_tile(cur, 0, false);
            if (ok && have_prev) ok = load_tile(prev, prev.nkv - 1, true);
            // this item's Q once both heads issued the previous item's last QK
            if (ok && n > 0) ok = tc_warp_wait(bar(B_QEMPTY), (n - 1) & 1, abort_flag);
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(B_QFULL), 2 * Lay::kQ);
                // a missing second head reads past the last head: the tile is zero-filled
                for (int h = 0; h < 2; ++h)
                    for (int half = 0; half < kHalves; ++half)
                        tma_load_3d(sbase + (h ? OFF_QB : OFF_QA) + half * kHalf, &p.tm_q, half * 64,
                                    h ? (cur.hb >= 0 ? cur.hb : p.Hq) : cur.ha, cur.q0 + cur.m0,
                                    bar(B_QFULL));
            }
            __syncwarp();
            for (int j = 1; ok && j < cur.nkv; ++j)
                ok = load_tile(cur, j, false) && load_tile(cur, j - 1, true);
            prev = cur;
            have_prev = true;
            ++n;
        }
        if (ok && have_prev) ok = load_tile(prev, prev.nkv - 1, true);
        if (!ok && lane == 0) tc_abort(p.err, abort_flag);
        // no copy may still be in flight at exit: the last load of every slot, the last Q
        if (lane == 0) {
            for (long long i = L > kRing ? L - kRing : 0; i < L; ++i)
                if (!mbar_wait(bar(B_FULL + static_cast<int>(i % kRing)), static_cast<uint32_t>((i / kRing) & 1)))
                    tc_abort(p.err, abort_flag);
            if (n > 0 && !mbar_wait(bar(B_QFULL), (n - 1) & 1)) tc_abort(p.err, abort_flag);
        }
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        // ============================ MMA issuer of one head =============================
        const int h = warp - 1;
        constexpr uint32_t IQK = idesc_f16(BM, BN, E::kIsBf16, false);
        constexpr uint32_t IPV = idesc_f16(BM, HD, E::kIsBf16, true);
        // Descriptors are built once; each MMA adds a compile-time offset (in 16-byte units) to a
        // base. Rebuilding a descriptor from its address before every MMA halves the issue rate.
        const uint64_t dq = smem_desc_sw128(sbase + (h ? OFF_QB : OFF_QA), 16, 1024);
        const uint64_t dp = smem_desc_sw128(sbase + (h ? OFF_PB : OFF_PA), 16, 1024);
        const uint64_t dk0 = smem_desc_sw128(sbase + OFF_RING, 16, 1024);
        const uint64_t dv0 = smem_desc_sw128(sbase + OFF_RING, kHalf, 1024);
        const uint32_t s_tm = tmem + (h ? 128 : 0), o_tm = tmem + 256 + (h ? 128 : 0);
        const uint32_t p_tm = tmem + 256 + HD + (h ? 128 : 0);  // P in TMEM (head dim 64)
        auto qk = [&](int slot) {  // S = Q K^T: A = Q (K-major), B = K rows (K-major)
            const uint64_t kb = dk0 + slot * Lay::kKVDesc;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                tc_mma_ss(s_tm, dq + off, kb + off, IQK, kk > 0);
            }
        };
        auto pv = [&](int slot, bool acc) {  // O += P V: A = P (K-major), B = V rows (N-major)
            const uint64_t vb = dv0 + slot * Lay::kKVDesc;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                if constexpr (kPTmem)
                    tc_mma_ts(o_tm, p_tm + kk * 8, vb + ((kk * 2048) >> 4), IPV, (acc || kk > 0));
                else
                    tc_mma_ss(o_tm, dp + off, vb + ((kk * 2048) >> 4), IPV, (acc || kk > 0));
            }
        };
        long long ci = 0;  // loads consumed
        auto next_load = [&](int &slot) -> bool {
            slot = static_cast<int>(ci % kRing);
            const bool r = tc_warp_wait(bar(B_FULL + slot), static_cast<uint32_t>((ci / kRing) & 1), abort_flag);
            ++ci;
            return r;
        };
        // QK of the first tile of the item read as number `n`
        auto first_qk = [&](const ItemInfo &it, int n) -> bool {
            int slot;
            if (!tc_warp_wait(bar(B_QFULL), n & 1, abort_flag) || !next_load(slot)) return false;
            tc_fence_after();
            if (lane == 0) {
                qk(slot);
                tc_commit(bar(B_S + h));
                tc_commit(bar(B_EMPTY + slot));
                if (it.nkv == 1) tc_commit(bar(B_QEMPTY));
            }
            __syncwarp();
            return true;
        };
        int n = 0, zt = 0;  // items read, zero-tail items finished
        long long t = 0;    // tiles of this head so far (global over the CTA's items)
        ItemInfo cur{}, nxt{};
        bool ok = read_item(0, cur);
        const bool active = ok && cur.nkv > 0;  // the CTA got at least one item
        n = 1;
        int item_no = 0;  // index of `cur` among the CTA's items
        if (active) ok = first_qk(cur, 0);
        int j = 0;
        while (ok && active) {
            // S(t + 1) as soon as the softmax holds S(t) in registers
            if (!(ok = tc_warp_wait(bar(B_F + h), static_cast<uint32_t>(t & 1), abort_flag))) break;
            bool has_next = true;
            if (j + 1 < cur.nkv) {
                int slot;
                if (!(ok = next_load(slot))) break;
                tc_fence_after();
                if (lane == 0) {
                    qk(slot);
                    tc_commit(bar(B_S + h));
                    tc_commit(bar(B_EMPTY + slot));
                    if (j + 1 == cur.nkv - 1) tc_commit(bar(B_QEMPTY));
                }
                __syncwarp();
            } else {
                if (!(ok = read_item(n, nxt))) break;
                ++n;
                has_next = nxt.nkv > 0;
                if (has_next && !(ok = first_qk(nxt, item_no + 1))) break;
            }
            // PV of tile j of the current item
            int slot;
            if (!(ok = tc_warp_wait(bar(B_P + h), static_cast<uint32_t>(t & 1), abort_flag) && next_load(slot)))
                break;
            const int last_valid = cur.n_end - (cur.nkv - 1) * BN;
            if (j == cur.nkv - 1 && last_valid < BN) {
                // The last tile may hold rows past the keys (unwritten slots or another prompt):
                // zero them before any PV reads them (P is zero there, but 0 * NaN is not).
                if (h == 0) {
                    if (zt > 0 && !(ok = tc_warp_wait(bar(B_VZACK), static_cast<uint32_t>((zt - 1) & 1), abort_flag)))
                        break;
                    unsigned char *vt = smem + OFF_RING + slot * Lay::kKV;
                    for (int c = lane; c < (BN - last_valid) * (HD / 8); c += 32) {  // 16-byte chunks
                        const int r = last_valid + c / (HD / 8), c16 = c % (HD / 8);
                        *reinterpret_cast<uint4 *>(vt + (c16 >> 3) * kHalf + r * 128 + (c16 & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_VZ));
                } else {
                    if (!(ok = tc_warp_wait(bar(B_VZ), zt & 1, abort_flag))) break;
                    if (lane == 0) mbar_arrive(bar(B_VZACK));
                }
                ++zt;
            }
            // the previous item's output must be out of TMEM before its O is overwritten
            if (j == 0 && item_no > 0 && !(ok = tc_warp_wait(bar(B_OFREE + h), (item_no - 1) & 1, abort_flag)))
                break;
            tc_fence_after();
            if (lane == 0) {
                pv(slot, j > 0);
                tc_commit(bar(B_O + h));
                tc_commit(bar(B_EMPTY + slot));
            }
            __syncwarp();
            ++t;
            if (++j == cur.nkv) {
                if (!has_next) break;
                cur = nxt;
                j = 0;
                ++item_no;
            }
        }
        if (!ok && lane == 0) tc_abort(p.err, abort_flag);
        // every MMA this thread issued has finished before the TMEM can be freed
        if (lane == 0) {
            tc_commit(bar(B_END + h));
            if (!mbar_wait(bar(B_END + h), 0)) tc_abort(p.err, abort_flag);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // =================================== softmax ===================================
        const int h = warp >= 8 ? 1 : 0;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // row of the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t srow = tmem + lane_off + (h ? 128 : 0);
        const uint32_t orow = tmem + lane_off + 256 + (h ? 128 : 0);
        // this row of P (half 0) in shared memory; with P in TMEM it serves the output stage only
        auto prow_of = [&]() { return smem + (h ? OFF_PB : OFF_PA) + r * 128; };
        const uint32_t s_full = bar(B_S + h), s_free = bar(B_F + h), p_full = bar(B_P + h);
        const uint32_t o_done = bar(B_O + h), o_free = bar(B_OFREE + h);
        long long t = 0;  // tiles of this head so far
        bool ok = true;
        ItemInfo it{};
        for (int n = 0; ok; ++n) {
            if (!(ok = read_item(n, it)) || it.nkv == 0) break;
            const int lim = p.causal ? min(it.kl, it.P + it.m0 + r + 1) : it.kl;  // keys this row may see
            float m_use = -INFINITY, l = 0.f;
            for (int j = 0; j < it.nkv; ++j, ++t) {
                if (!(ok = tc_warp_wait(s_full, static_cast<uint32_t>(t & 1), abort_flag))) break;
                tc_fence_after();
                uint32_t sv[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t(&chunk)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c);
                    tmem_ld32(srow + c * 32, chunk);
                }
                tmem_wait_ld();
                // S may be overwritten by the next tile's QK from here on
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free);
                const int n0 = j * BN;
                if (n0 + BN > lim) {
#pragma unroll
                    for (int e = 0; e < 128; ++e)
                        if (n0 + e >= lim) sv[e] = 0xff800000u;  // -inf
                }
                // row maximum of the raw scores (the scale is positive, so it is applied once)
                float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < 128; ++e) mq[e & 3] = fmaxf(mq[e & 3], __uint_as_float(sv[e]));
                const float mraw = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                const float mx = mraw == -INFINITY ? -INFINITY : mraw * p.scale_log2;
                // move the reference max only when it grew by more than 2^8 (or was unset)
                const bool need = mx > m_use + 8.f;
                const float f = need ? fast_exp2(m_use - mx) : 1.f;  // 0 while m_use is unset
                if (need) m_use = mx;
                const float mu = m_use == -INFINITY ? 0.f : m_use;
                // p = 2^(s * scale - m) on fp32 pairs, packed to 16-bit pairs
                const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(-mu, -mu);
                uint64_t l2 = f2_pack(0.f, 0.f);
                uint32_t pk[64];
#pragma unroll
                for (int e = 0; e < 128; e += 2) {
                    const uint64_t x2 = f2_fma(u2_pack(sv[e], sv[e + 1]), sc2, nm2);
                    const float p0 = fast_exp2(f2_lo(x2)), p1 = fast_exp2(f2_hi(x2));
                    l2 = f2_add(l2, f2_pack(p0, p1));
                    pk[e >> 1] = E::pack2(p0, p1);
                }
                l = l * f + (f2_lo(l2) + f2_hi(l2));
                // the previous tile's PV has consumed P and completed O
                if (t > 0) {
                    if (!(ok = tc_warp_wait(o_done, static_cast<uint32_t>((t - 1) & 1), abort_flag))) break;
                    tc_fence_after();
                }
                if constexpr (kPTmem) {
                    // P in its own TMEM columns (the A operand of the PV MMA)
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        tmem_st4(orow + HD + 4 * c, pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                    tmem_wait_st();
                } else {
                    // P row r: 16-byte chunk q of half q / 8 sits at chunk (q % 8) ^ (r % 8) of the
                    // 128-byte row (the 128-byte swizzle the MMA descriptor names). The warp's rows
                    // may still be the source of the previous item's output store.
                    if (j == 0) {
                        if (lane == 0) bulk_wait_read();
                        __syncwarp();
                    }
                    unsigned char *prow = prow_of();
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        *reinterpret_cast<uint4 *>(prow + (q >> 3) * kHalf + (((q & 7) ^ (r & 7)) << 4)) =
                            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
                // O(t - 1) is complete: rescale it before this tile's PV adds to it
                if (j > 0 && __any_sync(kFull, need)) {
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(orow + c * 32, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
                        tmem_st32(orow + c * 32, ov);
                    }
                    tmem_wait_st();
                }
                if constexpr (!kPTmem) fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
            }
            if (ok) ok = tc_warp_wait(o_done, static_cast<uint32_t>((t - 1) & 1), abort_flag);
            if (!ok) break;
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint32_t ov[HD / 2];  // the output row, packed
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(orow + c * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2)
                    ov[c * 16 + (e >> 1)] = E::pack2(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
            }
            // O is out of TMEM: the next item's first PV may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            // The warp's 32 rows go out through their own rows of the P buffer (swizzled like P):
            // two TMA stores when all 32 rows belong to the item, else row-wide 16-byte stores.
            // With P in TMEM nothing else has waited for the previous item's store to read them.
            if constexpr (kPTmem) {
                if (lane == 0) bulk_wait_read();
                __syncwarp();
            }
            unsigned char *prow = prow_of();
#pragma unroll
            for (int c = 0; c < HD / 8; ++c)
                *reinterpret_cast<uint4 *>(prow + (c >> 3) * kHalf + (((c & 7) ^ (r & 7)) << 4)) =
                    make_uint4(ov[4 * c], ov[4 * c + 1], ov[4 * c + 2], ov[4 * c + 3]);
            const unsigned char *pw = smem + (h ? OFF_PB : OFF_PA);
            const int head = h ? it.hb : it.ha;  // < 0: this pair has no second head
            if (head < 0) {
                __syncwarp();
            } else if (quarter * 32 + 32 <= it.mrows) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int row0 = it.q0 + it.m0 + quarter * 32;
                    for (int half = 0; half < kHalves; ++half)
                        tma_store_3d(&p.tm_o, half * 64, head, row0,
                                     smem_addr(pw + half * kHalf + quarter * 32 * 128));
                    bulk_commit();
                }
            } else {
                __syncwarp();
#pragma unroll 4
                for (int i = 0; i < HD / 8; ++i) {  // 32 rows x HD / 8 chunks of 16 bytes
                    const int k = i * 32 + lane, rr = quarter * 32 + k / (HD / 8), c = k % (HD / 8);
                    const uint4 u = *reinterpret_cast<const uint4 *>(pw + (c >> 3) * kHalf + rr * 128 +
                                                                     (((c & 7) ^ (rr & 7)) << 4));
                    if (rr < it.mrows)
                        *reinterpret_cast<uint4 *>(out + (static_cast<size_t>(it.q0 + it.m0 + rr) * p.Hq +
                                                          head) * HD + c * 8) = u;
                }
            }
            __syncwarp();  // the rows are read before the next tile's P overwrites them
        }
        if (lane == 0) bulk_wait_all();  // the output stores are complete before the CTA exits
        __syncwarp();
        if (!ok && lane == 0) tc_abort(p.err, abort_flag);
    }
    // ------------------------------------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_free(tmem, 512);
    }
    // the last CTA to finish resets the work counter for the next launch
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1ull) == gridDim.x - 1) {
            p.sched[0] = 0;
            p.sched[1] = 0;
            __threadfence();
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_tc() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// [rows, heads, hd] tensor, box [box_rows, 1, 64], 128-byte swizzle
bool encode_rows(CUtensorMap *m, const void *base, pa_dtype dt, int heads, int hd, long long rows, int box_rows) {
    auto fn = encode_fn_tc();
    if (!fn || rows <= 0) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(hd) * 2, static_cast<cuuint64_t>(heads) * hd * 2};
    cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Work counters of the persistent launches: [slot][0] the next work item, [slot][1] CTAs done.
// Each launch takes the next slot, so launches in flight on different streams do not share one,
// and its last CTA resets the pair to zero for the launch that takes the slot next.
constexpr int kSchedSlots = 64;
__device__ unsigned long long g_sched[kSchedSlots][2];

unsigned long long *sched_slot() {
    static std::atomic<unsigned> next{0};
    static unsigned long long *base[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!base[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_sched) != cudaSuccess) return nullptr;
        base[dev] = static_cast<unsigned long long *>(ptr);
    }
    return base[dev] + 2 * (next.fetch_add(1u) % kSchedSlots);
}

template <class E, int HD>
cudaError_t launch_tc_typed(const TcParams &prm, cudaStream_t stream) {
    auto kern = prefill_tc_kernel<E, HD>;
    constexpr int kSmem = TcLayout<HD>::kSmem;
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    const long long ctas = prm.n_items < device_sm_count() ? prm.n_items : device_sm_count();
    kern<<<static_cast<unsigned>(ctas > 0 ? ctas : 1), kThreads, kSmem, stream>>>(prm);
    return cudaGetLastError();
}

}  // namespace

// Rows per K/V box for the tensor-core path: 128 for packed keys; for a pool, the largest power of
// two dividing the block size, capped at 128. The path needs at least 8 (a whole 1 KB swizzle atom).
int tc_box_rows(const PrefillArgs &a) {
    if (!a.block_tables) return 128;
    int R = 1;
    while (R < 128 && a.block_size % (2 * R) == 0) R *= 2;
    return R;
}

bool tc_prefill_supported(const PrefillArgs &a) {
    // the output rows leave through TMA stores and 16-byte stores
    const bool out_aligned = (reinterpret_cast<uintptr_t>(a.out) & 15u) == 0;
    return (a.D == 64 || a.D == 128) && tc_box_rows(a) >= 8 && a.total_q > 0 &&
           (a.block_tables ? true : a.total_k > 0) && out_aligned;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream) {
    TcParams prm{};
    const int R = tc_box_rows(a);
    const void *kb = a.block_tables ? a.k_cache : a.k;
    const void *vb = a.block_tables ? a.v_cache : a.v;
    const long long krows = a.block_tables ? static_cast<long long>(a.num_blocks) * a.block_size
                                           : static_cast<long long>(a.total_k);
    if (!encode_rows(&prm.tm_q, a.q, a.dtype, a.Hq, a.D, a.total_q, 128) ||
        !encode_rows(&prm.tm_k, kb, a.dtype, a.Hkv, a.D, krows, R) ||
        !encode_rows(&prm.tm_v, vb, a.dtype, a.Hkv, a.D, krows, R) ||
        !encode_rows(&prm.tm_o, a.out, a.dtype, a.Hq, a.D, a.total_q, 32))
        return cudaErrorInvalidValue;
    prm.cu_q = a.cu_q;
    prm.cu_k = a.cu_k;
    prm.block_tables = a.block_tables;
    prm.out = a.out;
    prm.err = a.err;
    prm.S = a.S;
    prm.Hq = a.Hq;
    prm.Hkv = a.Hkv;
    prm.G = a.Hq / a.Hkv;
    prm.max_blocks = a.max_blocks;
    prm.num_blocks = a.num_blocks;
    prm.causal = a.causal;
    prm.max_seqlen_q = a.max_seqlen_q;
    prm.box_rows = R;
    prm.row_blocks = (a.max_seqlen_q + BM - 1) / BM;
    prm.pairs = a.Hkv * ((prm.G + 1) / 2);
    // prompts per band: the K/V of a band (at most max_seqlen_k keys a prompt) within 64 MB of L2
    const double kv_bytes = static_cast<double>(a.max_seqlen_k > 0 ? a.max_seqlen_k : 1) * a.Hkv * a.D * 4;
    prm.band = static_cast<int>(std::max(1.0, std::min(static_cast<double>(a.S), 64.0 * (1 << 20) / kv_bytes)));
    const long long bands = (a.S + prm.band - 1) / prm.band;
    prm.n_items = bands * prm.band * prm.pairs * prm.row_blocks;
    prm.sched = sched_slot();
    if (!prm.sched) return cudaErrorInvalidDevice;
    prm.geom.block_size = a.block_size;
    prm.geom.shift = log2_if_pow2(a.block_size);
    prm.scale_log2 = a.scale * kLog2e;
    if (a.D == 64)
        return a.dtype == PA_BF16 ? launch_tc_typed<BF16, 64>(prm, stream) : launch_tc_typed<F16, 64>(prm, stream);
    return a.dtype == PA_BF16 ? launch_tc_typed<BF16, 128>(prm, stream) : launch_tc_typed<F16, 128>(prm, stream);
}

}  // namespace pa
