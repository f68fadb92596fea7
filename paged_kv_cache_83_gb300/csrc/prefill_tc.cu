// prefill_tc.cu: varlen causal prefill with a paged prefix (pa_prefill_varlen) on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Source: "nano-vLLM Part 4", section 3 (prefill: packed prompts, variable-length attention with an
// optional prefix block table); smzdm nano-vLLM deep dive, "GPU执行优化" (cu_seqlens mark sequence
// boundaries) and "模型实现细节" (prefix cache used when cu_seqlens_k > cu_seqlens_q); "mini-vLLM"
// (prompts attending causally to themselves).
//
// One CTA computes 128 query rows of one sequence for two query heads that share a kv head (a
// GQA pair), so every K/V tile it loads serves 256 rows. Shapes: head dim 128, even group sizes.
//
//   warp 0      producer: TMA loads of the two Q tiles, then of 128-key K and V tiles through the
//               block table (or from the packed k, v), 128-byte swizzled, into a 3-slot ring in
//               the order the MMAs consume them (K0, K1, V0, K2, V1, ...).
//   warps 1, 2  one MMA issuer per head (one thread each; warp 1 owns the 512 TMEM columns):
//                 S_h = Q_h K^T   as soon as the softmax has read S_h of the previous tile,
//                 O_h += P_h V    as soon as P_h is in shared memory.
//               Both operands of both MMAs come from shared memory, so S of the next tile is
//               computed while the softmax still works on the current one.
//   warps 4-7   softmax of head A, warps 8-11 softmax of head B: thread = one query row = one
//               TMEM lane. S is read once into registers (then released), masked (causal bound
//               P + row, context end), row max, P = 2^(s - m) in bf16/fp16 stored to shared
//               memory in the swizzled layout the PV MMA reads. O is rescaled in TMEM only when
//               the row max grew by more than 2^8 (the normaliser uses the same reference, so the
//               result is exact).
//   TMEM columns: S_A 0-127, S_B 128-255, O_A 256-383, O_B 384-511.
// Every wait is bounded (PA_DEVERR_TIMEOUT); on a timeout every role drains what it started
// (TMA, MMAs) before the TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "pa_internal.h"

namespace pa {

namespace {

constexpr int BM = 128, BN = 128, HD = 128;
constexpr int kThreads = 384;
constexpr int kHalf = BM * 64 * 2;  // one 128-row x 64-column half tile: 16 KB
constexpr int kTile = 2 * kHalf;    // 128 x 128 elements: 32 KB
constexpr int kRing = 3;            // K/V tile slots
constexpr uint32_t kTileDesc = kTile >> 4;  // one tile further, in descriptor address units
constexpr int OFF_QA = 0, OFF_QB = kTile, OFF_PA = 2 * kTile, OFF_PB = 3 * kTile, OFF_RING = 4 * kTile,
              OFF_BAR = OFF_RING + kRing * kTile;
// per-head barriers take index base + h (h = 0 for head A, 1 for head B)
enum {
    B_Q = 0,
    B_FULL = 1,                // + slot: a K/V tile landed (TMA transaction count)
    B_EMPTY = B_FULL + kRing,  // + slot: both heads' MMAs are done with it (two commits)
    B_S = B_EMPTY + kRing,     // + h: S = Q K^T is in TMEM
    B_F = B_S + 2,             // + h: the softmax warps have read S (4 arrivals)
    B_P = B_F + 2,             // + h: P is in shared memory (4 arrivals)
    B_O = B_P + 2,             // + h: O += P V is done, so P's buffer is free again
    B_END = B_O + 2,           // + h: every MMA of that head has completed
    B_VZ = B_END + 2,          // the last V tile's rows past the keys are zero
    NBAR
};
constexpr int kSmem = OFF_BAR + NBAR * 8 + 16 + 1024;  // + tmem base, abort flag, alignment slack
static_assert(kSmem <= 232448, "shared memory per CTA");
constexpr unsigned kFull = 0xffffffffu;

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v;  // q: [total_q, Hq, 128]; k, v: [rows, Hkv, 128]; boxes [.,1,64]
    const int32_t *cu_q, *cu_k, *block_tables;
    void *out;
    int32_t *err;
    int S, Hq, Hkv, G, max_blocks, num_blocks, causal, max_seqlen_q, box_rows;
    BlockGeom geom;
    float scale_log2;
};

__device__ __forceinline__ bool tc_warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    const bool ok = mbar_wait(bar, parity) && !*abort_flag;
    const bool all = __all_sync(kFull, ok);
    __syncwarp();
    return all;
}

__device__ __forceinline__ void tc_abort(int32_t *err, volatile int *abort_flag) {
    raise_err(err, PA_DEVERR_TIMEOUT);
    *abort_flag = 1;
}

// The K/V tiles go through the ring in the order the MMAs consume them:
//   K0, K1, V0, K2, V1, ..., K(n-1), V(n-2), V(n-1)
// (the next tile's QK is issued before the current tile's PV). Load i uses slot i % kRing.
__device__ __forceinline__ int load_index_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int load_index_v(int j, int nkv) { return j == nkv - 1 ? 2 * nkv - 1 : 2 * j + 2; }
__device__ __forceinline__ void load_item(int i, int nkv, int &j, bool &is_v) {
    if (i == 0) {
        j = 0, is_v = false;
    } else if (i & 1) {
        const int t = (i - 1) >> 1;
        if (t + 1 < nkv) j = t + 1, is_v = false;
        else j = nkv - 1, is_v = true;
    } else {
        j = (i - 2) >> 1, is_v = true;
    }
}

template <class E>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
    using T = typename E::T;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = sbase + OFF_BAR;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + NBAR * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_BAR + NBAR * 8 + 4);
    auto bar = [&](int i) { return bar0 + 8u * i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mb = gridDim.x - 1 - blockIdx.x;  // row blocks with the most keys first
    const int pair = blockIdx.y, s = blockIdx.z;
    const int hA = 2 * pair, hB = 2 * pair + 1, g = hA / p.G;

    const int q0 = p.cu_q[s], ql = p.cu_q[s + 1] - q0;
    const int k0 = p.cu_k[s], kl = p.cu_k[s + 1] - k0;
    if (ql < 0 || ql > p.max_seqlen_q) {
        if (mb == 0 && pair == 0 && tid == 0) raise_err(p.err, PA_DEVERR_LENGTH);
        return;
    }
    const int m0 = mb * BM;
    if (m0 >= ql) return;
    const int mrows = min(BM, ql - m0);
    T *out = static_cast<T *>(p.out);
    const int32_t *trow =
        p.block_tables ? p.block_tables + static_cast<size_t>(s) * p.max_blocks : nullptr;
    bool bad = kl < ql;
    if (trow && static_cast<long long>(kl) > static_cast<long long>(p.max_blocks) * p.geom.block_size)
        bad = true;
    const int P = kl - ql;
    const int n_end = bad ? 0 : (p.causal ? min(kl, P + m0 + mrows) : kl);
    const int nkv = (n_end + BN - 1) / BN;
    int table_bad = 0;
    if (!bad && trow) {
        const int nblk = p.geom.block_of(n_end - 1) + 1;
        for (int i = tid; i < nblk; i += kThreads) {
            const int id = trow[i];
            if (id < 0 || id >= p.num_blocks) table_bad = 1;
        }
    }
    table_bad = __syncthreads_or(table_bad);
    if (bad || table_bad) {  // the item is skipped: its rows are zero
        if (tid == 0) raise_err(p.err, bad ? PA_DEVERR_LENGTH : PA_DEVERR_TABLE);
        for (int i = tid; i < mrows * HD * 2; i += kThreads) {
            const int r = i / (2 * HD), h = (i / HD) & 1, d = i % HD;
            out[(static_cast<size_t>(q0 + m0 + r) * p.Hq + (h ? hB : hA)) * HD + d] = T(0.f);
        }
        return;
    }
    const int last_valid = n_end - (nkv - 1) * BN;  // keys in the last tile
    const bool zero_tail = last_valid < BN;         // its V rows past the keys must be zeroed

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) {
            uint32_t count = 1;
            if (i >= B_EMPTY && i < B_EMPTY + kRing) count = 2;
            if (i >= B_F && i < B_O) count = 4;  // B_F, B_P
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

    if (warp == 0) {
        // =================================== producer ===================================
        prefetch_tmap(&p.tm_q);
        prefetch_tmap(&p.tm_k);
        prefetch_tmap(&p.tm_v);
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(B_Q), 2 * kTile);
            for (int h = 0; h < 2; ++h)
                for (int half = 0; half < 2; ++half)
                    tma_load_3d(sbase + (h ? OFF_QB : OFF_QA) + half * kHalf, &p.tm_q, half * 64,
                                h ? hB : hA, q0 + m0, bar(B_Q));
        }
        __syncwarp();
        const int R = p.box_rows, nbox = BN / R;
        const uint32_t box_bytes = static_cast<uint32_t>(R) * 128;  // one half-row box
        const int nload = 2 * nkv;
        int issued = 0, cur_j = -1, row = -1;
        uint32_t bytes = 0;
        for (int i = 0; i < nload; ++i) {
            int j;
            bool is_v;
            load_item(i, nkv, j, is_v);
            if (j != cur_j) {
                // this lane's box (lanes 0 .. nbox-1): its first key row, or -1 past the keys
                const int n0 = j * BN;
                row = -1;
                if (lane < nbox && n0 + lane * R < n_end) {
                    const int pos = n0 + lane * R;
                    row = trow ? trow[p.geom.block_of(pos)] * p.geom.block_size + p.geom.offset_of(pos)
                               : k0 + pos;
                }
                bytes = __popc(__ballot_sync(kFull, row >= 0)) * box_bytes * 2;  // both halves
                cur_j = j;
            }
            const int slot = i % kRing;
            const uint32_t ph = (i / kRing) & 1;
            if (!tc_warp_wait(bar(B_EMPTY + slot), ph ^ 1, abort_flag)) {
                if (lane == 0) tc_abort(p.err, abort_flag);
                break;
            }
            if (lane == 0) mbar_arrive_expect_tx(bar(B_FULL + slot), bytes);
            __syncwarp();
            if (row >= 0) {
                const uint32_t dst = sbase + OFF_RING + slot * kTile + lane * R * 128;
                for (int half = 0; half < 2; ++half)
                    tma_load_3d(dst + half * kHalf, is_v ? &p.tm_v : &p.tm_k, half * 64, g, row,
                                bar(B_FULL + slot));
            }
            issued = i + 1;
        }
        // The last tile may hold rows past the keys (unwritten slots or another prompt): zero its
        // V rows there before any PV reads them (P is zero there, but 0 * NaN is not).
        if (issued == nload && zero_tail) {
            const int i = nload - 1, slot = i % kRing;
            if (tc_warp_wait(bar(B_FULL + slot), (i / kRing) & 1, abort_flag)) {
                unsigned char *vt = smem + OFF_RING + slot * kTile;
                for (int c = lane; c < (BN - last_valid) * 16; c += 32) {  // 16-byte chunks
                    const int r = last_valid + c / 16, c16 = c % 16;
                    *reinterpret_cast<uint4 *>(vt + (c16 >> 3) * kHalf + r * 128 + (c16 & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_VZ));
            } else if (lane == 0) {
                tc_abort(p.err, abort_flag);
            }
        }
        // no copy may still be in flight at exit: the last load of every slot
        if (lane == 0) {
            for (int i = issued > kRing ? issued - kRing : 0; i < issued; ++i)
                if (!mbar_wait(bar(B_FULL + i % kRing), (i / kRing) & 1)) tc_abort(p.err, abort_flag);
            if (!mbar_wait(bar(B_Q), 0)) tc_abort(p.err, abort_flag);
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
        auto qk = [&](int slot) {  // S = Q K^T: A = Q (K-major), B = K rows (K-major)
            const uint64_t kb = dk0 + slot * kTileDesc;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                tc_mma_ss(s_tm, dq + off, kb + off, IQK, kk > 0);
            }
        };
        auto pv = [&](int slot, int j) {  // O += P V: A = P (K-major), B = V rows (N-major)
            const uint64_t vb = dv0 + slot * kTileDesc;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                tc_mma_ss(o_tm, dp + off, vb + ((kk * 2048) >> 4), IPV, (j > 0 || kk > 0));
            }
        };
        bool ok = tc_warp_wait(bar(B_Q), 0, abort_flag) && tc_warp_wait(bar(B_FULL), 0, abort_flag);
        if (ok) {
            tc_fence_after();
            if (lane == 0) {
                qk(0);
                tc_commit(bar(B_S + h));
                tc_commit(bar(B_EMPTY));
            }
            __syncwarp();
        }
        for (int j = 0; ok && j < nkv; ++j) {
            // S(j+1) as soon as the softmax holds S(j) in registers
            ok = tc_warp_wait(bar(B_F + h), j & 1, abort_flag);
            if (!ok) break;
            if (j + 1 < nkv) {
                const int i = load_index_k(j + 1), slot = i % kRing;
                ok = tc_warp_wait(bar(B_FULL + slot), (i / kRing) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    qk(slot);
                    tc_commit(bar(B_S + h));
                    tc_commit(bar(B_EMPTY + slot));
                }
                __syncwarp();
            }
            const int i = load_index_v(j, nkv), slot = i % kRing;
            ok = tc_warp_wait(bar(B_P + h), j & 1, abort_flag) &&
                 tc_warp_wait(bar(B_FULL + slot), (i / kRing) & 1, abort_flag);
            if (ok && j == nkv - 1 && zero_tail) ok = tc_warp_wait(bar(B_VZ), 0, abort_flag);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
                pv(slot, j);
                tc_commit(bar(B_O + h));
                tc_commit(bar(B_EMPTY + slot));
            }
            __syncwarp();
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
        unsigned char *prow = smem + (h ? OFF_PB : OFF_PA) + r * 128;  // this row of P, half 0
        const int hq = h ? hB : hA;
        const int lim = p.causal ? min(kl, P + m0 + r + 1) : kl;  // keys this row may see
        const uint32_t s_full = bar(B_S + h), s_free = bar(B_F + h), p_full = bar(B_P + h);
        const uint32_t o_done = bar(B_O + h);
        float m_use = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            if (!(ok = tc_warp_wait(s_full, j & 1, abort_flag))) break;
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
            // P(j-1) has been consumed and O(j-1) is complete
            if (j > 0) {
                if (!(ok = tc_warp_wait(o_done, (j - 1) & 1, abort_flag))) break;
                tc_fence_after();
                if (__any_sync(kFull, need)) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(orow + c * 32, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
                        tmem_st32(orow + c * 32, ov);
                    }
                    tmem_wait_st();
                }
            }
            // P row r: 16-byte chunk q of half q / 8 sits at chunk (q % 8) ^ (r % 8) of the
            // 128-byte row (the 128-byte swizzle the MMA descriptor names)
#pragma unroll
            for (int q = 0; q < 16; ++q)
                *reinterpret_cast<uint4 *>(prow + (q >> 3) * kHalf + (((q & 7) ^ (r & 7)) << 4)) =
                    make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok) ok = tc_warp_wait(o_done, (nkv - 1) & 1, abort_flag);
        if (!ok) {
            if (lane == 0) tc_abort(p.err, abort_flag);
        } else {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            T *orow_g = out + (static_cast<size_t>(q0 + m0 + r) * p.Hq + hq) * HD;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld32(orow + c * 32, v);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2)
                    pk[e >> 1] = E::pack2(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
                if (r < mrows) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow_g + c * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
        }
    }
    // ------------------------------------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_free(tmem, 512);
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

// [rows, heads, 128] tensor, box [box_rows, 1, 64], 128-byte swizzle
bool encode_rows(CUtensorMap *m, const void *base, pa_dtype dt, int heads, long long rows, int box_rows) {
    auto fn = encode_fn_tc();
    if (!fn || rows <= 0) return false;
    cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(heads) * 256};
    cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class E>
cudaError_t launch_tc_typed(const TcParams &prm, cudaStream_t stream) {
    auto kern = prefill_tc_kernel<E>;
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    dim3 grid((prm.max_seqlen_q + BM - 1) / BM, prm.Hq / 2, prm.S);
    kern<<<grid, kThreads, kSmem, stream>>>(prm);
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
    return a.D == 128 && (a.Hq / a.Hkv) % 2 == 0 && tc_box_rows(a) >= 8 && a.total_q > 0 &&
           (a.block_tables ? true : a.total_k > 0);
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream) {
    TcParams prm{};
    const int R = tc_box_rows(a);
    const void *kb = a.block_tables ? a.k_cache : a.k;
    const void *vb = a.block_tables ? a.v_cache : a.v;
    const long long krows = a.block_tables ? static_cast<long long>(a.num_blocks) * a.block_size
                                           : static_cast<long long>(a.total_k);
    if (!encode_rows(&prm.tm_q, a.q, a.dtype, a.Hq, a.total_q, 128) ||
        !encode_rows(&prm.tm_k, kb, a.dtype, a.Hkv, krows, R) ||
        !encode_rows(&prm.tm_v, vb, a.dtype, a.Hkv, krows, R))
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
    prm.geom.block_size = a.block_size;
    prm.geom.shift = log2_if_pow2(a.block_size);
    prm.scale_log2 = a.scale * kLog2e;
    return a.dtype == PA_BF16 ? launch_tc_typed<BF16>(prm, stream) : launch_tc_typed<F16>(prm, stream);
}

}  // namespace pa
