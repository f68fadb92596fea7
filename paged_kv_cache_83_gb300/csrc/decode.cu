// decode.cu: paged grouped-query decode attention (pa_decode): split-K kernel + merge kernel.
//
// Source: "nano-vLLM Part 4", section 3 (decode: one already-sampled token per sequence,
// attention over its cached history through a block table); "mini-vLLM" (one token per
// sequence attending to that sequence's cached keys and values, grouped-query attention).
//
// Design (GB300): decode reads every cached K/V row once and does ~G multiply-adds per byte,
// far below the HBM ridge, so the kernel is built to keep HBM busy, not to reach tensor cores.
//  * Work item = (sequence, kv head, chunk of `chunk` positions). One CTA computes the whole
//    GQA group (G query heads) of its kv head, so each K/V byte is read from HBM once.
//  * 64-position tiles of K and V are staged into shared memory with 16-byte cp.async copies,
//    STAGES deep; each copy's address goes through the block table (kept in shared memory for
//    the chunk). Rows past the context or in an invalid block are zero-filled and masked.
//  * QK: LPP lanes share one position, each holding E query elements per head in registers
//    (pre-multiplied by scale*log2 e); partial dots meet in a butterfly of shuffles. The K tile
//    is stored with a 16-byte-chunk XOR swizzle so these reads are free of bank conflicts.
//  * Softmax is online per warp in base 2; PV: each lane owns 8 output columns of a row
//    group and accumulates p * V from the unswizzled V tile.
//  * At the end the 4 warps' (max, sum, O) are combined in shared memory. A single-split
//    sequence writes its output directly; otherwise the normalised partial and its (max, sum)
//    go to the workspace and decode_merge_kernel combines the splits.
#include <math.h>

#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kTN = 64;             // positions per tile
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kWPos = kTN / kWarps;  // positions per warp per tile
constexpr unsigned kFull = 0xffffffffu;

template <int D, int G>
struct Shape {
    static constexpr int NCH = D / 8;  // 16-byte chunks per row
    static constexpr int E_RAW = G == 1 ? 64 : G == 2 ? 32 : G <= 4 ? 16 : 8;
    static constexpr int E = E_RAW < D / 2 ? E_RAW : D / 2;  // QK elements per lane
    static constexpr int LPP = D / E;                         // lanes per position in QK
    static constexpr int PPP = 32 / LPP;                      // positions per QK pass
    static constexpr int PASSES = kWPos / PPP;
    static constexpr int CPL = E / 8;                         // 16-byte chunks per lane in QK
    static constexpr int LPR = NCH;                           // PV lanes per row (8 columns each)
    static constexpr int RPI = 32 / LPR;                      // PV rows per warp instruction
    static constexpr int STAGES = D == 128 ? 3 : 4;
    static constexpr int TILE_BYTES = kTN * D * 2;
    static constexpr int TILES_BYTES = 2 * STAGES * TILE_BYTES;
    static constexpr int LOADS = kTN * NCH / kThreads;         // 16-byte copies per thread per tile
    // XOR applied to the chunk index of K row `row`: positions that share a bank phase in
    // QK get disjoint bank groups
    static __device__ __forceinline__ int swz(int row) {
        return LPP < 8 ? (row % (8 / LPP)) * LPP : 0;
    }
    static_assert(PASSES >= 1 && PPP * PASSES == kWPos, "QK mapping");
    static_assert(LOADS * kThreads == kTN * NCH, "loader mapping");
};

struct DecodeParams {
    const void *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    void *out;
    float *ws_o;   // [B, Hq, max_splits, D]
    float *ws_ml;  // [B, Hq, max_splits, 2]  (max in log2 units, sum)
    int32_t *err;
    int B, Hq, Hkv, max_blocks, num_blocks, chunk, max_splits, tbl_cap;
    BlockGeom geom;
    float scale_log2;
};

template <int D, int G>
constexpr int smem_bytes_for(int tbl_cap) {
    return Shape<D, G>::TILES_BYTES + tbl_cap * 4 + 2 * kWarps * G * kWPos * 4;
}

template <int D, int G, class E>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const DecodeParams p) {
    using S = Shape<D, G>;
    using T = typename E::T;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ks = smem;
    unsigned char *vs = smem + S::STAGES * S::TILE_BYTES;
    int *tbl = reinterpret_cast<int *>(smem + S::TILES_BYTES);
    float *sbuf = reinterpret_cast<float *>(tbl + p.tbl_cap);  // [warps][G][16] raw scores
    float *pbuf = sbuf + kWarps * G * kWPos;                    // [warps][G][16] probabilities

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hq0 = g * G;

    int n = p.context_lens[b];
    const long long cap = static_cast<long long>(p.max_blocks) * p.geom.block_size;
    if (n < 0 || n > cap) {
        if (split == 0 && tid == 0) raise_err(p.err, PA_DEVERR_LENGTH);
        n = 0;
    }
    if (n == 0) {  // no keys: zero output, written by the first split only
        if (split == 0) {
            T *o = static_cast<T *>(p.out) + (static_cast<size_t>(b) * p.Hq + hq0) * D;
            for (int i = tid; i < G * D; i += kThreads) o[i] = T(0.f);
        }
        return;
    }
    const int start = split * p.chunk;
    if (start >= n) return;
    const int end = min(start + p.chunk, n);
    const int nsplit = (n + p.chunk - 1) / p.chunk;
    const int ntiles = (end - start + kTN - 1) / kTN;

    // this chunk's block-table entries, checked once
    const int b0 = p.geom.block_of(start);
    const int nb = p.geom.block_of(end - 1) - b0 + 1;
    const int32_t *trow = p.block_tables + static_cast<size_t>(b) * p.max_blocks;
    int bad = 0;
    for (int i = tid; i < nb; i += kThreads) {
        int id = trow[b0 + i];
        if (id < 0 || id >= p.num_blocks) {
            bad = 1;
            id = -1;
        }
        tbl[i] = id;
    }
    bad = __syncthreads_or(bad);
    if (bad && tid == 0) raise_err(p.err, PA_DEVERR_TABLE);

    // query rows of the group, scaled into log2 units
    const int r = lane % S::LPP;
    float qf[G][S::CPL][8];
    {
        const T *qb = static_cast<const T *>(p.q) + (static_cast<size_t>(b) * p.Hq + hq0) * D;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int c = 0; c < S::CPL; ++c) {
                const uint4 u = *reinterpret_cast<const uint4 *>(qb + h * D + (c * S::LPP + r) * 8);
                unpack8<E>(u, qf[h][c]);
#pragma unroll
                for (int e = 0; e < 8; ++e) qf[h][c][e] *= p.scale_log2;
            }
    }

    const T *kcache = static_cast<const T *>(p.k_cache);
    const T *vcache = static_cast<const T *>(p.v_cache);
    auto load_tile = [&](int stage, int t) {
        const int t0 = start + t * kTN;
        const uint32_t kbase = smem_addr(ks + stage * S::TILE_BYTES);
        const uint32_t vbase = smem_addr(vs + stage * S::TILE_BYTES);
#pragma unroll
        for (int i = 0; i < S::LOADS; ++i) {
            const int id = tid + i * kThreads;
            const int row = id / S::NCH, ch = id % S::NCH;
            const int pos = t0 + row;
            int blk = -1;
            if (pos < end) blk = tbl[p.geom.block_of(pos) - b0];
            const bool ok = blk >= 0;
            const size_t slot =
                ok ? static_cast<size_t>(blk) * p.geom.block_size + p.geom.offset_of(pos) : 0;
            const size_t off = (slot * p.Hkv + g) * D + ch * 8;
            cp_async16(kbase + row * D * 2 + ((ch ^ S::swz(row)) * 16), kcache + off, ok ? 16 : 0);
            cp_async16(vbase + row * D * 2 + ch * 16, vcache + off, ok ? 16 : 0);
        }
    };

    float m_run[G], l_part[G], acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_run[h] = -INFINITY;
        l_part[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
    }

#pragma unroll
    for (int s = 0; s < S::STAGES - 1; ++s) {
        if (s < ntiles) load_tile(s, s);
        cp_async_commit();
    }

    const int rg = lane / S::LPR, cc = lane % S::LPR;
    float *sb = sbuf + warp * G * kWPos;
    float *pb = pbuf + warp * G * kWPos;

    for (int t = 0; t < ntiles; ++t) {
        cp_async_wait<S::STAGES - 2>();
        __syncthreads();
        {
            const int nt = t + S::STAGES - 1;
            if (nt < ntiles) load_tile(nt % S::STAGES, nt);
            cp_async_commit();
        }
        const int stage = t % S::STAGES;
        const int t0 = start + t * kTN;
        const uint32_t kb = smem_addr(ks + stage * S::TILE_BYTES);
        const uint32_t vb = smem_addr(vs + stage * S::TILE_BYTES);

        // scores of this warp's 16 positions
#pragma unroll
        for (int pass = 0; pass < S::PASSES; ++pass) {
            const int pl = pass * S::PPP + lane / S::LPP;
            const int row = warp * kWPos + pl;
            float dot[G];
#pragma unroll
            for (int h = 0; h < G; ++h) dot[h] = 0.f;
#pragma unroll
            for (int c = 0; c < S::CPL; ++c) {
                const int j = c * S::LPP + r;
                const uint4 u = lds128(kb + row * D * 2 + ((j ^ S::swz(row)) * 16));
                float kf[8];
                unpack8<E>(u, kf);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < 8; ++e) dot[h] = fmaf(qf[h][c][e], kf[e], dot[h]);
            }
#pragma unroll
            for (int off = S::LPP / 2; off >= 1; off >>= 1)
#pragma unroll
                for (int h = 0; h < G; ++h) dot[h] += __shfl_xor_sync(kFull, dot[h], off);
            const int pos = t0 + row;
            bool valid = pos < end;
            if (bad && valid) valid = tbl[p.geom.block_of(pos) - b0] >= 0;
            if (r == 0)
#pragma unroll
                for (int h = 0; h < G; ++h) sb[h * kWPos + pl] = valid ? dot[h] : -INFINITY;
        }
        __syncwarp();

        // online softmax; lanes 16..31 mirror lanes 0..15 so every lane keeps the running max
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float s = sb[h * kWPos + (lane & 15)];
            float mt = s;
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, off));
            const float m_new = fmaxf(m_run[h], mt);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = fast_exp2(m_run[h] - m_use);
            m_run[h] = m_new;
            const float pr = fast_exp2(s - m_use);
            l_part[h] = l_part[h] * alpha + (lane < 16 ? pr : 0.f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] *= alpha;
            if (lane < 16) pb[h * kWPos + lane] = pr;
        }
        __syncwarp();

        // O += P V
#pragma unroll
        for (int it = 0; it < kWPos / S::RPI; ++it) {
            const int pl = it * S::RPI + rg;
            const int row = warp * kWPos + pl;
            const uint4 u = lds128(vb + row * D * 2 + cc * 16);
            float vf[8];
            unpack8<E>(u, vf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float ph = pb[h * kWPos + pl];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(ph, vf[e], acc[h][e]);
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    // warp totals: sum l over lanes, sum O over row groups
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) l_part[h] += __shfl_xor_sync(kFull, l_part[h], off);
#pragma unroll
        for (int off = S::LPR; off < 32; off <<= 1)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(kFull, acc[h][e], off);
    }
    float *red_o = reinterpret_cast<float *>(ks);   // [warps][G][D]
    float *red_ml = red_o + kWarps * G * D;         // [warps][G][2]
    if (rg == 0)
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float4 *dst = reinterpret_cast<float4 *>(red_o + (warp * G + h) * D + cc * 8);
            dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
            dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
        }
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < G; ++h) {
            red_ml[(warp * G + h) * 2] = m_run[h];
            red_ml[(warp * G + h) * 2 + 1] = l_part[h];
        }
    __syncthreads();

    for (int idx = tid; idx < G * D; idx += kThreads) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_ml[(w * G + h) * 2]);
        const float mu = M == -INFINITY ? 0.f : M;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float sc = fast_exp2(red_ml[(w * G + h) * 2] - mu);
            L = fmaf(red_ml[(w * G + h) * 2 + 1], sc, L);
            O = fmaf(red_o[(w * G + h) * D + d], sc, O);
        }
        const float o = L > 0.f ? O / L : 0.f;
        const size_t bh = static_cast<size_t>(b) * p.Hq + hq0 + h;
        if (nsplit == 1) {
            static_cast<T *>(p.out)[bh * D + d] = T(o);
        } else {
            p.ws_o[(bh * p.max_splits + split) * D + d] = o;
            if (d == 0) {
                p.ws_ml[(bh * p.max_splits + split) * 2] = M;
                p.ws_ml[(bh * p.max_splits + split) * 2 + 1] = L;
            }
        }
    }
}

// One warp per (sequence, query head): combine the splits' normalised partials.
template <int D, class E>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p) {
    using T = typename E::T;
    constexpr int PER = D / 32;  // output columns per lane
    const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (wid >= p.B * p.Hq) return;
    const int b = wid / p.Hq;
    const int n = p.context_lens[b];
    const long long cap = static_cast<long long>(p.max_blocks) * p.geom.block_size;
    if (n <= 0 || n > cap) return;  // the split kernel wrote zeros
    const int nsplit = (n + p.chunk - 1) / p.chunk;
    if (nsplit <= 1) return;  // the split kernel wrote the output

    const float *ml = p.ws_ml + static_cast<size_t>(wid) * p.max_splits * 2;
    const float *os = p.ws_o + static_cast<size_t>(wid) * p.max_splits * D;
    float M = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, ml[2 * s]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    const float mu = M == -INFINITY ? 0.f : M;

    float W = 0.f, o[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = 0.f;
    for (int s = 0; s < nsplit; ++s) {
        const float w = ml[2 * s + 1] * fast_exp2(ml[2 * s] - mu);
        W += w;
        const float *src = os + static_cast<size_t>(s) * D + lane * PER;
        if constexpr (PER == 4) {
            const float4 x = *reinterpret_cast<const float4 *>(src);
            o[0] = fmaf(w, x.x, o[0]); o[1] = fmaf(w, x.y, o[1]);
            o[2] = fmaf(w, x.z, o[2]); o[3] = fmaf(w, x.w, o[3]);
        } else {
            const float2 x = *reinterpret_cast<const float2 *>(src);
            o[0] = fmaf(w, x.x, o[0]); o[1] = fmaf(w, x.y, o[1]);
        }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint32_t packed[PER / 2];
#pragma unroll
    for (int e = 0; e < PER / 2; ++e) packed[e] = E::pack2(o[2 * e] * inv, o[2 * e + 1] * inv);
    T *dst = static_cast<T *>(p.out) + static_cast<size_t>(wid) * D + lane * PER;
    if constexpr (PER == 4)
        *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
    else
        *reinterpret_cast<uint32_t *>(dst) = packed[0];
}

template <int D, int G, class E>
cudaError_t launch_typed(const DecodeParams &prm, const DecodePlan &plan, cudaStream_t stream) {
    const int smem = smem_bytes_for<D, G>(plan.tbl_cap);
    auto kern = decode_split_kernel<D, G, E>;
    static int configured_smem = 0;  // per instantiation; raised once per size
    if (smem > configured_smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured_smem = smem;
    }
    dim3 grid(plan.max_splits, prm.Hkv, prm.B);
    kern<<<grid, kThreads, smem, stream>>>(prm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || plan.max_splits <= 1) return e;
    const int warps = prm.B * prm.Hq;
    decode_merge_kernel<D, E><<<(warps + 3) / 4, 128, 0, stream>>>(prm);
    return cudaGetLastError();
}

template <int D, class E>
cudaError_t dispatch_group(int G, const DecodeParams &prm, const DecodePlan &plan,
                           cudaStream_t stream) {
    switch (G) {
        case 1: return launch_typed<D, 1, E>(prm, plan, stream);
        case 2: return launch_typed<D, 2, E>(prm, plan, stream);
        case 3: return launch_typed<D, 3, E>(prm, plan, stream);
        case 4: return launch_typed<D, 4, E>(prm, plan, stream);
        case 5: return launch_typed<D, 5, E>(prm, plan, stream);
        case 6: return launch_typed<D, 6, E>(prm, plan, stream);
        case 7: return launch_typed<D, 7, E>(prm, plan, stream);
        case 8: return launch_typed<D, 8, E>(prm, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

DecodePlan plan_decode(int B, int Hq, int Hkv, int D, int max_blocks_per_seq, int block_size) {
    DecodePlan plan{};
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    const long long tiles_max = (max_ctx + kTN - 1) / kTN;
    const int ctas_per_sm = D == 128 ? 2 : 3;
    const long long target = static_cast<long long>(device_sm_count()) * ctas_per_sm * 4;
    const long long pairs = static_cast<long long>(B) * Hkv;
    // guess the mean context as half the maximum; cut chunks so ~4 waves of CTAs exist, but
    // never let one CTA stream more than ~256 KB (tail) or less than one tile
    const long long expect_tiles = pairs * ((tiles_max + 1) / 2);
    long long tpc = (expect_tiles + target - 1) / (target > 0 ? target : 1);
    const long long tpc_max = D == 128 ? 8 : 16;
    if (tpc < 1) tpc = 1;
    if (tpc > tpc_max) tpc = tpc_max;
    plan.chunk = static_cast<int>(tpc * kTN);
    plan.max_splits = max_ctx > 0 ? static_cast<int>((max_ctx + plan.chunk - 1) / plan.chunk) : 1;
    plan.tbl_cap = plan.chunk / block_size + 2;
    plan.ws_bytes = plan.max_splits > 1
                        ? static_cast<size_t>(B) * Hq * plan.max_splits * (D + 2) * sizeof(float)
                        : 0;
    return plan;
}

cudaError_t launch_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    DecodeParams prm{};
    prm.q = a.q;
    prm.k_cache = a.k_cache;
    prm.v_cache = a.v_cache;
    prm.block_tables = a.block_tables;
    prm.context_lens = a.context_lens;
    prm.out = a.out;
    float *ws = static_cast<float *>(a.workspace);
    prm.ws_o = ws;
    prm.ws_ml = ws ? ws + static_cast<size_t>(a.B) * a.Hq * plan.max_splits * a.D : nullptr;
    prm.err = a.err;
    prm.B = a.B;
    prm.Hq = a.Hq;
    prm.Hkv = a.Hkv;
    prm.max_blocks = a.max_blocks;
    prm.num_blocks = a.num_blocks;
    prm.chunk = plan.chunk;
    prm.max_splits = plan.max_splits;
    prm.tbl_cap = plan.tbl_cap;
    prm.geom.block_size = a.block_size;
    prm.geom.shift = log2_if_pow2(a.block_size);
    prm.scale_log2 = a.scale * kLog2e;
    const int G = a.Hq / a.Hkv;
    if (a.D == 128)
        return a.dtype == PA_BF16 ? dispatch_group<128, BF16>(G, prm, plan, stream)
                                  : dispatch_group<128, F16>(G, prm, plan, stream);
    return a.dtype == PA_BF16 ? dispatch_group<64, BF16>(G, prm, plan, stream)
                              : dispatch_group<64, F16>(G, prm, plan, stream);
}

}  // namespace pa
