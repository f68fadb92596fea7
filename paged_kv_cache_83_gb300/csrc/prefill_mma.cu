// prefill_mma.cu: varlen causal prefill with a paged prefix (pa_prefill_varlen), warp-level
// mma.sync version: the general path for the launches the tcgen05 kernel (prefill_tc.cu) does not
// take (pool block sizes without an 8-row power-of-two divisor, an output that is not 16-byte
// aligned).
//
// Source: "nano-vLLM Part 4", section 3 (prefill: packed prompts, variable-length attention with
// an optional prefix block table); smzdm nano-vLLM deep dive, "GPU执行优化" (cu_seqlens mark the
// sequence boundaries) and "模型实现细节" (the prefix cache is used when cu_seqlens_k >
// cu_seqlens_q); "mini-vLLM" (prompts attending causally to themselves).
//
// Flash-attention tiling: a CTA owns 64 query rows of one (sequence, query head); each of its 4
// warps owns 16 rows. Key/value tiles of 64 rows are double-buffered in shared memory with
// 16-byte cp.async copies whose source rows come through the block table (pool) or straight from
// the packed k/v (no table). S = Q K^T and O += P V run on mma.sync.m16n8k16 with fp32
// accumulators; the online softmax is in base 2 with the scale folded in; P goes from the S
// accumulators to the A operand of the PV product without touching shared memory. Causal rows are
// aligned to the end of the keys (row r of a sequence with P cached keys sees keys 0 .. P + r).
// Tiles are XOR-swizzled by 16-byte chunk so ldmatrix reads are conflict free.
#include <math.h>

#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kBM = 64;  // query rows per CTA
constexpr int kBN = 64;  // keys per tile
constexpr int kThreads = 128;
constexpr unsigned kFull = 0xffffffffu;

struct PrefillParams {
    const void *q, *k, *v, *k_cache, *v_cache;
    const int32_t *cu_q, *cu_k, *block_tables;
    void *out;
    int32_t *err;
    int S, Hq, Hkv, G, max_blocks, num_blocks, causal, max_seqlen_q;
    BlockGeom geom;
    float scale_log2;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <class E>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<BF16>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<F16>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte offset of 16-byte chunk `ch` of row `row` in a swizzled tile with NCH chunks per row
template <int NCH>
__device__ __forceinline__ uint32_t swz_off(int row, int ch) {
    return row * NCH * 16 + ((ch ^ (row & 7)) * 16);
}

template <int D, class E>
__global__ void __launch_bounds__(kThreads, 2) prefill_mma_kernel(const PrefillParams p) {
    using T = typename E::T;
    constexpr int NCH = D / 8;
    constexpr int TILE = kBN * D * 2;
    constexpr int KSTEPS = D / 16;
    constexpr int DT = D / 8;  // 8-column output tiles
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *qs = smem;
    unsigned char *ks = smem + kBM * D * 2;
    unsigned char *vs = ks + 2 * TILE;

    const int mb = gridDim.x - 1 - blockIdx.x;  // longest (most keys) row blocks first
    const int h = blockIdx.y, s = blockIdx.z;
    const int g = h / p.G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int q0 = p.cu_q[s], ql = p.cu_q[s + 1] - q0;
    const int k0 = p.cu_k[s], kl = p.cu_k[s + 1] - k0;
    if (ql < 0 || ql > p.max_seqlen_q) {
        if (mb == 0 && h == 0 && tid == 0) raise_err(p.err, PA_DEVERR_LENGTH);
        return;  // row range unknown: nothing is written
    }
    const int m0 = mb * kBM;
    if (m0 >= ql) return;
    const int mrows = min(kBM, ql - m0);
    T *out = static_cast<T *>(p.out);
    bool length_bad = kl < ql;
    if (p.block_tables && static_cast<long long>(kl) > static_cast<long long>(p.max_blocks) * p.geom.block_size)
        length_bad = true;
    if (length_bad) {
        if (mb == 0 && h == 0 && tid == 0) raise_err(p.err, PA_DEVERR_LENGTH);
        for (int i = tid; i < mrows * D; i += kThreads)
            out[(static_cast<size_t>(q0 + m0 + i / D) * p.Hq + h) * D + i % D] = T(0.f);
        return;
    }
    const int P = kl - ql;
    const int n_end = p.causal ? min(kl, P + m0 + mrows) : kl;  // keys any row here may see
    const int ntiles = (n_end + kBN - 1) / kBN;
    const int32_t *trow =
        p.block_tables ? p.block_tables + static_cast<size_t>(s) * p.max_blocks : nullptr;

    // check the table entries this CTA will read
    int bad = 0;
    if (trow) {
        const int nblk = n_end > 0 ? p.geom.block_of(n_end - 1) + 1 : 0;
        for (int i = tid; i < nblk; i += kThreads) {
            const int id = trow[i];
            if (id < 0 || id >= p.num_blocks) bad = 1;
        }
    }
    bad = __syncthreads_or(bad);
    if (bad && tid == 0) raise_err(p.err, PA_DEVERR_TABLE);

    const T *qg = static_cast<const T *>(p.q);
    const T *ksrc = static_cast<const T *>(trow ? p.k_cache : p.k);
    const T *vsrc = static_cast<const T *>(trow ? p.v_cache : p.v);

    // Q tile (rows past the prompt are zero)
    for (int i = tid; i < kBM * NCH; i += kThreads) {
        const int row = i / NCH, ch = i % NCH;
        const bool ok = row < mrows;
        const size_t off = (static_cast<size_t>(q0 + (ok ? m0 + row : 0)) * p.Hq + h) * D + ch * 8;
        cp_async16(smem_addr(qs) + swz_off<NCH>(row, ch), qg + off, ok ? 16 : 0);
    }
    // returns the element offset of key j's row for kv head g, or -1 when it must not be read
    auto key_off = [&](int j) -> long long {
        if (j >= n_end) return -1;
        long long slot;
        if (trow) {
            const int id = trow[p.geom.block_of(j)];
            if (id < 0 || id >= p.num_blocks) return -1;
            slot = static_cast<long long>(id) * p.geom.block_size + p.geom.offset_of(j);
        } else {
            slot = k0 + j;
        }
        return (slot * p.Hkv + g) * D;
    };
    auto load_kv = [&](int stage, int t) {
        const int n0 = t * kBN;
        const uint32_t kb = smem_addr(ks + stage * TILE), vb = smem_addr(vs + stage * TILE);
        for (int i = tid; i < kBN * NCH; i += kThreads) {
            const int row = i / NCH, ch = i % NCH;
            const long long off = key_off(n0 + row);
            const bool ok = off >= 0;
            const size_t o = ok ? static_cast<size_t>(off) + ch * 8 : 0;
            cp_async16(kb + swz_off<NCH>(row, ch), ksrc + o, ok ? 16 : 0);
            cp_async16(vb + swz_off<NCH>(row, ch), vsrc + o, ok ? 16 : 0);
        }
    };

    load_kv(0, 0);
    cp_async_commit();

    uint32_t qf[KSTEPS][4];
    float o_acc[DT][4];
#pragma unroll
    for (int i = 0; i < DT; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    // this thread's two rows (relative to m0) in the accumulator layout
    const int rowA = warp * 16 + (lane >> 2);
    const int rowB = rowA + 8;
    const int limA = p.causal ? P + m0 + rowA + 1 : kl;  // keys visible to each row
    const int limB = p.causal ? P + m0 + rowB + 1 : kl;

    for (int t = 0; t < ntiles; ++t) {
        cp_async_wait<0>();
        __syncthreads();
        if (t + 1 < ntiles) load_kv((t + 1) & 1, t + 1);
        cp_async_commit();
        if (t == 0) {
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int ch = kk * 2 + (lane >> 4);
                ldsm_x4(smem_addr(qs) + swz_off<NCH>(row, ch), qf[kk][0], qf[kk][1], qf[kk][2],
                        qf[kk][3]);
            }
        }
        const int stage = t & 1;
        const uint32_t kb = smem_addr(ks + stage * TILE), vb = smem_addr(vs + stage * TILE);
        const int n0 = t * kBN;

        // S = Q K^T for this warp's 16 rows x 64 keys
        float sacc[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                const int row = np * 16 + (lane & 7) + (lane >> 4) * 8;
                const int ch = kk * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kb + swz_off<NCH>(row, ch), b0, b1, b2, b3);
                mma16816<E>(sacc[2 * np], qf[kk], b0, b1);
                mma16816<E>(sacc[2 * np + 1], qf[kk], b2, b3);
            }
        }

        // scale, mask, online softmax (two rows per thread; 4 lanes share a row)
        const bool need_mask = bad || (n0 + kBN > min(limA, kl)) || (n0 + kBN > kl);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = sacc[nt][e] * p.scale_log2;
                if (need_mask) {
                    const int j = n0 + nt * 8 + (lane & 3) * 2 + (e & 1);
                    const int lim = e < 2 ? limA : limB;
                    bool ok = j < lim && j < kl;
                    if (ok && bad) ok = key_off(j) >= 0;
                    if (!ok) x = -INFINITY;
                }
                sacc[nt][e] = x;
            }
        float alpha[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) mx = fmaxf(mx, fmaxf(sacc[nt][2 * rr], sacc[nt][2 * rr + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
            const float m_new = fmaxf(m_run[rr], mx);
            const float mu = m_new == -INFINITY ? 0.f : m_new;
            alpha[rr] = fast_exp2(m_run[rr] - mu);
            m_run[rr] = m_new;
            float sum = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                sacc[nt][2 * rr] = fast_exp2(sacc[nt][2 * rr] - mu);
                sacc[nt][2 * rr + 1] = fast_exp2(sacc[nt][2 * rr + 1] - mu);
                sum += sacc[nt][2 * rr] + sacc[nt][2 * rr + 1];
            }
            l_run[rr] = l_run[rr] * alpha[rr] + sum;
        }
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
            o_acc[dt][0] *= alpha[0];
            o_acc[dt][1] *= alpha[0];
            o_acc[dt][2] *= alpha[1];
            o_acc[dt][3] *= alpha[1];
        }

        // O += P V
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
            uint32_t a[4];
            a[0] = E::pack2(sacc[2 * kk][0], sacc[2 * kk][1]);
            a[1] = E::pack2(sacc[2 * kk][2], sacc[2 * kk][3]);
            a[2] = E::pack2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
            a[3] = E::pack2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
            for (int dp = 0; dp < DT / 2; ++dp) {
                const int row = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int ch = dp * 2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vb + swz_off<NCH>(row, ch), b0, b1, b2, b3);
                mma16816<E>(o_acc[2 * dp], a, b0, b1);
                mma16816<E>(o_acc[2 * dp + 1], a, b2, b3);
            }
        }
    }
    cp_async_wait<0>();

    // normalise and store
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        l_run[rr] += __shfl_xor_sync(kFull, l_run[rr], 1);
        l_run[rr] += __shfl_xor_sync(kFull, l_run[rr], 2);
    }
    const float invA = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f;
    const float invB = l_run[1] > 0.f ? 1.f / l_run[1] : 0.f;
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
        const int d = dt * 8 + (lane & 3) * 2;
        if (rowA < mrows)
            *reinterpret_cast<uint32_t *>(out + (static_cast<size_t>(q0 + m0 + rowA) * p.Hq + h) * D + d) =
                E::pack2(o_acc[dt][0] * invA, o_acc[dt][1] * invA);
        if (rowB < mrows)
            *reinterpret_cast<uint32_t *>(out + (static_cast<size_t>(q0 + m0 + rowB) * p.Hq + h) * D + d) =
                E::pack2(o_acc[dt][2] * invB, o_acc[dt][3] * invB);
    }
}

template <int D, class E>
cudaError_t launch_typed(const PrefillParams &prm, cudaStream_t stream) {
    constexpr int smem = kBM * D * 2 + 4 * kBN * D * 2;
    auto kern = prefill_mma_kernel<D, E>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid((prm.max_seqlen_q + kBM - 1) / kBM, prm.Hq, prm.S);
    kern<<<grid, kThreads, smem, stream>>>(prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
    if (a.S == 0 || a.max_seqlen_q == 0) return cudaSuccess;
    if (tc_prefill_supported(a)) return launch_prefill_tc(a, stream);
    PrefillParams prm{};
    prm.q = a.q;
    prm.k = a.k;
    prm.v = a.v;
    prm.k_cache = a.k_cache;
    prm.v_cache = a.v_cache;
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
    prm.geom.block_size = a.block_size;
    prm.geom.shift = log2_if_pow2(a.block_size);
    prm.scale_log2 = a.scale * kLog2e;
    if (a.D == 128)
        return a.dtype == PA_BF16 ? launch_typed<128, BF16>(prm, stream)
                                  : launch_typed<128, F16>(prm, stream);
    return a.dtype == PA_BF16 ? launch_typed<64, BF16>(prm, stream)
                              : launch_typed<64, F16>(prm, stream);
}

}  // namespace pa
