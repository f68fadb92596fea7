// decode_short.cu: paged grouped-query decode (pa_decode, pa_store_decode) for short contexts.
//
// Source: "nano-vLLM Part 4", section 3 (decode: one already-sampled token per sequence,
// attention over its cached history through a block table); "mini-vLLM" (one token per sequence
// attending to that sequence's cached keys and values, grouped-query attention).
//
// When no sequence can hold more than kShortMaxPos positions (the table's width times the block
// size), a step is a few hundred KB at most and its time is the chain of dependent memory round
// trips, not bandwidth. This kernel keeps that chain short: one CTA per (sequence, kv head) reads
// the length, the query rows and the whole table row together (one round trip), then copies every
// K and V row of the sequence into shared memory with 16-byte cp.async copies, consecutive lanes on
// consecutive chunks of a row (a second one), and computes the scores (a thread per position), the
// softmax and P V from shared memory, and writes the output. No warp roles, no pipeline, no
// partial results, no merge.
//
// Semantics are those of the persistent kernel (decode.cu): context 0 gives zero rows; a length
// outside [0, table width * block size] gives zero rows and PA_DEVERR_LENGTH; a table entry
// outside [0, num_blocks) masks its positions and raises PA_DEVERR_TABLE. With k_new / v_new (the
// fused store) position n - 1 takes its K / V row from them, and the row is also written to the
// pool slot of that position when its table entry is valid.
#include <math.h>

#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kShortThreads = 256;
constexpr int kShortMaxPos = 256;  // positions per sequence this kernel takes (one per thread)

struct ShortParams {
    const void *q, *k_new, *v_new;
    void *k_cache, *v_cache, *out;
    const int32_t *block_tables, *context_lens;
    int32_t *err;
    int Hq, Hkv, max_blocks, num_blocks;
    BlockGeom geom;
    float scale_log2;
};

// dynamic shared memory: K and V rows [kShortMaxPos][D] (16-bit; the 16-byte chunk c of row r at
// chunk c ^ (r % 8), so that a thread per row reads them without bank conflicts), scores
// [G][kShortMaxPos], query rows [G][D], block ids [kShortMaxPos], P V partials [subsets][G][D],
// reductions
template <int D, int G>
struct ShortSmem {
    static constexpr int kSub = kShortThreads / (D / 2);  // position subsets of the P V loop
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + kShortMaxPos * D * 2;
    static constexpr int OFF_S = OFF_V + kShortMaxPos * D * 2;
    static constexpr int OFF_Q = OFF_S + G * kShortMaxPos * 4;
    static constexpr int OFF_ID = OFF_Q + G * D * 4;
    static constexpr int OFF_PV = OFF_ID + kShortMaxPos * 4;
    static constexpr int OFF_RED = OFF_PV + kSub * G * D * 4;
    static constexpr int BYTES = OFF_RED + 2 * (kShortThreads / 32) * G * 4 + 2 * G * 4;
};

template <int D, int G, class E>
__global__ void __launch_bounds__(kShortThreads) decode_short_kernel(const __grid_constant__ ShortParams p) {
    using T = typename E::T;
    using L = ShortSmem<D, G>;
    constexpr int NCH = D / 8;  // 16-byte chunks per row
    extern __shared__ __align__(16) unsigned char smem[];
    float *sc = reinterpret_cast<float *>(smem + L::OFF_S);  // [G][kShortMaxPos]
    float *qs = reinterpret_cast<float *>(smem + L::OFF_Q);  // [G][D], scaled by scale * log2 e
    int *ids = reinterpret_cast<int *>(smem + L::OFF_ID);
    float *pvp = reinterpret_cast<float *>(smem + L::OFF_PV);  // [kSub][G][D]
    float *red = reinterpret_cast<float *>(smem + L::OFF_RED);  // [2][warps][G]
    float *stat = red + 2 * (kShortThreads / 32) * G;           // row max [G], sum [G]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / p.Hkv, g = blockIdx.x % p.Hkv;
    // the next grid may launch now; nothing this grid reads is touched before the grids it
    // depends on have completed
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // the length, the whole table row (at most kShortMaxPos entries) and the G query rows
    // (scaled), loaded together
    const int n = p.context_lens[b];
    const int32_t *trow = p.block_tables + static_cast<size_t>(b) * p.max_blocks;
    for (int i = tid; i < p.max_blocks; i += kShortThreads) ids[i] = trow[i];
    const T *qg = static_cast<const T *>(p.q) + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * G) * D;
    for (int i = tid; i < G * NCH; i += kShortThreads) {
        float f[8];
        unpack8<E>(reinterpret_cast<const uint4 *>(qg)[i], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) qs[i * 8 + e] = f[e] * p.scale_log2;
    }
    const long long cap = static_cast<long long>(p.max_blocks) * p.geom.block_size;
    T *out = static_cast<T *>(p.out) + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * G) * D;
    if (n <= 0 || n > cap) {
        if ((n < 0 || n > cap) && g == 0 && tid == 0) raise_err(p.err, PA_DEVERR_LENGTH);
        for (int i = tid; i < G * D / 8; i += kShortThreads)
            reinterpret_cast<uint4 *>(out)[i] = make_uint4(0, 0, 0, 0);
        return;
    }
    __syncthreads();

    // every K and V row of the sequence into shared memory: 16-byte copies, consecutive lanes on
    // consecutive chunks of a row; a masked row (table entry outside the pool) is zero-filled.
    // With the fused store the last position's rows come from k_new / v_new.
    const size_t new_row = (static_cast<size_t>(b) * p.Hkv + g) * D;
    bool bad = false;
    for (int i = tid; i < n * NCH; i += kShortThreads) {
        const int pos = i / NCH, c = i % NCH;
        const int id = ids[p.geom.block_of(pos)];
        const bool valid = id >= 0 && id < p.num_blocks;
        const bool is_new = p.k_new != nullptr && pos == n - 1;
        const size_t row = valid ? (static_cast<size_t>(id) * p.geom.block_size + p.geom.offset_of(pos)) * p.Hkv + g : 0;
        const T *ksrc = is_new ? static_cast<const T *>(p.k_new) + new_row : static_cast<const T *>(p.k_cache) + row * D;
        const T *vsrc = is_new ? static_cast<const T *>(p.v_new) + new_row : static_cast<const T *>(p.v_cache) + row * D;
        const int bytes = valid || is_new ? 16 : 0;
        const uint32_t off = static_cast<uint32_t>(pos * D * 2 + ((c ^ (pos & 7)) << 4));
        cp_async16(smem_addr(smem + L::OFF_K + off), ksrc + c * 8, bytes);
        cp_async16(smem_addr(smem + L::OFF_V + off), vsrc + c * 8, bytes);
        bad |= !valid;
    }
    cp_async_commit();
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_err(p.err, PA_DEVERR_TABLE);
    cp_async_wait<0>();
    __syncthreads();
    if (p.k_new != nullptr && tid < 2 * NCH) {
        // the fused store: the new token's K and V rows, now in shared memory, into the pool slot of
        // position n - 1 (when its table entry is valid); nothing in this launch reads that slot
        const int pos = n - 1, c = tid % NCH;
        const int id = ids[p.geom.block_of(pos)];
        if (id >= 0 && id < p.num_blocks) {
            const size_t row = (static_cast<size_t>(id) * p.geom.block_size + p.geom.offset_of(pos)) * p.Hkv + g;
            const bool is_v = tid >= NCH;
            const uint4 w = *reinterpret_cast<const uint4 *>(smem + (is_v ? L::OFF_V : L::OFF_K) + pos * D * 2 +
                                                             ((c ^ (pos & 7)) << 4));
            reinterpret_cast<uint4 *>(static_cast<T *>(is_v ? p.v_cache : p.k_cache) + row * D)[c] = w;
        }
    }

    // scores: a thread per position, its K row from shared memory, the query rows broadcast
    float mloc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) mloc[h] = -INFINITY;
    for (int pos = tid; pos < n; pos += kShortThreads) {
        const int id = ids[p.geom.block_of(pos)];
        if (id < 0 || id >= p.num_blocks) {  // a table entry outside the pool: the position is masked
#pragma unroll
            for (int h = 0; h < G; ++h) sc[h * kShortMaxPos + pos] = -INFINITY;
            continue;
        }
        float acc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = 0.f;
        const unsigned char *krow = smem + L::OFF_K + pos * D * 2;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float kf[8];
            unpack8<E>(*reinterpret_cast<const uint4 *>(krow + ((c ^ (pos & 7)) << 4)), kf);
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h] = fmaf(qs[h * D + c * 8 + e], kf[e], acc[h]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            sc[h * kShortMaxPos + pos] = acc[h];
            mloc[h] = fmaxf(mloc[h], acc[h]);
        }
    }

    // row max per head across the CTA
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float m = mloc[h];
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) red[warp * G + h] = m;
    }
    __syncthreads();
    if (tid < G) {
        float m = -INFINITY;
        for (int w = 0; w < kShortThreads / 32; ++w) m = fmaxf(m, red[w * G + tid]);
        stat[tid] = m;
    }
    __syncthreads();
    // p = 2^(s - m) in place, and the row sums
    float lloc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const float m = stat[h];
        const float mu = m == -INFINITY ? 0.f : m;  // every position masked: p = 0
        lloc[h] = 0.f;
        for (int pos = tid; pos < n; pos += kShortThreads) {
            const float e = fast_exp2(sc[h * kShortMaxPos + pos] - mu);
            sc[h * kShortMaxPos + pos] = e;
            lloc[h] += e;
        }
        for (int o = 16; o >= 1; o >>= 1) lloc[h] += __shfl_xor_sync(0xffffffffu, lloc[h], o);
        if (lane == 0) red[(kShortThreads / 32 + warp) * G + h] = lloc[h];
    }
    __syncthreads();
    if (tid < G) {
        float l = 0.f;
        for (int w = 0; w < kShortThreads / 32; ++w) l += red[(kShortThreads / 32 + w) * G + tid];
        stat[G + tid] = l;
    }
    // O = P V: thread = two output columns of one subset of the positions, all G heads
    const int d2 = tid % (D / 2), sub = tid / (D / 2);
    float o0[G], o1[G];
#pragma unroll
    for (int h = 0; h < G; ++h) o0[h] = o1[h] = 0.f;
    for (int pos = sub; pos < n; pos += L::kSub) {
        // columns 2 d2, 2 d2 + 1: 16-byte chunk d2 / 4 of the row, stored at chunk (d2 / 4) ^ (pos % 8)
        const uint32_t w = *reinterpret_cast<const uint32_t *>(
            smem + L::OFF_V + pos * D * 2 + ((((d2 >> 2) ^ (pos & 7))) << 4) + (d2 & 3) * 4);
        const float2 v = E::unpack2(w);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float pr = sc[h * kShortMaxPos + pos];
            o0[h] = fmaf(pr, v.x, o0[h]);
            o1[h] = fmaf(pr, v.y, o1[h]);
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        pvp[(sub * G + h) * D + 2 * d2] = o0[h];
        pvp[(sub * G + h) * D + 2 * d2 + 1] = o1[h];
    }
    __syncthreads();
    for (int i = tid; i < G * D / 2; i += kShortThreads) {
        const int h = i / (D / 2), c = i % (D / 2);
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int s = 0; s < L::kSub; ++s) {
            x += pvp[(s * G + h) * D + 2 * c];
            y += pvp[(s * G + h) * D + 2 * c + 1];
        }
        const float l = stat[G + h];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        reinterpret_cast<uint32_t *>(out + static_cast<size_t>(h) * D)[c] = E::pack2(x * inv, y * inv);
    }
}

template <int D, int G, class E>
cudaError_t launch_short_typed(const ShortParams &prm, int pairs, cudaStream_t stream) {
    constexpr int smem = ShortSmem<D, G>::BYTES;
    auto kern = decode_short_kernel<D, G, E>;
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    // launched as a programmatic dependent of what precedes it in the stream, like the
    // persistent kernels: its launch overlaps the tail of the grid before it
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(pairs);
    cfg.blockDim = dim3(kShortThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <int D, class E>
cudaError_t dispatch_short(int G, const ShortParams &prm, int pairs, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_short_typed<D, 1, E>(prm, pairs, stream);
        case 2: return launch_short_typed<D, 2, E>(prm, pairs, stream);
        case 3: return launch_short_typed<D, 3, E>(prm, pairs, stream);
        case 4: return launch_short_typed<D, 4, E>(prm, pairs, stream);
        case 5: return launch_short_typed<D, 5, E>(prm, pairs, stream);
        case 6: return launch_short_typed<D, 6, E>(prm, pairs, stream);
        case 7: return launch_short_typed<D, 7, E>(prm, pairs, stream);
        case 8: return launch_short_typed<D, 8, E>(prm, pairs, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool short_decode_supported(const DecodeArgs &a) {
    // every sequence fits the kernel's shared memory (an upper bound from the table's width), and
    // one (sequence, kv head) per CTA stays within a few waves of the SMs
    const long long max_ctx = static_cast<long long>(a.max_blocks) * a.block_size;
    const long long pairs = static_cast<long long>(a.B) * a.Hkv;
    return max_ctx <= kShortMaxPos && pairs <= 4ll * device_sm_count() && a.Hq / a.Hkv <= 8 &&
           (a.D == 64 || a.D == 128);
}

cudaError_t launch_decode_short(const DecodeArgs &a, cudaStream_t stream) {
    ShortParams prm{};
    prm.q = a.q;
    prm.k_new = a.k_new;
    prm.v_new = a.v_new;
    prm.k_cache = const_cast<void *>(a.k_cache);
    prm.v_cache = const_cast<void *>(a.v_cache);
    prm.out = a.out;
    prm.block_tables = a.block_tables;
    prm.context_lens = a.context_lens;
    prm.err = a.err;
    prm.Hq = a.Hq;
    prm.Hkv = a.Hkv;
    prm.max_blocks = a.max_blocks;
    prm.num_blocks = a.num_blocks;
    prm.geom.block_size = a.block_size;
    prm.geom.shift = log2_if_pow2(a.block_size);
    prm.scale_log2 = a.scale * kLog2e;
    const int G = a.Hq / a.Hkv, pairs = a.B * a.Hkv;
    if (a.D == 128)
        return a.dtype == PA_BF16 ? dispatch_short<128, BF16>(G, prm, pairs, stream)
                                  : dispatch_short<128, F16>(G, prm, pairs, stream);
    return a.dtype == PA_BF16 ? dispatch_short<64, BF16>(G, prm, pairs, stream)
                              : dispatch_short<64, F16>(G, prm, pairs, stream);
}

}  // namespace pa
