// store_kv.cu: the slot-mapped K/V scatter (pa_store_kv).
//
// Source: "nano-vLLM Part 4", section 3 (each step writes the new tokens' K/V through per-token
// slot mappings); smzdm nano-vLLM deep dive, "模型实现细节" (store_kvcache puts each new K and V
// row at its physical position).
//
// A token's K row for all kv heads (Hkv * D elements) is contiguous in the source and, in the
// [num_blocks, block_size, Hkv, D] pool, contiguous at slot * Hkv * D. So the scatter is a
// gather-free row copy: every thread moves 16-byte chunks, with UNROLL independent loads in
// flight before its stores, and the grid is a few resident waves of the SMs. It is bound by
// HBM: 2 reads + 2 writes of T * Hkv * D * 2 bytes.
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kStoreThreads = 256;
constexpr int kStoreUnroll = 4;

__global__ void __launch_bounds__(kStoreThreads)
store_kv_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint4 *__restrict__ kc,
                uint4 *__restrict__ vc, const int32_t *__restrict__ slot_mapping, int T,
                int row16, long long num_slots, int32_t *err) {
    const unsigned total = static_cast<unsigned>(T) * static_cast<unsigned>(row16);
    const unsigned stride = gridDim.x * blockDim.x;
    for (unsigned base = blockIdx.x * blockDim.x + threadIdx.x; base < total;
         base += stride * kStoreUnroll) {
        uint4 kr[kStoreUnroll], vr[kStoreUnroll];
        long long dst[kStoreUnroll];
#pragma unroll
        for (int u = 0; u < kStoreUnroll; ++u) {
            const unsigned idx = base + u * stride;
            dst[u] = -1;
            if (idx < total) {
                const unsigned t = idx / static_cast<unsigned>(row16);
                const unsigned c = idx - t * static_cast<unsigned>(row16);
                const long long s = __ldg(slot_mapping + t);
                if (s >= num_slots) {
                    if (c == 0) raise_err(err, PA_DEVERR_SLOT);
                } else if (s >= 0) {
                    dst[u] = s * row16 + c;
                    kr[u] = ldg_stream(k + idx);
                    vr[u] = ldg_stream(v + idx);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kStoreUnroll; ++u) {
            if (dst[u] >= 0) {
                stg128(kc + dst[u], kr[u]);
                stg128(vc + dst[u], vr[u]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_store_kv(const StoreArgs &a, cudaStream_t stream) {
    const int row16 = a.Hkv * a.D / 8;  // 16-byte chunks per token row
    const long long total = static_cast<long long>(a.T) * row16;
    if (total == 0) return cudaSuccess;
    const long long per_cta = static_cast<long long>(kStoreThreads) * kStoreUnroll;
    long long grid = (total + per_cta - 1) / per_cta;
    const long long cap = static_cast<long long>(device_sm_count()) * 8;
    if (grid > cap) grid = cap;
    store_kv_kernel<<<static_cast<unsigned>(grid), kStoreThreads, 0, stream>>>(
        static_cast<const uint4 *>(a.k), static_cast<const uint4 *>(a.v),
        static_cast<uint4 *>(a.k_cache), static_cast<uint4 *>(a.v_cache), a.slot_mapping, a.T,
        row16, static_cast<long long>(a.num_blocks) * a.block_size, a.err);
    return cudaGetLastError();
}

}  // namespace pa
