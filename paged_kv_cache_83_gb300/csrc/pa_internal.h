// pa_internal.h: argument bundles and launchers behind the C ABI (include/pa.h).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "pa_common.cuh"

namespace pa {

int device_sm_count();  // SMs of the current device (cached per device)

// ------------------------------------------------------------------------------------------
// Staging between host memory and the device by the SMs (stage.cu).
// The device address of the host range [p, p + bytes) when the device may load and store it
// directly: page-locked memory registered with CUDA whose first and last bytes map to device
// addresses bytes - 1 apart. nullptr otherwise (pageable or other memory, a range that leaves its
// allocation, no CUDA device).
void *mapped_host(const void *p, size_t bytes);
// Copies bytes (a multiple of 4; both addresses 16-byte aligned) with a kernel on `stream`;
// dependent: launched as a programmatic dependent of the previous grid (which must let it launch
// early and complete before this one reads).
cudaError_t launch_stage(void *dst, const void *src, size_t bytes, bool dependent, cudaStream_t stream);

// ------------------------------------------------------------------------------------------
struct StoreArgs {
    const void *k, *v;
    void *k_cache, *v_cache;
    const int32_t *slot_mapping;
    int T, num_blocks, block_size, Hkv, D;
    int32_t *err;
};
cudaError_t launch_store_kv(const StoreArgs &a, cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// Decode: one persistent CTA per SM streams an equal share of the (sequence, kv head, tile)
// space; pieces of a context shared by two CTAs are combined by a small merge kernel.
struct DecodePlan {
    size_t ws_bytes;  // scratch: per SM two partial results and one record
};
// allow_wide: the D = 64 tensor-core kernels may run two CTAs per SM on large batches (the
// launch and its workspace differ); the no-alloc entry point keeps one
DecodePlan plan_decode(int B, int Hq, int Hkv, int D, int max_blocks_per_seq, int block_size,
                       bool allow_wide = true);

struct DecodeArgs {
    void *out;
    const void *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    int B, Hq, Hkv, D, max_blocks, block_size, num_blocks;
    float scale;
    pa_dtype dtype;
    void *workspace;
    int32_t *err;
    const void *k_new = nullptr, *v_new = nullptr;  // fused store + decode: new rows [B, Hkv, D]
    bool allow_wide = true;                           // see plan_decode
};
cudaError_t launch_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream);
// short contexts (decode_short.cu): at most 256 positions per sequence by the table's width, one
// CTA per (sequence, kv head), no workspace; launch_decode takes it when it applies
bool short_decode_supported(const DecodeArgs &a);
cudaError_t launch_decode_short(const DecodeArgs &a, cudaStream_t stream);
// the dynamic-tail units (K2) of the last completed launch on this workspace (pa_decode's launch
// configuration), read from unit 0's record; -1 on invalid sizes or a failed copy
int decode_debug_tail_units(const void *workspace, int B, int Hq, int Hkv, int D,
                            int max_blocks_per_seq, int block_size);
// pa_decode with the choice of allow_wide (pa_decode: allowed; pa_decode_noalloc: not, so that
// its fixed scratch covers the same shapes whatever the batch)
pa_status decode_entry(void *out, const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                       int B, int Hq, int Hkv, int D, int block_size, int num_blocks, float scale,
                       pa_dtype dtype, void *workspace, size_t workspace_bytes, int32_t *err,
                       cudaStream_t stream, bool allow_wide);

// ------------------------------------------------------------------------------------------
struct PrefillArgs {
    void *out;
    const void *q, *k, *v, *k_cache, *v_cache;
    const int32_t *cu_q, *cu_k, *block_tables;
    int S, max_seqlen_q, max_blocks, Hq, Hkv, D, block_size, num_blocks, causal;
    int max_seqlen_k;      // the caller's bound on keys per sequence: orders the work, nothing else
    int total_q, total_k;  // rows of q / out, and of the packed k, v
    float scale;
    pa_dtype dtype;
    int32_t *err;
};
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream);
// tensor-core (tcgen05) prefill: head dim 64 or 128, any group size, K/V boxes of >= 8 rows
bool tc_prefill_supported(const PrefillArgs &a);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream);

inline int log2_if_pow2(int x) {
    if (x <= 0 || (x & (x - 1))) return -1;
    int s = 0;
    while ((1 << s) < x) ++s;
    return s;
}

}  // namespace pa
