// pa_api.cu: the C ABI declared in include/pa.h: argument checks, then the kernel launchers.
#include <limits.h>

#include "pa_internal.h"

namespace pa {

int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    if (dev < 64) cached[dev] = n;
    return n;
}

}  // namespace pa

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dtype_ok(pa_dtype d) { return d == PA_F16 || d == PA_BF16; }

// head / dim checks shared by the attention calls
pa_status check_heads(int Hq, int Hkv, int D) {
    if (Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv) return PA_ERR_SHAPE;
    if (Hq / Hkv > 8 || (D != 64 && D != 128)) return PA_ERR_UNSUPPORTED;
    if (Hq > 65535 || Hkv > 65535) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

pa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// pa_store_decode_host's device workspace: the staged inputs and output at 256-byte offsets,
// then pa_decode's workspace
struct HostStage {
    size_t q, kn, vn, bt, cl, out, ws, total;
};
HostStage host_stage(int B, int Hq, int Hkv, int D, int max_blocks, size_t ws_bytes) {
    HostStage s{};
    size_t o = 0;
    const size_t qb = static_cast<size_t>(B) * Hq * D * 2, kb = static_cast<size_t>(B) * Hkv * D * 2;
    s.q = o;
    o += align256(qb);
    s.kn = o;
    o += align256(kb);
    s.vn = o;
    o += align256(kb);
    s.bt = o;
    o += align256(static_cast<size_t>(B) * max_blocks * 4);
    s.cl = o;
    o += align256(static_cast<size_t>(B) * 4);
    s.out = o;
    o += align256(qb);
    s.ws = o;
    s.total = o + align256(ws_bytes);
    return s;
}

}  // namespace

extern "C" {

const char *pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_NULL: return "a required pointer is NULL";
        case PA_ERR_SHAPE: return "inconsistent or out-of-range size";
        case PA_ERR_DTYPE: return "unknown dtype";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or alignment";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_CUDA: return "CUDA runtime error";
    }
    return "unknown status";
}

pa_status pa_store_kv(const void *k, const void *v, void *k_cache, void *v_cache,
                      const int32_t *slot_mapping, int T, int num_blocks, int block_size, int Hkv,
                      int D, pa_dtype dtype, int32_t *err, cudaStream_t stream) {
    if (!dtype_ok(dtype)) return PA_ERR_DTYPE;
    if (T < 0 || num_blocks < 0 || block_size < 1 || Hkv < 1 || D < 1) return PA_ERR_SHAPE;
    if (D % 8) return PA_ERR_UNSUPPORTED;
    if (T == 0) return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_NULL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_UNSUPPORTED;
    if (static_cast<long long>(T) * Hkv * D / 8 > UINT_MAX / 2) return PA_ERR_UNSUPPORTED;
    pa::StoreArgs a{k, v, k_cache, v_cache, slot_mapping, T, num_blocks, block_size, Hkv, D, err};
    return from_cuda(pa::launch_store_kv(a, stream));
}

size_t pa_decode_workspace_size(int B, int Hq, int Hkv, int D, int max_blocks_per_seq,
                                int block_size) {
    if (B <= 0 || check_heads(Hq, Hkv, D) != PA_OK || max_blocks_per_seq < 0 || block_size < 1)
        return 0;
    if (static_cast<long long>(max_blocks_per_seq) * block_size > INT_MAX) return 0;
    return pa::plan_decode(B, Hq, Hkv, D, max_blocks_per_seq, block_size).ws_bytes;
}

int pa_decode_debug_tail_units(const void *workspace, int B, int Hq, int Hkv, int D,
                               int max_blocks_per_seq, int block_size) {
    if (pa_decode_workspace_size(B, Hq, Hkv, D, max_blocks_per_seq, block_size) == 0) return -1;
    return pa::decode_debug_tail_units(workspace, B, Hq, Hkv, D, max_blocks_per_seq, block_size);
}

}  // extern "C"

namespace pa {
pa_status decode_entry(void *out, const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                       int B, int Hq, int Hkv, int D, int block_size, int num_blocks, float scale,
                       pa_dtype dtype, void *workspace, size_t workspace_bytes, int32_t *err,
                       cudaStream_t stream, bool allow_wide) {
    if (!dtype_ok(dtype)) return PA_ERR_DTYPE;
    if (B < 0 || max_blocks_per_seq < 0 || block_size < 1 || num_blocks < 0) return PA_ERR_SHAPE;
    pa_status st = check_heads(Hq, Hkv, D);
    if (st != PA_OK) return st;
    if (static_cast<long long>(max_blocks_per_seq) * block_size > INT_MAX) return PA_ERR_SHAPE;
    if (B > 65535) return PA_ERR_UNSUPPORTED;
    if (B == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !context_lens ||
        (max_blocks_per_seq > 0 && !block_tables))
        return PA_ERR_NULL;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_UNSUPPORTED;
    if (static_cast<long long>(num_blocks) * block_size > INT_MAX) return PA_ERR_UNSUPPORTED;
    const pa::DecodePlan plan = pa::plan_decode(B, Hq, Hkv, D, max_blocks_per_seq, block_size, allow_wide);
    if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes || !aligned16(workspace)))
        return PA_ERR_WORKSPACE;
    pa::DecodeArgs a{out,  q,         k_cache,           v_cache,    block_tables,
                     context_lens, B, Hq,                Hkv,        D,
                     max_blocks_per_seq,  block_size, num_blocks, scale, dtype,
                     workspace,    err};
    a.allow_wide = allow_wide;
    return from_cuda(pa::launch_decode(a, plan, stream));
}
}  // namespace pa

extern "C" {

pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int B, int Hq, int Hkv, int D, int block_size,
                    int num_blocks, float scale, pa_dtype dtype, void *workspace,
                    size_t workspace_bytes, int32_t *err, cudaStream_t stream) {
    return pa::decode_entry(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, B,
                            Hq, Hkv, D, block_size, num_blocks, scale, dtype, workspace,
                            workspace_bytes, err, stream, true);
}

pa_status pa_store_decode(void *out, const void *q, const void *k_new, const void *v_new,
                          void *k_cache, void *v_cache, const int32_t *block_tables,
                          int max_blocks_per_seq, const int32_t *context_lens, int B, int Hq,
                          int Hkv, int D, int block_size, int num_blocks, float scale,
                          pa_dtype dtype, void *workspace, size_t workspace_bytes, int32_t *err,
                          cudaStream_t stream) {
    if (!dtype_ok(dtype)) return PA_ERR_DTYPE;
    if (B < 0 || max_blocks_per_seq < 0 || block_size < 1 || num_blocks < 0) return PA_ERR_SHAPE;
    pa_status st = check_heads(Hq, Hkv, D);
    if (st != PA_OK) return st;
    if (static_cast<long long>(max_blocks_per_seq) * block_size > INT_MAX) return PA_ERR_SHAPE;
    if (B > 65535) return PA_ERR_UNSUPPORTED;
    if (B == 0) return PA_OK;
    if (!out || !q || !k_new || !v_new || !k_cache || !v_cache || !context_lens ||
        (max_blocks_per_seq > 0 && !block_tables))
        return PA_ERR_NULL;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(k_new) || !aligned16(v_new))
        return PA_ERR_UNSUPPORTED;
    if (static_cast<long long>(num_blocks) * block_size > INT_MAX) return PA_ERR_UNSUPPORTED;
    const pa::DecodePlan plan = pa::plan_decode(B, Hq, Hkv, D, max_blocks_per_seq, block_size);
    if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes || !aligned16(workspace)))
        return PA_ERR_WORKSPACE;
    pa::DecodeArgs a{out,  q,         k_cache,           v_cache,    block_tables,
                     context_lens, B, Hq,                Hkv,        D,
                     max_blocks_per_seq,  block_size, num_blocks, scale, dtype,
                     workspace,    err};
    a.k_new = k_new;
    a.v_new = v_new;
    return from_cuda(pa::launch_decode(a, plan, stream));
}

size_t pa_store_decode_host_workspace_size(int B, int Hq, int Hkv, int D, int max_blocks_per_seq,
                                           int block_size) {
    if (B <= 0 || check_heads(Hq, Hkv, D) != PA_OK || max_blocks_per_seq < 0 || block_size < 1)
        return 0;
    if (static_cast<long long>(max_blocks_per_seq) * block_size > INT_MAX) return 0;
    const size_t ws = pa::plan_decode(B, Hq, Hkv, D, max_blocks_per_seq, block_size).ws_bytes;
    return host_stage(B, Hq, Hkv, D, max_blocks_per_seq, ws).total;
}

size_t pa_store_decode_host_layout(int B, int Hq, int Hkv, int D, int max_blocks_per_seq,
                                   size_t *offsets) {
    if (B <= 0 || check_heads(Hq, Hkv, D) != PA_OK || max_blocks_per_seq < 0) return 0;
    const HostStage s = host_stage(B, Hq, Hkv, D, max_blocks_per_seq, 0);
    if (offsets) {
        offsets[0] = s.q;
        offsets[1] = s.kn;
        offsets[2] = s.vn;
        offsets[3] = s.bt;
        offsets[4] = s.cl;
    }
    return s.cl + static_cast<size_t>(B) * 4;
}

pa_status pa_store_decode_host(void *out_host, const void *q_host, const void *k_new_host,
                               const void *v_new_host, void *k_cache, void *v_cache,
                               const int32_t *block_tables_host, int max_blocks_per_seq,
                               const int32_t *context_lens_host, int B, int Hq, int Hkv, int D,
                               int block_size, int num_blocks, float scale, pa_dtype dtype,
                               void *workspace, size_t workspace_bytes, int32_t *err,
                               cudaStream_t stream) {
    if (!dtype_ok(dtype)) return PA_ERR_DTYPE;
    if (B < 0 || max_blocks_per_seq < 0 || block_size < 1 || num_blocks < 0) return PA_ERR_SHAPE;
    pa_status st = check_heads(Hq, Hkv, D);
    if (st != PA_OK) return st;
    if (static_cast<long long>(max_blocks_per_seq) * block_size > INT_MAX) return PA_ERR_SHAPE;
    if (B > 65535) return PA_ERR_UNSUPPORTED;
    if (B == 0) return PA_OK;
    if (!out_host || !q_host || !k_new_host || !v_new_host || !k_cache || !v_cache || !context_lens_host ||
        (max_blocks_per_seq > 0 && !block_tables_host))
        return PA_ERR_NULL;
    const size_t ws = pa::plan_decode(B, Hq, Hkv, D, max_blocks_per_seq, block_size).ws_bytes;
    const HostStage s = host_stage(B, Hq, Hkv, D, max_blocks_per_seq, ws);
    if (!workspace || workspace_bytes < s.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PA_ERR_WORKSPACE;
    char *w = static_cast<char *>(workspace);
    const size_t qb = static_cast<size_t>(B) * Hq * D * 2, kb = static_cast<size_t>(B) * Hkv * D * 2;
    const size_t tb = static_cast<size_t>(B) * max_blocks_per_seq * 4;
    // inputs packed at the staged offsets (the layout pa_store_decode_host_layout gives) move in
    // one copy; otherwise one copy per input, in stream order before the launches
    const char *h = static_cast<const char *>(q_host);
    const bool packed = static_cast<const char *>(k_new_host) == h + (s.kn - s.q) &&
                        static_cast<const char *>(v_new_host) == h + (s.vn - s.q) &&
                        (tb == 0 || reinterpret_cast<const char *>(block_tables_host) == h + (s.bt - s.q)) &&
                        reinterpret_cast<const char *>(context_lens_host) == h + (s.cl - s.q);
    if (packed) {
        // page-locked and mapped: the SMs pull the span across; otherwise the copy engine
        const size_t span = s.cl - s.q + static_cast<size_t>(B) * 4;
        const void *dev_in = aligned16(h) ? pa::mapped_host(h, span) : nullptr;
        const cudaError_t e = dev_in ? pa::launch_stage(w + s.q, dev_in, span, false, stream)
                                     : cudaMemcpyAsync(w + s.q, h, span, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return PA_ERR_CUDA;
    } else if (cudaMemcpyAsync(w + s.q, q_host, qb, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(w + s.kn, k_new_host, kb, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(w + s.vn, v_new_host, kb, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        (tb > 0 && cudaMemcpyAsync(w + s.bt, block_tables_host, tb, cudaMemcpyHostToDevice, stream) != cudaSuccess) ||
        cudaMemcpyAsync(w + s.cl, context_lens_host, static_cast<size_t>(B) * 4, cudaMemcpyHostToDevice, stream) !=
            cudaSuccess)
        return PA_ERR_CUDA;
    st = pa_store_decode(w + s.out, w + s.q, w + s.kn, w + s.vn, k_cache, v_cache,
                         tb > 0 ? reinterpret_cast<const int32_t *>(w + s.bt) : nullptr, max_blocks_per_seq,
                         reinterpret_cast<const int32_t *>(w + s.cl), B, Hq, Hkv, D, block_size, num_blocks,
                         scale, dtype, ws > 0 ? w + s.ws : nullptr, ws, err, stream);
    if (st != PA_OK) return st;
    void *dev_out = aligned16(out_host) ? pa::mapped_host(out_host, qb) : nullptr;
    return from_cuda(dev_out ? pa::launch_stage(dev_out, w + s.out, qb, true, stream)
                             : cudaMemcpyAsync(out_host, w + s.out, qb, cudaMemcpyDeviceToHost, stream));
}

pa_status pa_prefill_varlen(void *out, const void *q, const void *k, const void *v,
                            const void *k_cache, const void *v_cache,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int S,
                            int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                            const int32_t *block_tables, int max_blocks_per_seq, int Hq, int Hkv,
                            int D, int block_size, int num_blocks, float scale, int causal,
                            pa_dtype dtype, int32_t *err, cudaStream_t stream) {
    if (!dtype_ok(dtype)) return PA_ERR_DTYPE;
    if (S < 0 || max_seqlen_q < 0 || total_q < 0 || (!block_tables && total_k < 0) ||
        (causal != 0 && causal != 1))
        return PA_ERR_SHAPE;
    pa_status st = check_heads(Hq, Hkv, D);
    if (st != PA_OK) return st;
    if (block_tables &&
        (block_size < 1 || max_blocks_per_seq < 1 || num_blocks < 1 ||
         static_cast<long long>(max_blocks_per_seq) * block_size > INT_MAX))
        return PA_ERR_SHAPE;
    if (S > 65535) return PA_ERR_UNSUPPORTED;
    if (S == 0 || max_seqlen_q == 0 || total_q == 0) return PA_OK;
    if (!out || !q || !cu_seqlens_q || !cu_seqlens_k) return PA_ERR_NULL;
    if (block_tables && static_cast<long long>(num_blocks) * block_size > INT_MAX)
        return PA_ERR_UNSUPPORTED;
    if (block_tables ? (!k_cache || !v_cache) : (!k || !v)) return PA_ERR_NULL;
    const void *kk = block_tables ? k_cache : k;
    const void *vv = block_tables ? v_cache : v;
    if (!aligned16(out) || !aligned16(q) || !aligned16(kk) || !aligned16(vv))
        return PA_ERR_UNSUPPORTED;
    pa::PrefillArgs a{};
    a.out = out;
    a.q = q;
    a.k = k;
    a.v = v;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.block_tables = block_tables;
    a.S = S;
    a.total_q = total_q;
    a.total_k = block_tables ? 0 : total_k;
    a.max_seqlen_q = max_seqlen_q;
    a.max_seqlen_k = max_seqlen_k;  // a hint for the work order only
    a.max_blocks = max_blocks_per_seq;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.block_size = block_size < 1 ? 1 : block_size;
    a.num_blocks = num_blocks;
    a.causal = causal;
    a.scale = scale;
    a.dtype = dtype;
    a.err = err;
    return from_cuda(pa::launch_prefill(a, stream));
}

}  // extern "C"
