// decode_noalloc.cu: pa_decode_noalloc, a decode entry point that allocates nothing.
//
// Some callers cannot hand the library scratch memory: a host framework that owns every device
// allocation and gives its plugins none, a process whose device memory is already fully
// reserved by another allocator, or a step loop where cudaMalloc's implicit device
// synchronisation is not acceptable. For them the split-K partial results of pa_decode live in
// one file-scope device array of fixed size, which every GPU that loads this library keeps
// until the process exits. Everything else is pa_decode itself, called with that array as its
// workspace.
#include <atomic>

#include "pa_internal.h"

namespace {

// Split-K scratch shared by every pa_decode_noalloc call on a device.
static __device__ __align__(256) unsigned char g_decode_scratch[PA_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
// device address of g_decode_scratch, per device; host threads may fill a slot concurrently (they
// all store the same address), so the slots are atomics
std::atomic<void *> g_scratch_ptr[kMaxDevices];

// The host-side name g_decode_scratch is not a device address; look the address up once per
// device, with that device current, and keep it. A cudaDeviceReset (or a reset of the primary
// context) reloads the module, which may move the array: the kept address is then stale, which
// the header states.
pa_status scratch_for_current_device(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *ptr = p;
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void *out, const void *q, const void *k_cache,
                                       const void *v_cache, const int32_t *block_tables,
                                       int max_blocks_per_seq, const int32_t *context_lens, int B,
                                       int Hq, int Hkv, int D, int block_size, int num_blocks,
                                       float scale, pa_dtype dtype, int32_t *err,
                                       cudaStream_t stream) {
    void *scratch = nullptr;
    pa_status st = scratch_for_current_device(&scratch);
    if (st != PA_OK) return st;
    // pa_decode checks every argument and returns PA_ERR_WORKSPACE when these sizes need more
    // scratch than the fixed array holds. The partial results it keeps there are written before
    // they are read, so nothing has to be cleared between calls.
    // (one CTA per SM for every shape: the fixed scratch is sized for that)
    return pa::decode_entry(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, B,
                            Hq, Hkv, D, block_size, num_blocks, scale, dtype, scratch,
                            PA_DECODE_NOALLOC_SCRATCH_BYTES, err, stream, false);
}
