// stage.cu: moves a step's inputs from host memory into the device workspace and its output back,
// with the SMs' own loads and stores instead of the copy engine.
//
// Source: "nano-vLLM Part 4" section 3 (every decode step ships its new inputs to the device and
// reads its result back, while the KV cache stays resident).
//
// Host memory that is page-locked and registered with CUDA is mapped into the device's address
// space; on a GB300 the SMs reach it over the chip-to-chip link. A copy of a couple of MB as one
// copy-engine transfer costs about as much as the bytes would take at 100 GB/s; the same bytes
// moved by a few hundred CTAs with 16-byte accesses in flight everywhere take a fraction of that.
// Host-side loads bypass the caches (each step's inputs are new); stores write through.
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kStageThreads = 256;
constexpr int kStageUnroll = 4;

// Copies `bytes` bytes (a multiple of 4) from src to dst, both 16-byte aligned. Launched as a
// programmatic dependent it first waits for the grids it depends on; either way it lets the next
// grid launch early (that grid waits for this one before it reads what this one writes).
__global__ void __launch_bounds__(kStageThreads) stage_kernel(char *__restrict__ dst,
                                                             const char *__restrict__ src,
                                                             long long bytes) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const long long n16 = bytes >> 4;
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    const long long stride = static_cast<long long>(gridDim.x) * kStageThreads;
    long long i = static_cast<long long>(blockIdx.x) * kStageThreads + threadIdx.x;
    for (; i + (kStageUnroll - 1) * stride < n16; i += kStageUnroll * stride) {
        uint4 v[kStageUnroll];
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) v[u] = __ldcv(s + i + u * stride);
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) __stwt(d + i + u * stride, v[u]);
    }
    for (; i < n16; i += stride) __stwt(d + i, __ldcv(s + i));
    const int tail4 = static_cast<int>((bytes & 15) >> 2);
    if (blockIdx.x == 0 && threadIdx.x < tail4) {
        const unsigned *s4 = reinterpret_cast<const unsigned *>(src + (n16 << 4));
        unsigned *d4 = reinterpret_cast<unsigned *>(dst + (n16 << 4));
        __stwt(d4 + threadIdx.x, __ldcv(s4 + threadIdx.x));
    }
}

}  // namespace

void *mapped_host(const void *p, size_t bytes) {
    if (!p || bytes == 0) return nullptr;
    cudaPointerAttributes a{}, z{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
    const char *last = static_cast<const char *>(p) + (bytes - 1);
    if (cudaPointerGetAttributes(&z, last) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (z.type != cudaMemoryTypeHost || !z.devicePointer ||
        static_cast<char *>(z.devicePointer) != static_cast<char *>(a.devicePointer) + (bytes - 1))
        return nullptr;
    return a.devicePointer;
}

cudaError_t launch_stage(void *dst, const void *src, size_t bytes, bool dependent, cudaStream_t stream) {
    if (bytes == 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u || (bytes & 3u))
        return cudaErrorInvalidValue;
    const long long n16 = static_cast<long long>(bytes >> 4);
    const long long per_cta = static_cast<long long>(kStageThreads) * kStageUnroll;
    long long grid = (n16 + per_cta - 1) / per_cta;
    const long long cap = 2LL * device_sm_count();
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kStageThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, stage_kernel, static_cast<char *>(dst), static_cast<const char *>(src),
                              static_cast<long long>(bytes));
}

}  // namespace pa
