// wait_probe.cu: a test-only kernel for the library's bounded mbarrier wait.
//
// Built by the tests into its own shared library (tests/native/_build/libwait_probe.so), never
// into libpagedattn.so and never launched by a product call. It compiles the library's own wait
// (pa::mbar_wait from csrc/pa_common.cuh, 0.5 s limit) and the same give-up path the decode and
// prefill kernels take: on a wait that runs out, set PA_DEVERR_TIMEOUT in *err and return. The
// kernel issues no TMA, bulk copy or MMA, so nothing is in flight when it gives up.
#ifndef PA_TEST_HOOKS
#error "wait_probe.cu is test infrastructure: build it with -DPA_TEST_HOOKS"
#endif

#include "../../paged_kv_cache_83_gb300/csrc/pa_common.cuh"

namespace {

// One warp. An mbarrier expecting one arrival; with `arrive` lane 0 arrives (phase 0 completes and
// the wait returns at once), without it nothing ever arrives and every lane's wait must give up.
__global__ void wait_probe_kernel(int32_t *err, int arrive, unsigned long long *elapsed_ns) {
    __shared__ alignas(8) unsigned long long bar;
    const uint32_t b = pa::smem_addr(&bar);
    if (threadIdx.x == 0) {
        pa::mbar_init(b, 1);
        pa::fence_mbar_init();
    }
    __syncwarp();
    if (arrive && threadIdx.x == 0) pa::mbar_arrive(b);
    const uint64_t t0 = pa::globaltimer_ns();
    const bool ok = pa::mbar_wait(b, 0);  // every lane waits, as in the kernels
    __syncwarp();
    const unsigned all_ok = __all_sync(0xffffffffu, ok);
    if (threadIdx.x == 0) {
        *elapsed_ns = pa::globaltimer_ns() - t0;
        if (!all_ok) pa::raise_err(err, PA_DEVERR_TIMEOUT);
    }
}

}  // namespace

// Launches the probe on `stream` (err, elapsed_ns: device pointers). 0 on a successful launch,
// else the CUDA error code.
extern "C" int pa_test_wait_probe(int32_t *err, int arrive, unsigned long long *elapsed_ns,
                                  cudaStream_t stream) {
    wait_probe_kernel<<<1, 32, 0, stream>>>(err, arrive, elapsed_ns);
    return static_cast<int>(cudaGetLastError());
}
