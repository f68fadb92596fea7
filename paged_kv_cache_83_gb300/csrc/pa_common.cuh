// pa_common.cuh: small device helpers shared by the kernels of the paged KV-cache library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// ------------------------------------------------------------------------------------------
// element types
// ------------------------------------------------------------------------------------------

struct F16 {
    using T = __half;
    // two packed elements (one 32-bit word) to two floats
    static __device__ __forceinline__ float2 unpack2(uint32_t w) {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        return __half22float2(h);
    }
    static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

struct BF16 {
    using T = __nv_bfloat16;
    // bf16 is the top half of an fp32: widening is a shift / mask
    static __device__ __forceinline__ float2 unpack2(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

// 8 packed elements (16 bytes) to 8 floats
template <class E>
__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    float2 a = E::unpack2(u.x), b = E::unpack2(u.y), c = E::unpack2(u.z), d = E::unpack2(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// ------------------------------------------------------------------------------------------
// math
// ------------------------------------------------------------------------------------------

// 2^x with the SFU instruction (flushes subnormal results to zero; 2^-inf = 0)
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------------------------------
// memory
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy through L2 only; src_bytes == 0 writes 16 zero bytes and reads
// nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// streaming 16-byte global load (read once: do not keep in L1)
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void stg128(void *p, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void raise_err(int32_t *err, int bits) {
    if (err) atomicOr(err, bits);
}

// position -> (block index in the table row, offset in the block); block_size is a power of two
// when shift >= 0
struct BlockGeom {
    int block_size;
    int shift;  // log2(block_size) or -1
    __device__ __forceinline__ int block_of(int pos) const {
        return shift >= 0 ? (pos >> shift) : (pos / block_size);
    }
    __device__ __forceinline__ int offset_of(int pos) const {
        return shift >= 0 ? (pos & (block_size - 1)) : (pos % block_size);
    }
};

}  // namespace pa
