// device_common.cuh -- small device helpers shared by the kernels of libtg.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "tg_internal.h"

namespace tgi {

// d = c + sum_b a.u8[b] * b.s8[b]: unsigned bytes of a times signed bytes of b.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// d = c + sum_b a.s8[b] * b.s8[b].
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Sum of the four signed bytes of v.
__device__ __forceinline__ int byte_sum_s8(uint32_t v) { return dp4a_ss(v, 0x01010101u, 0); }

// 16-byte load that bypasses L1 allocation: each weight byte is read once.
__device__ __forceinline__ uint4 ldg_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int64_t warp_sum_i64(int64_t v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_i32(int v) { return __reduce_add_sync(0xffffffffu, v); }

// Programmatic dependent launch: allow the next kernel on the stream to start
// launching, and wait until the previous kernel on the stream has finished and
// its writes are visible. Both are no-ops for a kernel launched without the
// programmatic-serialization attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace tgi

// Each translation unit holds one device error word, set by a kernel that
// gives up a bounded wait; the host reads and clears it through the unit's
// take function.
#define TGI_DEFINE_DEVICE_ERROR(fn_name)                                                      \
    static __device__ int tgi_device_error_word = 0;                                          \
    namespace tgi {                                                                           \
    int fn_name(void *stream)                                                                 \
    {                                                                                         \
        int v = 0, zero = 0;                                                                  \
        cudaStream_t s = static_cast<cudaStream_t>(stream);                                  \
        if (cudaMemcpyFromSymbolAsync(&v, tgi_device_error_word, sizeof(int), 0,             \
                                      cudaMemcpyDeviceToHost, s) != cudaSuccess)              \
            return TG_ERR_CUDA;                                                               \
        if (cudaMemcpyToSymbolAsync(tgi_device_error_word, &zero, sizeof(int), 0,            \
                                    cudaMemcpyHostToDevice, s) != cudaSuccess)                \
            return TG_ERR_CUDA;                                                               \
        if (cudaStreamSynchronize(s) != cudaSuccess)                                          \
            return TG_ERR_CUDA;                                                               \
        return v ? TG_ERR_DEVICE : TG_OK;                                                     \
    }                                                                                         \
    }
