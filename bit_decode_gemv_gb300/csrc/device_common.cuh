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

// L2 policy for data read once per call (a weight stream larger than L2): its
// lines are the first evicted, so the stream recycles a small part of L2 and the
// rest -- kernel code, activations, per-row sums, histograms -- stays resident.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint4 ldg_stream(const void *p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
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

// ---------------------------------------------------------------------------
// mbarriers and bulk (TMA) copies into shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Arrive once on the mbarrier and add `bytes` to the transfer count its phase waits for.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bulk (TMA) copy global -> shared, completing `bytes` on the mbarrier.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// The same with an L2 cache policy (l2_evict_first_policy for a stream read once).
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// One test of phase `parity` of an mbarrier (true once the phase has completed).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// ---------------------------------------------------------------------------
// Warp-level MMAs (16x8x16, fp32 accumulate) used where a few tokens, or the
// LNS8 class sums, make a contraction too small for the tensor-memory MMA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Exact fp32 integer of magnitude at most 2^22 -> int (through the 1.5 * 2^23
// magic number, so no conversion instruction is needed).
__device__ __forceinline__ int int_of_f32(float v) { return __float_as_int(v + 12582912.0f) - 0x4B400000; }

// ---------------------------------------------------------------------------
// LNS8 fragment layout -> compact mask words. Entry j (16 bytes) of a row pair
// (q, q + 8) of a 16-row block holds, in words u = 0..3, the W_nonzero bits of
// both rows in bytes 0 and 2 and the W_negative bits in bytes 1 and 3 (see
// tg.h). Two byte permutes and two shift-and-merge steps give one 32-lane
// W_nonzero and one W_negative word per row; lns8_lane_col names the group
// lane of each bit, the same for both rows.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int lns8_lane_col(int j, int bit)
{
    const int x = 7 - (bit & 7);
    const int c = (x >> 2) + 2 * ((bit >> 3) & 1) + 4 * (x & 1);
    return 16 * c + 2 * j + 8 * ((x >> 1) & 1) + (bit >> 4);
}

__device__ __forceinline__ void lns8_compact_words(uint4 w, uint32_t &nz0, uint32_t &ng0, uint32_t &nz1,
                                                   uint32_t &ng1)
{
    const uint32_t nza0 = __byte_perm(w.x, w.y, 0x6240), nga0 = __byte_perm(w.x, w.y, 0x7351);
    const uint32_t nza1 = __byte_perm(w.z, w.w, 0x6240), nga1 = __byte_perm(w.z, w.w, 0x7351);
    nz0 = (nza0 & 0xAAAAAAAAu) | ((nza1 >> 1) & 0x55555555u);
    nz1 = ((nza0 << 1) & 0xAAAAAAAAu) | (nza1 & 0x55555555u);
    ng0 = (nga0 & 0xAAAAAAAAu) | ((nga1 >> 1) & 0x55555555u);
    ng1 = ((nga0 << 1) & 0xAAAAAAAAu) | (nga1 & 0x55555555u);
}

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
