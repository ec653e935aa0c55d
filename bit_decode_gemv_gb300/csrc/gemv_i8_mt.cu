// gemv_i8_mt.cu -- the ternary (or binary Q1_0) GEMV for a few tokens on the
// CUDA cores (integer_engine.md §4.1/§4.2 with §4.4 int8 activations):
//
//     y[m][r] = sum_g arshift( d[r][g] * P[m][r][g], frac ),
//     P = sum_{i in g} t[r][i] * x[m][i]
//
// The lane arithmetic is the batch-1 kernel's (gemv_i8.cu): a masked mask word
// is a dp4a operand of four unsigned bytes (t + 2) * 4^j (ternary) or
// 2^j * [t = +1] (Q1_0). What changes with several tokens is that the masked
// words depend on the weights only: each lane forms a group's 32 of them once
// and reuses them for every token, so a token costs one dp4a per four weights
// and one broadcast 16-byte shared load per sixteen, and the weights are read
// from memory once for all tokens.
//
// int64 fixed-point activations (integer engine §4.4; exact modulo 2^64 as
// its §5 states): each x is split into signed base-256 digits s_0..s_7 in
// [-128, 127] with x = sum_l 256^l s_l (mod 2^64) -- the bytes of
// (x + 0x8080...80) XOR 0x8080...80 -- and every digit plane is an ordinary
// int8 activation vector for the arithmetic above. Per group and token the
// planes' P_l are recombined as sum_l P_l 2^(8l) in wrapping 64-bit
// arithmetic, multiplied by d, floored and summed, all modulo 2^64. Only the
// planes up to the highest nonzero digit of the staged tokens are processed
// (one plane for activations in int8 range, three for magnitudes below 2^23).
//
// tg_gemv_i8 sends this kernel calls of two or more tokens with int64
// activations (and one token whose digit planes do not fit the one-token
// kernel of gemv_i8.cu), and int8 calls of two to four tokens whose
// activations do not fit the shared memory of the few-token kernels in
// gemv_i8.cu (this one stages tokens in chunks).
//
// Mapping: one CTA per 32-row tile (lane l of every warp owns row 32T + l),
// the CTA's warps split the groups GPW at a time with every mask load of a
// batch issued before its compute, as in the batch-1 kernel. The tokens are
// staged in shared memory in chunks that fit; each (token, group) result is
// added into the token's per-row int64 sum with a shared-memory atomic, an
// integer sum, so the order does not matter.

#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "tg.h"
#include "tg_internal.h"

namespace {

using tgi::dp4a_us;
using tgi::kTileRows;

constexpr int kMaxWarps = 16;
constexpr size_t kStageBytes = 144 * 1024;   // token activations staged per chunk

__device__ __forceinline__ uint32_t and_xor(uint32_t w, uint32_t mask, uint32_t flip)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(w), "r"(mask), "r"(flip));
    return r;
}

// The 32 dp4a operands of one row's group. Ternary: word u (0..7) column j
// (0..3) -> (w_u & (3 << 2j per byte)) ^ (2 << 2j per byte) = (t + 2) * 4^j.
// Q1_0: word u (0..3) column j (0..7) -> w_u & (1 << j per byte).
template <bool kQ1>
__device__ __forceinline__ void masked_words(const uint4 &m0, const uint4 &m1, uint32_t (&wm)[32])
{
    if constexpr (kQ1) {
        const uint32_t w[4] = {m0.x, m0.y, m0.z, m0.w};
#pragma unroll
        for (int u = 0; u < 4; u++)
#pragma unroll
            for (int j = 0; j < 8; j++)
                wm[8 * u + j] = w[u] & (0x01010101u << j);
    } else {
        const uint32_t w[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
        for (int u = 0; u < 8; u++)
#pragma unroll
            for (int j = 0; j < 4; j++)
                wm[4 * u + j] = and_xor(w[u], 0x03030303u << (2 * j), 0x02020202u << (2 * j));
    }
}

// P of one token for one row's group from its masked words; xg = the group's
// 128 activations in shared memory, tg = their sum.
template <bool kQ1>
__device__ __forceinline__ int group_p(const uint32_t (&wm)[32], const int8_t *xg, int tg)
{
    if constexpr (kQ1) {
        int a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const uint4 lo = *reinterpret_cast<const uint4 *>(xg + 32 * u);
            const uint4 hi = *reinterpret_cast<const uint4 *>(xg + 32 * u + 16);
            const uint32_t xv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int j = 0; j < 8; j++)
                a[j] = dp4a_us(wm[8 * u + j], xv[j], a[j]);
        }
        int pos = 0;
#pragma unroll
        for (int j = 0; j < 8; j++)
            pos += a[j] >> j;
        return 2 * pos - tg;   // 2 * pos_sum - block_total
    } else {
        int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(xg + 16 * u);
            a0 = dp4a_us(wm[4 * u + 0], xv.x, a0);
            a1 = dp4a_us(wm[4 * u + 1], xv.y, a1);
            a2 = dp4a_us(wm[4 * u + 2], xv.z, a2);
            a3 = dp4a_us(wm[4 * u + 3], xv.w, a3);
        }
        return a0 + (a1 >> 2) + (a2 >> 4) + (a3 >> 6) - 2 * tg;
    }
}

// The signed base-256 digits of x (mod 2^64), byte l = digit l.
__device__ __forceinline__ uint64_t signed_digits(uint64_t x)
{
    return (x + 0x8080808080808080ull) ^ 0x8080808080808080ull;
}

template <bool kX64>
__host__ __device__ constexpr int planes_max() { return kX64 ? 8 : 1; }

template <int GPW, bool kQ1, bool kX64>
__global__ void __launch_bounds__(kMaxWarps * 32)
gemv_i8_mt_kernel(const uint4 *__restrict__ masks, const int32_t *__restrict__ scales,
                  const void *__restrict__ xv, int64_t *__restrict__ y, int N, int G, int M, int chunk,
                  int frac)
{
    constexpr int kChunks = kQ1 ? 32 : 64;   // uint4 per (tile, group)
    constexpr int kPlanes = planes_max<kX64>();
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int top_plane;
    const int K = G * 128;
    const size_t vrows = (size_t)chunk * kPlanes;                                      // staged activation rows
    int8_t *xs = reinterpret_cast<int8_t *>(smem);                                   // [vrows][K]
    int *tsum = reinterpret_cast<int *>(smem + vrows * K);                             // [vrows][G]
    unsigned long long *ysum = reinterpret_cast<unsigned long long *>(
        smem + vrows * K + ((vrows * G * 4 + 15) & ~(size_t)15));                      // [chunk][32]
    const int8_t *x = static_cast<const int8_t *>(xv);
    const uint64_t *x64 = static_cast<const uint64_t *>(xv);

    const int tile = blockIdx.x;
    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint4 *tmask = masks + (size_t)tile * G * kChunks;
    const int32_t *tscale = scales + (size_t)tile * G * kTileRows;
    const int row = tile * kTileRows + lane;

    for (int m0 = 0; m0 < M; m0 += chunk) {
        const int mc = min(chunk, M - m0);
        // this warp's first batch of groups: every load in flight before the staging
        uint4 r0[GPW], r1[GPW];
        int32_t dg[GPW];
        auto load_batch = [&](int g0) {
#pragma unroll
            for (int j = 0; j < GPW; j++) {
                const int g = g0 + j * nwarps;
                if (g < G) {
                    r0[j] = tgi::ldg_stream(tmask + (size_t)g * kChunks + lane);
                    r1[j] = kQ1 ? make_uint4(0, 0, 0, 0) : tgi::ldg_stream(tmask + (size_t)g * kChunks + 32 + lane);
                    dg[j] = __ldg(tscale + (size_t)g * kTileRows + lane);
                } else {
                    r0[j] = r1[j] = make_uint4(0, 0, 0, 0);
                    dg[j] = 0;
                }
            }
        };
        load_batch(warp);
        if (m0 == 0) {
            // launched as a programmatic dependent (constant weights): the next
            // kernel may start now; x and y are touched only after the wait
            tgi::pdl_launch_dependents();
            tgi::pdl_wait();
        }

        // stage the chunk's activations (row t * planes + l holds digit plane l
        // of token t), their group totals, zero the row sums
        int planes = 1;
        if constexpr (kX64) {
            const uint64_t *xc = x64 + (size_t)m0 * K;
            if (threadIdx.x == 0)
                top_plane = 0;
            __syncthreads();
            // (loads in batches of kScanBatch per thread, issued before they are used:
            // one at a time they were a chain of L2 round trips)
            int top = 0;
            constexpr int kScanBatch = 4;
            for (int base = threadIdx.x; base < mc * K; base += kScanBatch * blockDim.x) {
                uint64_t raw[kScanBatch];
#pragma unroll
                for (int u = 0; u < kScanBatch; u++) {
                    const int i = base + u * blockDim.x;
                    raw[u] = i < mc * K ? __ldg(reinterpret_cast<const unsigned long long *>(xc) + i) : 0ull;
                }
#pragma unroll
                for (int u = 0; u < kScanBatch; u++) {
                    const uint64_t dv = signed_digits(raw[u]);   // 0 for x = 0
                    if (dv)
                        top = max(top, (63 - __clzll((long long)dv)) >> 3);
                }
            }
            top = (int)__reduce_max_sync(0xffffffffu, (unsigned)top);
            if (lane == 0)
                atomicMax(&top_plane, top);
            __syncthreads();
            planes = top_plane + 1;
#pragma unroll 2
            for (int i = threadIdx.x; i < mc * (K / 4); i += blockDim.x) {
                const int t = i / (K / 4), c = i - t * (K / 4);
                const ulonglong2 *src = reinterpret_cast<const ulonglong2 *>(xc + (size_t)t * K + 4 * c);
                const ulonglong2 v01 = __ldg(src), v23 = __ldg(src + 1);
                const uint64_t dv[4] = {signed_digits(v01.x), signed_digits(v01.y), signed_digits(v23.x),
                                        signed_digits(v23.y)};
                for (int l = 0; l < planes; l++) {
                    const uint32_t word = (uint32_t)((dv[0] >> (8 * l)) & 0xFF) |
                                          ((uint32_t)((dv[1] >> (8 * l)) & 0xFF) << 8) |
                                          ((uint32_t)((dv[2] >> (8 * l)) & 0xFF) << 16) |
                                          ((uint32_t)((dv[3] >> (8 * l)) & 0xFF) << 24);
                    *reinterpret_cast<uint32_t *>(xs + ((size_t)t * planes + l) * K + 4 * c) = word;
                }
            }
            __syncthreads();
            for (int vg = warp; vg < mc * planes * G; vg += nwarps) {
                const uint32_t v = *(reinterpret_cast<const uint32_t *>(xs + (size_t)vg * 128) + lane);
                const int s = tgi::warp_sum_i32(tgi::byte_sum_s8(v));
                if (lane == 0)
                    tsum[vg] = s;
            }
        } else {
            const uint4 *xsrc = reinterpret_cast<const uint4 *>(x + (size_t)m0 * K);
            for (int i = threadIdx.x; i < mc * K / 16; i += blockDim.x)
                reinterpret_cast<uint4 *>(xs)[i] = __ldg(xsrc + i);
            for (int tgx = warp; tgx < mc * G; tgx += nwarps) {
                const uint32_t v =
                    __ldg(reinterpret_cast<const uint32_t *>(x + (size_t)m0 * K + (size_t)tgx * 128) + lane);
                const int s = tgi::warp_sum_i32(tgi::byte_sum_s8(v));
                if (lane == 0)
                    tsum[tgx] = s;
            }
        }
        for (int i = threadIdx.x; i < mc * 32; i += blockDim.x)
            ysum[i] = 0ull;
        __syncthreads();

        for (int g0 = warp;;) {
#pragma unroll
            for (int j = 0; j < GPW; j++) {
                const int g = g0 + j * nwarps;
                if (g < G) {
                    uint32_t wm[32];
                    masked_words<kQ1>(r0[j], r1[j], wm);
                    const int64_t d = dg[j];
                    for (int t = 0; t < mc; t++) {
                        if constexpr (kX64) {
                            // sum_l P_l 2^(8l), times d, floored: all modulo 2^64
                            uint64_t p64 = 0;
                            for (int l = 0; l < planes; l++) {
                                const int vt = t * planes + l;
                                const int P = group_p<kQ1>(wm, xs + (size_t)vt * K + (size_t)g * 128, tsum[vt * G + g]);
                                p64 += (uint64_t)(int64_t)P << (8 * l);
                            }
                            const int64_t v = (int64_t)(p64 * (uint64_t)d);
                            atomicAdd(&ysum[t * 32 + lane], (unsigned long long)(v >> frac));
                        } else {
                            const int P = group_p<kQ1>(wm, xs + (size_t)t * K + (size_t)g * 128, tsum[t * G + g]);
                            atomicAdd(&ysum[t * 32 + lane], (unsigned long long)((d * (int64_t)P) >> frac));
                        }
                    }
                }
            }
            g0 += nwarps * GPW;
            if (g0 >= G)
                break;
            load_batch(g0);
        }
        __syncthreads();
        for (int t = warp; t < mc; t += nwarps)
            if (row < N)
                y[(size_t)(m0 + t) * N + row] = (int64_t)ysum[t * 32 + lane];
        __syncthreads();   // xs and ysum are reused by the next chunk
    }
}

size_t mt_smem_bytes(int G, int chunk, int planes)
{
    const size_t rows = (size_t)chunk * planes;
    return rows * G * 128 + ((rows * G * 4 + 15) & ~(size_t)15) + (size_t)chunk * 32 * 8;
}

template <int GPW, bool kQ1, bool kX64>
cudaError_t launch_mt(const uint4 *masks, const int32_t *scales, const void *x, int64_t *y, int N, int G,
                      int tiles, int M, int frac, bool pdl, cudaStream_t s)
{
    auto kern = gemv_i8_mt_kernel<GPW, kQ1, kX64>;
    constexpr int kPlanes = planes_max<kX64>();
    int warps = (G + GPW - 1) / GPW;
    if (warps > kMaxWarps)
        warps = kMaxWarps;
    int chunk = (int)(kStageBytes / (kPlanes * ((size_t)G * 128 + 4 * (size_t)G) + 256));
    if (chunk > M)
        chunk = M;
    if (chunk < 1)
        chunk = 1;
    const size_t smem = mt_smem_bytes(G, chunk, kPlanes);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles);
    cfg.blockDim = dim3(warps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, masks, scales, x, y, N, G, M, chunk, frac);
}

template <bool kX64>
cudaError_t dispatch_mt(const uint4 *masks, const int32_t *scales, const void *x, int64_t *y, int N, int G,
                        int tiles, int M, bool q1, int frac, bool pdl, cudaStream_t s)
{
    if (q1)
        return G <= 32 ? launch_mt<2, true, kX64>(masks, scales, x, y, N, G, tiles, M, frac, pdl, s)
                       : launch_mt<4, true, kX64>(masks, scales, x, y, N, G, tiles, M, frac, pdl, s);
    return G <= 32 ? launch_mt<2, false, kX64>(masks, scales, x, y, N, G, tiles, M, frac, pdl, s)
                   : launch_mt<4, false, kX64>(masks, scales, x, y, N, G, tiles, M, frac, pdl, s);
}

}  // namespace

namespace tgi {

int gemv_i8_mt(const uint4 *masks, const int32_t *scales, const void *x, int64_t *y, int N, int G, int tiles,
               int M, bool q1, bool x64, int frac, bool pdl, cudaStream_t s)
{
    const size_t planes = x64 ? 8 : 1;
    if (planes * ((size_t)G * 128 + 4 * (size_t)G) + 256 > kStageBytes)
        return TG_ERR_SHAPE;   // one token's activation planes must fit
    const cudaError_t e = x64 ? dispatch_mt<true>(masks, scales, x, y, N, G, tiles, M, q1, frac, pdl, s)
                              : dispatch_mt<false>(masks, scales, x, y, N, G, tiles, M, q1, frac, pdl, s);
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace tgi
