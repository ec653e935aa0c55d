// gemv_i8_hmma.cu -- the ternary (or binary Q1_0) GEMV for a few tokens on the
// tensor cores through warp-level fp16 MMAs (integer_engine.md §4.1/§4.2 with
// §4.4 int8 activations and its §5 tensor-core mapping):
//
//     y[m][r] = sum_g arshift( d[r][g] * P[m][r][g], frac ),
//     P = sum_{i in g} t[r][i] * x[m][i]
//
// Exactness: t (-1, 0, +1) and int8 x are exact fp16 values, every product is
// exact, and one group's partial sums are integers of magnitude at most
// 128 * 128 = 2^14, exact in the fp32 accumulator. So a 16x8x16 MMA of
// (16 rows x 16 lanes of t) by (16 lanes x 8 tokens of x), accumulated over
// the group's eight K = 16 steps, yields P exactly; it is converted to an
// integer, scaled by d, floored by 2^frac and summed in int64 per group.
//
// Why warp MMAs here: with a handful of tokens the weights are the only large
// operand, each weight is used by M tokens only, and a 16x8x16 step covers
// 2048 multiply-adds for four A registers that a lane builds from its mask
// words with a shift, two masks and two byte permutes. The tensor-memory MMA
// of gemv_i8_mma.cu has a fixed cost per instruction that dominates at this N.
//
// A operand straight from the I8 mask layout: lane (q, t) of a warp needs,
// for K step s (= mask word s of a row: lanes 16s .. 16s + 15), the weights of
// rows q and q + 8 of a 16-row block at lanes 2t, 2t + 1, 2t + 8, 2t + 9. In
// word s lane 4j + b sits at bits 8b + 2j (W_nonzero) and 8b + 2j + 1
// (W_negative); after a shift by 16 (t & 1) + 2 (t >> 1) the four codes sit at
// bits 0, 8, 4 and 12, and a byte permute of the table (0, 0x3C, 0, 0xBC) by
// those codes in selector nibbles 1 and 3 gives the fp16 pair (0, +1.0, -1.0
// for codes 0, 1, 3). Q1_0 words (lane 32u + 4j + b at bit 8b + j) work the
// same way with one bit and the table (0, 0xBC, 0, 0x3C).
//
// B operand: the tokens' activations, staged once per CTA as fp16 rows in
// shared memory (16-byte global loads, an exact int8 -> fp16 conversion; the
// row stride is padded by 16 bytes so that the eight token rows of a fragment
// fall in different banks), in chunks of token tiles that fit. Lane (q, t) of
// K step s and token tile nt reads x[8 nt + q][16 s + 2t, +1] and
// [16 s + 2t + 8, +9] with two 32-bit loads. Tokens past M are zero rows.
//
// Mapping: one CTA per 32-row tile; warp w takes the tile's 16-row block w & 1
// and groups w >> 1, w >> 1 + W / 2, ...; its int64 sums stay in registers
// across its groups and are added into the CTA's per-(row, token) sums with
// shared-memory atomics at the end of each token chunk.

#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "tg.h"
#include "tg_internal.h"

namespace {

using tgi::kTileRows;

constexpr int kWarps = 8;
constexpr int kStageLoads = 8;               // activation loads per thread in flight while staging
constexpr size_t kFragBudget = 200 * 1024;   // shared memory for the B fragments of one chunk

// fp16 pair selected by the 2-bit codes in selector nibbles 1 and 3.
__device__ __forceinline__ uint32_t tern_pair(uint32_t sel) { return __byte_perm(0xBC003C00u, 0u, sel); }
__device__ __forceinline__ uint32_t q1_pair(uint32_t sel) { return __byte_perm(0x3C00BC00u, 0u, sel); }

// Two int8 (bytes sel_lo, sel_hi of v, given as a byte-permute selector) ->
// exact fp16 pair: x ^ 0x80 = x + 128 under the exponent byte 0x64 is
// 1024 + x + 128, minus 1152.
__device__ __forceinline__ uint32_t fp16x2_of_s8(uint32_t v, uint32_t sel)
{
    const uint32_t b = __byte_perm(v ^ 0x80808080u, 0x64646464u, sel);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(b), "r"(0x64806480u));
    return r;
}

// Sixteen int8 -> sixteen fp16, in order.
__device__ __forceinline__ void fp16_of_s8x16(uint4 v, uint4 &lo, uint4 &hi)
{
    lo = make_uint4(fp16x2_of_s8(v.x, 0x5140u), fp16x2_of_s8(v.x, 0x7362u), fp16x2_of_s8(v.y, 0x5140u),
                    fp16x2_of_s8(v.y, 0x7362u));
    hi = make_uint4(fp16x2_of_s8(v.z, 0x5140u), fp16x2_of_s8(v.z, 0x7362u), fp16x2_of_s8(v.w, 0x5140u),
                    fp16x2_of_s8(v.w, 0x7362u));
}

template <bool kQ1, int NT>
__global__ void __launch_bounds__(kWarps * 32)
gemv_i8_hmma_kernel(const uint4 *__restrict__ masks, const int32_t *__restrict__ scales,
                    const int8_t *__restrict__ x, int64_t *__restrict__ y, int N, int G, int M, int frac)
{
    constexpr int kChunks = kQ1 ? 32 : 64;   // uint4 per (tile, group)
    extern __shared__ __align__(16) unsigned char smem[];
    const int K = G * 128;
    const int stride = 2 * K + 16;   // bytes per fp16 token row (padded: see above)
    unsigned char *xs = smem;                                                                   // [8 NT][stride]
    unsigned long long *ysum = reinterpret_cast<unsigned long long *>(smem + (size_t)8 * NT * stride);  // [32][8 NT]

    const int tile = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = lane >> 2, t = lane & 3;
    const int blk = warp & 1;                  // 16-row block of the tile
    const int r0 = 16 * blk + q;               // tile-local rows r0 and r0 + 8
    const uint4 *tmask = masks + (size_t)tile * G * kChunks;
    const int32_t *tscale = scales + (size_t)tile * G * kTileRows;
    const uint32_t sh = kQ1 ? 16u * (t & 1) + (t >> 1) : 16u * (t & 1) + 2u * (t >> 1);

    for (int m0 = 0; m0 < M; m0 += 8 * NT) {
        const int mc = min(8 * NT, M - m0);
        // rows r0 and r0 + 8: mask words and scales of the warp's next group,
        // always one group ahead of the compute (the first one in flight while
        // the activations are staged)
        uint4 na0 = make_uint4(0u, 0u, 0u, 0u), na1 = na0, nb0 = na0, nb1 = na0;
        int32_t nda = 0, ndb = 0;
#define TG_HMMA_LOAD_GROUP(gg)                                                              \
    if ((gg) < G) {                                                                         \
        const uint4 *src = tmask + (size_t)(gg) * kChunks;                                  \
        na0 = tgi::ldg_stream(src + r0);                                                    \
        nb0 = tgi::ldg_stream(src + r0 + 8);                                                \
        if (!kQ1) {                                                                         \
            na1 = tgi::ldg_stream(src + 32 + r0);                                           \
            nb1 = tgi::ldg_stream(src + 32 + r0 + 8);                                       \
        }                                                                                   \
        nda = __ldg(tscale + (size_t)(gg) * kTileRows + r0);                                \
        ndb = __ldg(tscale + (size_t)(gg) * kTileRows + r0 + 8);                            \
    }
        TG_HMMA_LOAD_GROUP(warp >> 1)
        if (m0 == 0) {
            // launched as a programmatic dependent (constant weights): x and y
            // are touched only after the wait for the previous kernel
            tgi::pdl_wait();
        }
        // the chunk's activations as fp16 rows (rows past M are zero): eight
        // 16-byte loads per thread in flight at a time, then their conversion
        const int per_row = K / 16;
        const int items = 8 * NT * per_row;
        for (int base = threadIdx.x; base < items; base += kStageLoads * blockDim.x) {
            uint4 raw[kStageLoads];
#pragma unroll
            for (int u = 0; u < kStageLoads; u++) {
                const int i = base + u * blockDim.x;
                const int tok = i / per_row, c = i - tok * per_row;
                raw[u] = make_uint4(0u, 0u, 0u, 0u);
                if (i < items && tok < mc)
                    raw[u] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(m0 + tok) * K) + c);
            }
#pragma unroll
            for (int u = 0; u < kStageLoads; u++) {
                const int i = base + u * blockDim.x;
                if (i < items) {
                    const int tok = i / per_row, c = i - tok * per_row;
                    uint4 lo, hi;
                    fp16_of_s8x16(raw[u], lo, hi);
                    uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)tok * stride + 32 * c);
                    dst[0] = lo;
                    dst[1] = hi;
                }
            }
        }
        for (int i = threadIdx.x; i < 32 * 8 * NT; i += blockDim.x)
            ysum[i] = 0ull;
        __syncthreads();
        // the next kernel may launch once this CTA's activations are staged
        // (measured against releasing it right after the first weight loads:
        // 2560 x 2560 at M = 5 / 12: 6.24 / 9.59 -> 5.13 / 7.09 us per call,
        // the larger shapes within 1 %): fewer calls in flight at once
        if (m0 == 0)
            tgi::pdl_launch_dependents();

        int64_t acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int c = 0; c < 4; c++)
                acc[nt][c] = 0;

        for (int g = warp >> 1; g < G; g += kWarps / 2) {
            const uint4 wa[2] = {na0, na1}, wb[2] = {nb0, nb1};
            const int64_t da = nda, db = ndb;
            TG_HMMA_LOAD_GROUP(g + kWarps / 2)
            const uint32_t A[8] = {wa[0].x, wa[0].y, wa[0].z, wa[0].w, wa[1].x, wa[1].y, wa[1].z, wa[1].w};
            const uint32_t B[8] = {wb[0].x, wb[0].y, wb[0].z, wb[0].w, wb[1].x, wb[1].y, wb[1].z, wb[1].w};

            // two accumulator chains (even and odd K steps) per token tile; each
            // is an integer of magnitude at most 2^14, so their sum is exact
            float d[NT][4], e[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
#pragma unroll
                for (int c = 0; c < 4; c++)
                    d[nt][c] = e[nt][c] = 0.f;
#pragma unroll
            for (int s = 0; s < 8; s++) {
                uint32_t a0, a1, a2, a3;
                if constexpr (kQ1) {
                    // word s >> 1 holds lanes 32 (s >> 1) .. + 31; K step s is its
                    // half s & 1 (bits 4 (s & 1) + j of each byte)
                    const uint32_t va = A[s >> 1] >> (sh + 4u * (s & 1));
                    const uint32_t vb = B[s >> 1] >> (sh + 4u * (s & 1));
                    a0 = q1_pair(0x1010u | ((va << 5) & 0x2020u));
                    a1 = q1_pair(0x1010u | ((vb << 5) & 0x2020u));
                    a2 = q1_pair(0x1010u | ((va << 3) & 0x2020u));
                    a3 = q1_pair(0x1010u | ((vb << 3) & 0x2020u));
                } else {
                    const uint32_t va = A[s] >> sh, vb = B[s] >> sh;
                    a0 = tern_pair((va << 4) & 0x3030u);
                    a1 = tern_pair((vb << 4) & 0x3030u);
                    a2 = tern_pair(va & 0x3030u);
                    a3 = tern_pair(vb & 0x3030u);
                }
                const unsigned char *xk = xs + (size_t)q * stride + 2 * (128 * g + 16 * s + 2 * t);
#pragma unroll
                for (int nt = 0; nt < NT; nt++) {
                    const unsigned char *xr = xk + (size_t)8 * nt * stride;
                    tgi::mma_f16_16816((s & 1) ? e[nt] : d[nt], a0, a1, a2, a3, *reinterpret_cast<const uint32_t *>(xr),
                                  *reinterpret_cast<const uint32_t *>(xr + 16));
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
#pragma unroll
                for (int c = 0; c < 4; c++)
                    d[nt][c] += e[nt][c];
            // d[nt] = P of (row r0: tokens 8 nt + 2t, + 1), (row r0 + 8: same)
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                acc[nt][0] += (da * tgi::int_of_f32(d[nt][0])) >> frac;
                acc[nt][1] += (da * tgi::int_of_f32(d[nt][1])) >> frac;
                acc[nt][2] += (db * tgi::int_of_f32(d[nt][2])) >> frac;
                acc[nt][3] += (db * tgi::int_of_f32(d[nt][3])) >> frac;
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            const int tok = 8 * nt + 2 * t;
            atomicAdd(&ysum[r0 * 8 * NT + tok], (unsigned long long)acc[nt][0]);
            atomicAdd(&ysum[r0 * 8 * NT + tok + 1], (unsigned long long)acc[nt][1]);
            atomicAdd(&ysum[(r0 + 8) * 8 * NT + tok], (unsigned long long)acc[nt][2]);
            atomicAdd(&ysum[(r0 + 8) * 8 * NT + tok + 1], (unsigned long long)acc[nt][3]);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < 32 * mc; i += blockDim.x) {
            const int tok = i >> 5, rl = i & 31;
            const int row = tile * kTileRows + rl;
            if (row < N)
                y[(size_t)(m0 + tok) * N + row] = (int64_t)ysum[rl * 8 * NT + tok];
        }
        __syncthreads();   // xs and ysum are reused by the next chunk
    }
#undef TG_HMMA_LOAD_GROUP
}

size_t hmma_smem_bytes(int G, int NT) { return (size_t)8 * NT * (2 * 128 * (size_t)G + 16) + (size_t)32 * 8 * NT * 8; }

template <bool kQ1, int NT>
cudaError_t launch_hmma(const uint4 *masks, const int32_t *scales, const int8_t *x, int64_t *y, int N, int G,
                        int tiles, int M, int frac, bool pdl, cudaStream_t s)
{
    auto kern = gemv_i8_hmma_kernel<kQ1, NT>;
    const size_t smem = hmma_smem_bytes(G, NT);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, masks, scales, x, y, N, G, M, frac);
}

template <bool kQ1>
cudaError_t dispatch_hmma(const uint4 *masks, const int32_t *scales, const int8_t *x, int64_t *y, int N, int G,
                          int tiles, int M, int frac, bool pdl, cudaStream_t s)
{
    // token tiles per chunk: as many as M needs, as far as the fragments fit
    const int need = (M + 7) / 8;
    if (need >= 4 && hmma_smem_bytes(G, 4) <= kFragBudget)
        return launch_hmma<kQ1, 4>(masks, scales, x, y, N, G, tiles, M, frac, pdl, s);
    if (need >= 2 && hmma_smem_bytes(G, 2) <= kFragBudget)
        return launch_hmma<kQ1, 2>(masks, scales, x, y, N, G, tiles, M, frac, pdl, s);
    return launch_hmma<kQ1, 1>(masks, scales, x, y, N, G, tiles, M, frac, pdl, s);
}

}  // namespace

namespace tgi {

bool gemv_i8_hmma_fits(int G) { return hmma_smem_bytes(G, 1) <= kFragBudget; }

int gemv_i8_hmma(const uint4 *masks, const int32_t *scales, const int8_t *x, int64_t *y, int N, int G, int tiles,
                 int M, bool q1, int frac, bool pdl, cudaStream_t s)
{
    if (!gemv_i8_hmma_fits(G))
        return TG_ERR_SHAPE;
    const cudaError_t e = q1 ? dispatch_hmma<true>(masks, scales, x, y, N, G, tiles, M, frac, pdl, s)
                             : dispatch_hmma<false>(masks, scales, x, y, N, G, tiles, M, frac, pdl, s);
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace tgi
