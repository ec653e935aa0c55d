// lns8.cu -- LNS8 S1|E4|L3 eight-phase GEMV (BitState brief §3, §3.1, and the
// generic variant of §4, where the group's scale code is added before the
// L3/E4 split):
//
//   for every lane with t != 0 and activation code a != 0:
//     k = a + d[r][g] - 74;  k <= 0 -> exact zero;  k > 127 -> 127
//     A[r][k & 7] += (s_a XOR [t < 0]) ? -(1 << (k >> 3)) : (1 << (k >> 3))
//   S[r] = 2^-9 * sum_{p=0..7} A[r][p] * F[p],  F[p] = 2^((p - 2) / 8)
//
// Mapping: one CTA per tile of 32 rows, lane l of each warp owns row 32T + l,
// the warps split the groups. Each thread keeps its eight phase accumulators
// in its own shared-memory column (the phase index is data dependent, and a
// register array indexed at run time would live in local memory). The
// per-thread partials fit int32 (|A| <= K * 2^15 < 2^31 for K < 65536) and are
// summed into int64 at the end. S is materialised in the same kernel with
// explicitly rounded fp64 multiplies and adds in the order p = 0..7.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "device_common.cuh"
#include "tg.h"
#include "tg_internal.h"

TGI_DEFINE_DEVICE_ERROR(lns8_take_device_error)

namespace {

using tgi::kTileRows;

struct PhaseF {
    double f[8];
};

template <int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
lns8_phase_kernel(const uint4 *__restrict__ masks, const uint8_t *__restrict__ codes,
                  const uint8_t *__restrict__ xa, int64_t *__restrict__ A, double *__restrict__ S,
                  PhaseF F, int N, int G)
{
    extern __shared__ __align__(16) unsigned char smem[];
    uint8_t *xs = smem;                                                  // [G*128]
    int *acc = reinterpret_cast<int *>(smem + G * 128);                  // [8][WARPS*32]
    constexpr int BD = WARPS * 32;

    const int tile = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tid = threadIdx.x;
    const uint4 *tmask = masks + (size_t)tile * G * 64;
    const uint8_t *tcode = codes + (size_t)tile * G * kTileRows;

    const int K = G * 128;
    for (int i = tid; i < K / 16; i += BD)
        reinterpret_cast<uint4 *>(xs)[i] = __ldg(reinterpret_cast<const uint4 *>(xa) + i);
#pragma unroll
    for (int p = 0; p < 8; p++)
        acc[p * BD + tid] = 0;
    __syncthreads();

    for (int g = warp; g < G; g += WARPS) {
        const uint4 q0 = tgi::ldg_stream(tmask + g * 64 + lane);
        const uint4 q1 = tgi::ldg_stream(tmask + g * 64 + 32 + lane);
        const int e = (int)__ldg(tcode + g * kTileRows + lane) - 74;
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const uint8_t *xg = xs + g * 128;
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(xg + 16 * u);
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int j = 0; j < 4; j++) {
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    // lane 16u + 4j + b of the group
                    const uint32_t f = (w[u] >> (8 * b + 2 * j)) & 3u;
                    const uint32_t av = (xw[j] >> (8 * b)) & 0xffu;
                    const int a = (int)(av & 0x7fu);
                    int k = a + e;
                    if (f != 0u && a != 0 && k > 0) {
                        k = min(k, 127);
                        const int mag = 1 << (k >> 3);
                        const bool neg = ((av >> 7) ^ (f >> 1)) & 1u;
                        acc[(k & 7) * BD + tid] += neg ? -mag : mag;
                    }
                }
            }
        }
    }
    __syncthreads();

    if (warp == 0) {
        const int row = tile * kTileRows + lane;
        int64_t a8[8];
#pragma unroll
        for (int p = 0; p < 8; p++) {
            int64_t s = 0;
#pragma unroll
            for (int w = 0; w < WARPS; w++)
                s += acc[p * BD + w * 32 + lane];
            a8[p] = s;
        }
        if (row < N) {
#pragma unroll
            for (int p = 0; p < 8; p++)
                A[(size_t)row * 8 + p] = a8[p];
            if (S) {
                double sum = 0.0;
#pragma unroll
                for (int p = 0; p < 8; p++)
                    sum = __dadd_rn(sum, __dmul_rn((double)a8[p], F.f[p]));
                S[row] = __dmul_rn(sum, 0x1p-9);
            }
        }
    }
}

constexpr int kWarps = 4;

}  // namespace

extern "C" int tg_gemv_lns8_phase(const tg_layout *L, const void *w, const uint8_t *xa, int64_t *A,
                                  double *S, void *stream)
{
    if (!L || !w || !xa || !A)
        return TG_ERR_ARG;
    if (L->kind != TG_TERNARY_LNS8 || L->version != 1)
        return TG_ERR_ARG;
    if (!tgi::aligned(w, 256) || !tgi::aligned(xa, 16) || !tgi::aligned(A, 8) ||
        (S && !tgi::aligned(S, 8)))
        return TG_ERR_ARG;
    if (L->N < 1 || L->K < TG_GROUP || L->K % TG_GROUP)
        return TG_ERR_SHAPE;
    if (L->K >= 65536)   // per-thread int32 phase partials: K * 2^15 < 2^31
        return TG_ERR_BOUND;

    PhaseF F;
    for (int p = 0; p < 8; p++)
        F.f[p] = std::exp2((double)(p - 2) / 8.0);

    const auto *base = static_cast<const unsigned char *>(w);
    const uint4 *masks = reinterpret_cast<const uint4 *>(base + L->mask_off);
    const uint8_t *codes = base + L->scale_off;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int G = (int)L->G;
    const size_t smem = (size_t)G * 128 + 8 * kWarps * 32 * sizeof(int);
    auto kern = lns8_phase_kernel<kWarps>;
    if (smem > 48 * 1024) {
        if (smem > 200 * 1024)
            return TG_ERR_SHAPE;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return TG_ERR_CUDA;
    }
    kern<<<(int)L->tiles, kWarps * 32, smem, s>>>(masks, codes, xa, A, S, F, (int)L->N, G);
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}
