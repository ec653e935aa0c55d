// lmhead.cu -- vocab-scale lm_head over 8 base-3 planes with argmax and exact
// top-k (SKaiNET-transformers issue #337: BITNET_PLANES and
// BitNetTwoStageDecode; lowest-index tie-break from integer_engine.md §3.3).
//
// Weights arrive as two balanced base-3 digit groups per weight (tg.h):
// hi = planes 0-3 and lo = planes 4-7, both int8 in [-40, 40], W = 81 hi + lo.
// A row's dot products with x are plain signed-byte dp4a sums.
//
// Two-stage path (logits == NULL), all on one stream, no host round trip:
//   1. scan     every row: s1 = 81 * sum hi*x. Its planes 4-7 residual is at
//               most m[r] * sum|x| (m[r] = the row's max |lo| <= 40), so
//               lo_r = s*s1 - s*m*sum|x| <= exact_r <= s*s1 + s*m*sum|x| = hi_r.
//               Each warp also keeps the largest lo_r it saw.
//   2. select   tau = the k-th largest of those per-warp maxima. They are k or
//               more distinct rows' lower bounds, so tau <= the k-th largest
//               lower bound over all rows <= the k-th largest exact logit.
//   3. rescore  every row with hi_r >= tau (this includes every row of the true
//               top-k) is rescored exactly with planes 4-7 and appended as a key.
//   4. final    the top-k of the appended keys.
// Full path (logits != NULL): one scan over both digit groups writes every
// exact logit and each warp's best key; 2-4 as above on the exact keys.
//
// Keys. A score and its row pack into one int64, key = score * 2^b +
// (2^b - 1 - r) with 2^b >= N, so that a larger key means a larger score or,
// on a tie, a lower row index. Every key is distinct, so the top-k set and its
// order are unique whatever order the candidates were appended in.

#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "tg.h"
#include "tg_internal.h"

TGI_DEFINE_DEVICE_ERROR(lmhead_take_device_error)

namespace {

using tgi::dp4a_ss;

constexpr int kScanWarps = 8;       // warps per CTA of the scan kernels
constexpr int kSelThreads = 1024;   // threads of the selection kernels
constexpr int kSortMax = 8192;      // keys sorted at once in shared memory
constexpr uint64_t kSignBit = 0x8000000000000000ull;

struct Ws {
    int64_t *s1;      // [N]  stage-1 sum (two-stage path)
    int64_t *best;    // [kLmhMaxWarps]  per-warp largest lower bound / key
    int64_t *ctl;     // [0] tau, [1] candidate count
    uint64_t *cand;   // [N]  candidate keys, sign bit flipped (unsigned order)
};

__device__ __forceinline__ uint64_t to_ordered(int64_t v) { return (uint64_t)v ^ kSignBit; }
__device__ __forceinline__ int64_t from_ordered(uint64_t u) { return (int64_t)(u ^ kSignBit); }

// The lane's CPL chunks of x (16 bytes each): chunk lane + 32 j.
template <int CPL>
__device__ __forceinline__ void load_x(const int8_t *x, int C16, int lane, uint4 (&xr)[CPL],
                                       int64_t &sum_abs)
{
    int sa = 0;
#pragma unroll
    for (int j = 0; j < CPL; j++) {
        const int c = lane + 32 * j;
        xr[j] = c < C16 ? __ldg(reinterpret_cast<const uint4 *>(x) + c) : make_uint4(0, 0, 0, 0);
        const uint32_t v[4] = {xr[j].x, xr[j].y, xr[j].z, xr[j].w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
#pragma unroll
            for (int b = 0; b < 4; b++) {
                const int xb = (int)(int8_t)((v[q] >> (8 * b)) & 0xff);
                sa += xb < 0 ? -xb : xb;
            }
        }
    }
    sum_abs = (int64_t)tgi::warp_sum_i32(sa);
}

template <int CPL>
__device__ __forceinline__ int row_dot(const int8_t *row, int C16, int lane, const uint4 (&xr)[CPL])
{
    uint4 h[CPL];
#pragma unroll
    for (int j = 0; j < CPL; j++) {
        const int c = lane + 32 * j;
        h[j] = c < C16 ? tgi::ldg_stream(row + (size_t)c * 16) : make_uint4(0, 0, 0, 0);
    }
    int acc = 0;
#pragma unroll
    for (int j = 0; j < CPL; j++) {
        acc = dp4a_ss(h[j].x, xr[j].x, acc);
        acc = dp4a_ss(h[j].y, xr[j].y, acc);
        acc = dp4a_ss(h[j].z, xr[j].z, acc);
        acc = dp4a_ss(h[j].w, xr[j].w, acc);
    }
    return acc;
}

// 1. Stage-1 scan over planes 0-3; two rows per warp iteration keep 2 * CPL
// 16-byte loads per lane in flight.
template <int CPL>
__global__ void __launch_bounds__(kScanWarps * 32)
lmh_stage1_kernel(const int8_t *__restrict__ hi, const int32_t *__restrict__ s,
                  const uint8_t *__restrict__ m, const int8_t *__restrict__ x, Ws ws, int N, int K)
{
    const int lane = threadIdx.x & 31;
    const int wg = blockIdx.x * kScanWarps + (threadIdx.x >> 5);
    const int NW = gridDim.x * kScanWarps;
    const int C16 = K / 16;
    uint4 xr[CPL];
    int64_t sum_abs;
    load_x<CPL>(x, C16, lane, xr, sum_abs);

    int64_t best = INT64_MIN;
    for (int r = wg; r < N; r += 2 * NW) {
        const int r2 = r + NW;
        const int d1 = row_dot<CPL>(hi + (size_t)r * K, C16, lane, xr);
        const int d2 = r2 < N ? row_dot<CPL>(hi + (size_t)r2 * K, C16, lane, xr) : 0;
        const int t1 = tgi::warp_sum_i32(d1);
        const int t2 = tgi::warp_sum_i32(d2);
        if (lane == 0) {
            const int64_t s1 = 81 * (int64_t)t1;
            const int64_t sc = __ldg(s + r);
            ws.s1[r] = s1;
            best = max(best, sc * s1 - sc * (int64_t)__ldg(m + r) * sum_abs);
            if (r2 < N) {
                const int64_t s1b = 81 * (int64_t)t2;
                const int64_t scb = __ldg(s + r2);
                ws.s1[r2] = s1b;
                best = max(best, scb * s1b - scb * (int64_t)__ldg(m + r2) * sum_abs);
            }
        }
    }
    if (lane == 0)
        ws.best[wg] = best;
}

// Full path: exact logits from both digit groups, and each warp's best key.
template <int CPL>
__global__ void __launch_bounds__(kScanWarps * 32)
lmh_full_kernel(const int8_t *__restrict__ hi, const int8_t *__restrict__ lo,
                const int32_t *__restrict__ s, const int8_t *__restrict__ x, int64_t *__restrict__ logits,
                Ws ws, int N, int K, int idx_bits)
{
    const int lane = threadIdx.x & 31;
    const int wg = blockIdx.x * kScanWarps + (threadIdx.x >> 5);
    const int NW = gridDim.x * kScanWarps;
    const int C16 = K / 16;
    uint4 xr[CPL];
    int64_t sum_abs;
    load_x<CPL>(x, C16, lane, xr, sum_abs);
    const int64_t low_mask = ((int64_t)1 << idx_bits) - 1;

    int64_t best = INT64_MIN;
    for (int r = wg; r < N; r += NW) {
        const int dh = row_dot<CPL>(hi + (size_t)r * K, C16, lane, xr);
        const int dl = row_dot<CPL>(lo + (size_t)r * K, C16, lane, xr);
        const int th = tgi::warp_sum_i32(dh);
        const int tl = tgi::warp_sum_i32(dl);
        if (lane == 0) {
            const int64_t logit = (int64_t)__ldg(s + r) * (81 * (int64_t)th + (int64_t)tl);
            logits[r] = logit;
            best = max(best, logit * (low_mask + 1) + (low_mask - r));
        }
    }
    if (lane == 0)
        ws.best[wg] = best;
}

// Bitonic sort of P (a power of two) ordered keys in shared memory, descending.
__device__ void block_sort_desc(uint64_t *v, int P)
{
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            __syncthreads();
            for (int i = threadIdx.x; i < P / 2; i += blockDim.x) {
                const int a = 2 * i - (i & (stride - 1));
                const int b = a + stride;
                const uint64_t ua = v[a], ub = v[b];
                const bool desc = (a & size) == 0;
                if (desc ? (ua < ub) : (ua > ub)) {
                    v[a] = ub;
                    v[b] = ua;
                }
            }
        }
    }
    __syncthreads();
}

__host__ __device__ inline int next_pow2(int n)
{
    int p = 1;
    while (p < n)
        p <<= 1;
    return p;
}

// 2. tau = the k-th largest per-warp entry (INT64_MIN if there are fewer than k).
__global__ void __launch_bounds__(kSelThreads) lmh_threshold_kernel(Ws ws, int nw, int k)
{
    extern __shared__ __align__(16) uint64_t sv[];
    const int P = next_pow2(nw < 2 ? 2 : nw);
    for (int i = threadIdx.x; i < P; i += blockDim.x)
        sv[i] = i < nw ? to_ordered(ws.best[i]) : 0ull;
    block_sort_desc(sv, P);
    if (threadIdx.x == 0) {
        ws.ctl[0] = nw >= k ? from_ordered(sv[k - 1]) : INT64_MIN;
        ws.ctl[1] = 0;
    }
}

// Warp-aggregated append of this lane's key (if `take`) to the candidate list.
__device__ __forceinline__ void append_key(Ws ws, bool take, uint64_t key)
{
    const unsigned mask = __ballot_sync(0xffffffffu, take);
    if (!mask)
        return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(mask) - 1;
    unsigned long long base = 0;
    if (lane == leader)
        base = atomicAdd(reinterpret_cast<unsigned long long *>(ws.ctl + 1), (unsigned long long)__popc(mask));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (take)
        ws.cand[base + __popc(mask & ((1u << lane) - 1))] = key;
}

// 3. Rescore every row whose upper bound reaches tau, exactly, with planes 4-7.
template <int CPL>
__global__ void __launch_bounds__(kScanWarps * 32)
lmh_rescore_kernel(const int8_t *__restrict__ lo, const int32_t *__restrict__ s,
                   const uint8_t *__restrict__ m, const int8_t *__restrict__ x, Ws ws, int N, int K,
                   int idx_bits)
{
    const int lane = threadIdx.x & 31;
    const int wg = blockIdx.x * kScanWarps + (threadIdx.x >> 5);
    const int NW = gridDim.x * kScanWarps;
    const int C16 = K / 16;
    uint4 xr[CPL];
    int64_t sum_abs;
    load_x<CPL>(x, C16, lane, xr, sum_abs);
    const int64_t tau = ws.ctl[0];
    const int64_t low_mask = ((int64_t)1 << idx_bits) - 1;

    for (int base = wg * 32; base < N; base += NW * 32) {
        const int r = base + lane;
        bool cand = false;
        int64_t sc = 0, s1 = 0;
        if (r < N) {
            sc = __ldg(s + r);
            s1 = ws.s1[r];
            cand = sc * s1 + sc * (int64_t)__ldg(m + r) * sum_abs >= tau;
        }
        unsigned todo = __ballot_sync(0xffffffffu, cand);
        while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const int rc = base + src;
            const int64_t csc = __shfl_sync(0xffffffffu, sc, src);
            const int64_t cs1 = __shfl_sync(0xffffffffu, s1, src);
            const int t = tgi::warp_sum_i32(row_dot<CPL>(lo + (size_t)rc * K, C16, lane, xr));
            const int64_t exact = csc * (cs1 + (int64_t)t);
            const uint64_t key = to_ordered(exact * (low_mask + 1) + (low_mask - rc));
            if (lane == 0) {
                const unsigned long long slot =
                    atomicAdd(reinterpret_cast<unsigned long long *>(ws.ctl + 1), 1ull);
                ws.cand[slot] = key;
            }
        }
    }
}

// Full path, 3: append every row whose exact key reaches tau.
__global__ void __launch_bounds__(256)
lmh_collect_kernel(const int64_t *__restrict__ logits, Ws ws, int N, int idx_bits)
{
    const int64_t tau = ws.ctl[0];
    const int64_t low_mask = ((int64_t)1 << idx_bits) - 1;
    const int stride = gridDim.x * blockDim.x;
    for (int base = blockIdx.x * blockDim.x; base < N; base += stride) {
        const int r = base + threadIdx.x;
        int64_t key = INT64_MIN;
        if (r < N)
            key = logits[r] * (low_mask + 1) + (low_mask - r);
        append_key(ws, r < N && key >= tau, to_ordered(key));
    }
}

// 4. Top-k of the candidate keys: a running top-k kept at the front of a
// shared-memory buffer, refilled behind it chunk by chunk and re-sorted.
__global__ void __launch_bounds__(kSelThreads)
lmh_final_kernel(Ws ws, int k, int idx_bits, int32_t *__restrict__ argmax, int32_t *__restrict__ ids,
                 int64_t *__restrict__ scores, int32_t *__restrict__ ncand)
{
    extern __shared__ __align__(16) uint64_t sv[];
    const long long n = ws.ctl[1];
    int cap = (int)(n < kSortMax ? n : kSortMax);
    if (cap < 2 * k)
        cap = 2 * k;
    const int P = next_pow2(cap);
    for (int i = threadIdx.x; i < P; i += blockDim.x)
        sv[i] = i < n ? ws.cand[i] : 0ull;
    block_sort_desc(sv, P);
    for (long long off = P; off < n; off += P - k) {
        for (int i = k + threadIdx.x; i < P; i += blockDim.x) {
            const long long src = off + (i - k);
            sv[i] = src < n ? ws.cand[src] : 0ull;
        }
        block_sort_desc(sv, P);
    }
    const int64_t low_mask = ((int64_t)1 << idx_bits) - 1;
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
        if (j < n) {
            const int64_t key = from_ordered(sv[j]);
            ids[j] = (int32_t)(low_mask - (key & low_mask));
            scores[j] = key >> idx_bits;
        } else {
            ids[j] = -1;
            scores[j] = INT64_MIN;
        }
    }
    if (threadIdx.x == 0) {
        argmax[0] = n > 0 ? (int32_t)(low_mask - (from_ordered(sv[0]) & low_mask)) : -1;
        if (ncand)
            ncand[0] = (int32_t)n;
    }
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

Ws carve(void *ws, int64_t N)
{
    auto *p = static_cast<unsigned char *>(ws);
    Ws w;
    size_t off = 0;
    w.s1 = reinterpret_cast<int64_t *>(p + off);
    off += align256((size_t)N * 8);
    w.best = reinterpret_cast<int64_t *>(p + off);
    off += align256((size_t)tgi::kLmhMaxWarps * 8);
    w.ctl = reinterpret_cast<int64_t *>(p + off);
    off += 256;
    w.cand = reinterpret_cast<uint64_t *>(p + off);
    return w;
}

template <int CPL>
void launch_scan(bool full, int grid, cudaStream_t st, const int8_t *hi, const int8_t *lo,
                 const int32_t *s, const uint8_t *m, const int8_t *x, int64_t *logits, Ws ws, int N,
                 int K, int idx_bits)
{
    if (full)
        lmh_full_kernel<CPL><<<grid, kScanWarps * 32, 0, st>>>(hi, lo, s, x, logits, ws, N, K, idx_bits);
    else
        lmh_stage1_kernel<CPL><<<grid, kScanWarps * 32, 0, st>>>(hi, s, m, x, ws, N, K);
}

template <int CPL>
void launch_rescore(int grid, cudaStream_t st, const int8_t *lo, const int32_t *s, const uint8_t *m,
                    const int8_t *x, Ws ws, int N, int K, int idx_bits)
{
    lmh_rescore_kernel<CPL><<<grid, kScanWarps * 32, 0, st>>>(lo, s, m, x, ws, N, K, idx_bits);
}

}  // namespace

extern "C" size_t tg_lmhead_workspace_bytes(const tg_layout *L, int32_t k)
{
    if (!L || L->kind != TG_PLANES8 || L->N < 1 || k < 1)
        return 0;
    return align256((size_t)L->N * 8) + align256((size_t)tgi::kLmhMaxWarps * 8) + 256 +
           align256((size_t)L->N * 8);
}

extern "C" int tg_lmhead_argmax_topk(const tg_layout *L, const void *w, const int8_t *x, int32_t k,
                                     int64_t *logits, int32_t *argmax, int32_t *ids, int64_t *scores,
                                     int32_t *ncand, void *ws, size_t ws_bytes, void *stream)
{
    if (!L || !w || !x || !argmax || !ids || !scores)
        return TG_ERR_ARG;
    if (L->kind != TG_PLANES8 || L->version != 1)
        return TG_ERR_ARG;
    if (!tgi::aligned(w, 256) || !tgi::aligned(x, 16) || (logits && !tgi::aligned(logits, 8)) ||
        !tgi::aligned(argmax, 4) || !tgi::aligned(ids, 4) || !tgi::aligned(scores, 8) ||
        (ncand && !tgi::aligned(ncand, 4)))
        return TG_ERR_ARG;
    const int64_t N = L->N, K = L->K;
    if (N < 1 || K < TG_GROUP || K % TG_GROUP || k < 1 || k > TG_MAX_K || k > N)
        return TG_ERR_SHAPE;
    const int C16 = (int)(K / 16);
    const int cpl = (C16 + 31) / 32;
    if (cpl > 16)
        return TG_ERR_SHAPE;
    if (!ws || !tgi::aligned(ws, 256) || ws_bytes < tg_lmhead_workspace_bytes(L, k))
        return TG_ERR_WORKSPACE;
    int idx_bits = 1;
    while (((int64_t)1 << idx_bits) < N)
        idx_bits++;
    // |logit| <= max s * 3280 * 128 * K; the key adds idx_bits below it.
    const double max_logit = (double)L->max_abs_scale * 3280.0 * 128.0 * (double)K;
    if (L->max_abs_scale < 1 || max_logit * (double)((int64_t)1 << idx_bits) >= 4.0e18)
        return TG_ERR_BOUND;

    const auto *base = static_cast<const unsigned char *>(w);
    const int8_t *hi = reinterpret_cast<const int8_t *>(base + L->mask_off);
    const int8_t *lo = reinterpret_cast<const int8_t *>(base + L->aux_off);
    const int32_t *s = reinterpret_cast<const int32_t *>(base + L->scale_off);
    const uint8_t *m = base + L->aux2_off;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Ws wsp = carve(ws, N);

    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return TG_ERR_CUDA;
    int grid = nsm * 4;
    const int max_grid = tgi::kLmhMaxWarps / kScanWarps;
    if (grid > max_grid)
        grid = max_grid;
    const int need = (int)((N + kScanWarps - 1) / kScanWarps);
    if (grid > need)
        grid = need;
    const int nw = grid * kScanWarps;
    const bool full = logits != nullptr;
    const int n = (int)N, kk = (int)K;

#define TGI_CPL_CASE(C)                                                                            \
    case C:                                                                                        \
        launch_scan<C>(full, grid, st, hi, lo, s, m, x, logits, wsp, n, kk, idx_bits);             \
        break;
    switch (cpl) {
        TGI_CPL_CASE(1) TGI_CPL_CASE(2) TGI_CPL_CASE(3) TGI_CPL_CASE(4) TGI_CPL_CASE(5)
        TGI_CPL_CASE(6) TGI_CPL_CASE(7) TGI_CPL_CASE(8)
    default:
        launch_scan<16>(full, grid, st, hi, lo, s, m, x, logits, wsp, n, kk, idx_bits);
        break;
    }
#undef TGI_CPL_CASE

    const size_t sel_smem = (size_t)kSortMax * sizeof(uint64_t);
    if (cudaFuncSetAttribute(lmh_threshold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sel_smem) != cudaSuccess ||
        cudaFuncSetAttribute(lmh_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sel_smem) != cudaSuccess)
        return TG_ERR_CUDA;
    lmh_threshold_kernel<<<1, kSelThreads, sel_smem, st>>>(wsp, nw, k);

    if (full) {
        const int cgrid = (int)((N + 255) / 256 < nsm * 8 ? (N + 255) / 256 : nsm * 8);
        lmh_collect_kernel<<<cgrid, 256, 0, st>>>(logits, wsp, n, idx_bits);
    } else {
#define TGI_CPL_CASE(C)                                                                            \
    case C:                                                                                        \
        launch_rescore<C>(grid, st, lo, s, m, x, wsp, n, kk, idx_bits);                            \
        break;
        switch (cpl) {
            TGI_CPL_CASE(1) TGI_CPL_CASE(2) TGI_CPL_CASE(3) TGI_CPL_CASE(4) TGI_CPL_CASE(5)
            TGI_CPL_CASE(6) TGI_CPL_CASE(7) TGI_CPL_CASE(8)
        default:
            launch_rescore<16>(grid, st, lo, s, m, x, wsp, n, kk, idx_bits);
            break;
        }
#undef TGI_CPL_CASE
    }
    lmh_final_kernel<<<1, kSelThreads, sel_smem, st>>>(wsp, k, idx_bits, argmax, ids, scores, ncand);
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

extern "C" int tg_device_error(void *stream, int32_t *code)
{
    if (!code)
        return TG_ERR_ARG;
    int worst = TG_OK;
    const int r[3] = {tgi::gemv_take_device_error(stream), tgi::lns8_take_device_error(stream),
                      tgi::lmhead_take_device_error(stream)};
    for (int v : r) {
        if (v == TG_ERR_CUDA)
            return TG_ERR_CUDA;
        if (v != TG_OK)
            worst = v;
    }
    *code = worst;
    return TG_OK;
}
