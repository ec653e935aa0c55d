// lns8_purelns.cu -- the pure fractional-LNS reduction of the LNS8 product
// states (BitState brief §5.2), selected by TG_FLAG_LNS8_PURE_LNS on
// tg_gemv_lns8_phase. Approximate by design: there is no linear accumulator,
// every addition is a log-domain pairwise add with table corrections.
//
// Definition (this library's reading of §5.2; the oracle states the same):
//   value (s, L): s in {-1, 0, +1}, L = log magnitude in code units held as
//   the integer L * 2^F (F = internal fractional bits, 1..6); the value is
//   s * 2^((L - 74) / 8).
//   Count fold: a signed state population C != 0 of product code k becomes
//   (sign C, k 2^F + LOG8[|C|]), LOG8[n] = round(8 log2 n 2^F).
//   Pairwise add, hi = the operand with the larger L (the first on a tie),
//   diff = L_hi - L_lo: same sign -> L_hi + KP[diff]; opposite sign -> zero
//   if diff = 0, else L_hi + KM[diff]; KP[i] = round(8 log2(1 + 2^(-i/(8 2^F))) 2^F),
//   KM[i] = round(8 log2(1 - 2^(-i/(8 2^F))) 2^F), both 0 from (8F + 40) 2^F on.
//   Trees are balanced, left half first: per (group, phase p) over the sixteen
//   band slots k = 8b + p, per phase over the groups padded with zeros to a
//   power of two, then over the eight phases.
//
// Mapping: one warp per row, lane = group (or a run of groups when there are
// more than 32: a lane's local tree over its run, then the warp tree). A lane
// reads its row's four 16-byte LNS8 entries for the group, compacts them into
// W_nonzero / W_negative words (the byte-permute conversion of the state-set
// route), walks the set bits into a 128-bin population histogram in shared
// memory, and folds each phase's sixteen band slots, clearing each bin as it
// reads it. The histograms are stored bin-major ([bin][thread], rows of 260
// bytes), so the lanes of a warp reading the same bin touch consecutive bytes
// and lanes sharing a word that update different bins fall in different banks.
// Bins are 8-bit: a count lies in [-128, 128], and its two ends wrap to the same
// byte only when all 128 lanes of the group fell into that one bin, in which
// case the group's total of signs is that bin's count. The staged
// activation groups are 132 bytes apart, so lanes of different groups reading
// the same column fall in different banks. The group tree is a
// shuffle tree (lane i combines with lane i + 2^l, left operand first), and
// lane 0 reduces the eight phases. The tables are computed on the host from
// the definitions above and passed as a kernel parameter (23 KB at F = 6).
//
// Output: A[r][0] = s, A[r][1] = L * 2^F, A[r][2..7] = 0, and
// S[r] = s * 2^((L - 74) / 8) in fp64.

#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "device_common.cuh"
#include "tg.h"
#include "tg_internal.h"

namespace {

constexpr int kWarps = 8;             // rows per CTA (one warp each)
constexpr int kThreads = kWarps * 32;
constexpr int kBinStride = 260;       // bytes per histogram bin row (kThreads + a 4-byte bank skew)
constexpr int kXStride = 132;         // bytes between staged activation groups (33 words)
constexpr int kMaxF = 6;
constexpr int kLenMax = (8 * kMaxF + 40) << kMaxF;   // table length at F = 6
constexpr unsigned kFull = 0xffffffffu;

constexpr int kLog8 = 136;   // LOG8 entries stored ([0..128] used; 136 keeps what follows 16-byte aligned)

// 16-byte aligned so that the kernel can copy it to shared memory in 16-byte loads
struct alignas(16) LnsTables {
    int16_t log8[kLog8];
    int16_t kp[kLenMax];
    int16_t km[kLenMax];
};
static_assert(sizeof(LnsTables) < 30 * 1024, "kernel parameter space");
static_assert(offsetof(LnsTables, kp) % 16 == 0 && offsetof(LnsTables, km) % 16 == 0, "16-byte table rows");

struct Lv {
    int s;     // -1, 0, +1
    int lam;   // log magnitude * 2^F (meaningless when s = 0)
};

__device__ __forceinline__ Lv lns_add(Lv u, Lv v, const int16_t *kp, const int16_t *km, int len)
{
    if (u.s == 0)
        return v;
    if (v.s == 0)
        return u;
    const bool uhi = u.lam >= v.lam;
    const Lv hi = uhi ? u : v, lo = uhi ? v : u;
    const int diff = hi.lam - lo.lam;
    Lv r = hi;
    if (hi.s == lo.s)
        r.lam = hi.lam + (diff < len ? kp[diff] : 0);
    else if (diff == 0)
        r = Lv{0, 0};
    else
        r.lam = hi.lam + (diff < len ? km[diff] : 0);
    return r;
}

__device__ __forceinline__ Lv shfl_down(Lv v, int d)
{
    return Lv{__shfl_down_sync(kFull, v.s, d), __shfl_down_sync(kFull, v.lam, d)};
}

// The eight phase aggregates of one (row, group): population histogram, count
// fold, a balanced tree over the sixteen band slots of each phase. bins is the
// thread's histogram column (bin k at bins[k * kBinStride], a count modulo 256);
// it is all zero on entry and is left all zero.
__device__ void group_phases(const uint4 *__restrict__ ent, int half, const uint8_t *xg, int e, int8_t *bins,
                             const int16_t *log8, const int16_t *kp, const int16_t *km, int len, int F, Lv (&ph)[8])
{
    uint4 ev[4];   // the four entries' loads issued together
    int tot = 0;   // the group's total of signs
#pragma unroll
    for (int j = 0; j < 4; j++)
        ev[j] = tgi::ldg_stream(ent + j);
#pragma unroll
    for (int j = 0; j < 4; j++) {
        uint32_t nz0, ng0, nz1, ng1;
        tgi::lns8_compact_words(ev[j], nz0, ng0, nz1, ng1);
        uint32_t nz = half ? nz1 : nz0;
        const uint32_t ng = half ? ng1 : ng0;
        while (nz) {
            const int b = __ffs((int)nz) - 1;
            nz &= nz - 1u;
            const unsigned a = xg[tgi::lns8_lane_col(j, b)];
            const int code = (int)(a & 0x7fu);
            int k = code + e;
            if (code == 0 || k <= 0)
                continue;
            k = min(k, 127);
            const int d = (((ng >> b) & 1u) ^ (a >> 7)) ? -1 : 1;
            bins[k * kBinStride] = (int8_t)(bins[k * kBinStride] + d);
            tot += d;
        }
    }
#pragma unroll 2
    for (int p = 0; p < 8; p++) {
        Lv v[16];
#pragma unroll
        for (int b = 0; b < 16; b++) {
            int8_t *slot = bins + (8 * b + p) * kBinStride;
            const int c8 = *slot;
            *slot = 0;
            const int c = c8 == -128 ? tot : c8;   // +-128: every lane in this bin
            v[b] = c == 0 ? Lv{0, 0} : Lv{c > 0 ? 1 : -1, ((8 * b + p) << F) + log8[c > 0 ? c : -c]};
        }
#pragma unroll
        for (int w = 1; w < 16; w *= 2)
#pragma unroll
            for (int i = 0; i < 16; i += 2 * w)
                v[i] = lns_add(v[i], v[i + w], kp, km, len);
        ph[p] = v[0];
    }
}

__global__ void __launch_bounds__(kThreads, 4)
lns8_purelns_kernel(const uint4 *__restrict__ masks, const uint8_t *__restrict__ codes,
                    const uint8_t *__restrict__ xa, int64_t *__restrict__ A, double *__restrict__ S, int N, int G,
                    int Gp, int F, int len, const __grid_constant__ LnsTables T)
{
    extern __shared__ __align__(16) unsigned char smem[];
    // only the len entries of each table that F uses are held (len is a
    // multiple of 8, so every region starts on a 16-byte boundary)
    int16_t *log8 = reinterpret_cast<int16_t *>(smem);                  // [kLog8]
    int16_t *kp = log8 + kLog8;                                         // [len]
    int16_t *km = kp + len;                                             // [len]
    int8_t *bins_all = reinterpret_cast<int8_t *>(km + len);            // [128][kBinStride]
    uint8_t *xs = reinterpret_cast<uint8_t *>(bins_all + 128 * kBinStride);   // [G][kXStride]
    static_assert((128 * kBinStride) % 16 == 0, "staged activation alignment");
    static_assert((kLog8 * 2) % 16 == 0, "table alignment");

    if ((reinterpret_cast<uintptr_t>(&T) & 15u) == 0) {
        // 16-byte copies: each distinct parameter address a warp reads is a
        // separate constant-cache access, so wide loads take 8x fewer
        const uint4 *src = reinterpret_cast<const uint4 *>(&T);
        uint4 *dst = reinterpret_cast<uint4 *>(smem);
        constexpr int kLogV = kLog8 / 8, kTabV = kLenMax / 8;
        const int lv = len / 8;
        for (int i = threadIdx.x; i < kLogV + 2 * lv; i += blockDim.x) {
            const int t = i < kLogV ? 0 : 1 + (i - kLogV) / lv;   // 0 log8, 1 kp, 2 km
            const int o = i < kLogV ? i : (i - kLogV) - (t - 1) * lv;
            dst[i] = src[t == 0 ? o : kLogV + (t - 1) * kTabV + o];
        }
    } else {
        for (int i = threadIdx.x; i < kLog8; i += blockDim.x)
            log8[i] = T.log8[i];
        for (int i = threadIdx.x; i < len; i += blockDim.x) {
            kp[i] = T.kp[i];
            km[i] = T.km[i];
        }
    }
    for (int i = threadIdx.x; i < 128 * kBinStride / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(bins_all)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < G * 32; i += blockDim.x)
        reinterpret_cast<uint32_t *>(xs)[(i >> 5) * (kXStride / 4) + (i & 31)] =
            __ldg(reinterpret_cast<const uint32_t *>(xa) + i);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + warp;
    if (row >= N)
        return;
    int8_t *bins = bins_all + threadIdx.x;
    const int blk = row >> 4, q = row & 7, half = (row >> 3) & 1;
    const int gpl = Gp > 32 ? Gp / 32 : 1;   // groups per lane

    // this lane's phase aggregates: a tree over its run of groups
    Lv ph[8];
#pragma unroll
    for (int p = 0; p < 8; p++)
        ph[p] = Lv{0, 0};
    if (gpl == 1) {
        // one group per lane: its phase aggregates are the lane's run
        if (lane < G) {
            const uint4 *ent = masks + ((size_t)blk * G + lane) * 32 + 4 * q;
            const int e = (int)codes[((size_t)blk * G + lane) * 16 + (row & 15)] - 74;
            group_phases(ent, half, xs + (size_t)lane * kXStride, e, bins, log8, kp, km, len, F, ph);
        }
    } else if (lane * gpl < Gp) {
        Lv run[8][8];   // [phase][level] partial trees of the run (gpl <= 2^7 groups)
        int filled = 0;
        for (int i = 0; i < gpl; i++) {
            const int g = lane * gpl + i;
            Lv cur[8];
            if (g < G) {
                const uint4 *ent = masks + ((size_t)blk * G + g) * 32 + 4 * q;
                const int e = (int)codes[((size_t)blk * G + g) * 16 + (row & 15)] - 74;
                group_phases(ent, half, xs + (size_t)g * kXStride, e, bins, log8, kp, km, len, F, cur);
            } else {
#pragma unroll
                for (int p = 0; p < 8; p++)
                    cur[p] = Lv{0, 0};
            }
            // binary-counter merge: after 2^m groups the level-m slot holds
            // the balanced tree of those 2^m groups, left half first
            int lvl = 0;
            for (int c = i; c & 1; c >>= 1, lvl++)
#pragma unroll
                for (int p = 0; p < 8; p++)
                    cur[p] = lns_add(run[p][lvl], cur[p], kp, km, len);
#pragma unroll
            for (int p = 0; p < 8; p++)
                run[p][lvl] = cur[p];
            filled = lvl;
        }
#pragma unroll
        for (int p = 0; p < 8; p++)
            ph[p] = run[p][filled];
    }
    // the tree over the lanes' runs, left operand first
    for (int d = 1; d < 32 && d * gpl < Gp; d *= 2)
#pragma unroll
        for (int p = 0; p < 8; p++) {
            const Lv o = shfl_down(ph[p], d);
            if ((lane & (2 * d - 1)) == 0)
                ph[p] = lns_add(ph[p], o, kp, km, len);
        }
    if (lane == 0) {
#pragma unroll
        for (int w = 1; w < 8; w *= 2)
#pragma unroll
            for (int i = 0; i < 8; i += 2 * w)
                ph[i] = lns_add(ph[i], ph[i + w], kp, km, len);
        const Lv R = ph[0];
        int64_t *a = A + (size_t)row * 8;
        a[0] = R.s;
        a[1] = R.s == 0 ? 0 : R.lam;
#pragma unroll
        for (int p = 2; p < 8; p++)
            a[p] = 0;
        if (S)
            S[row] = R.s == 0 ? 0.0 : (double)R.s * exp2(((double)R.lam / (double)(1 << F) - 74.0) / 8.0);
    }
}

// The tables of the definition above, on the host.
void build_tables(int F, LnsTables &T, int &len)
{
    const double scale = std::ldexp(1.0, F);
    len = (8 * F + 40) << F;
    for (int i = 0; i < kLog8; i++)
        T.log8[i] = 0;
    for (int n = 1; n <= 128; n++)
        T.log8[n] = (int16_t)std::llround(8.0 * std::log2((double)n) * scale);
    for (int i = 0; i < kLenMax; i++) {
        if (i >= len) {
            T.kp[i] = T.km[i] = 0;
            continue;
        }
        const double q = std::exp2(-(double)i / (8.0 * scale));
        T.kp[i] = (int16_t)std::llround(8.0 * std::log2(1.0 + q) * scale);
        T.km[i] = i == 0 ? (int16_t)0 : (int16_t)std::llround(8.0 * std::log2(1.0 - q) * scale);
    }
}

}  // namespace

namespace tgi {

int lns8_purelns(const uint4 *masks, const uint8_t *codes, const uint8_t *xa, int64_t *A, double *S, int N, int G,
                 int F, cudaStream_t s)
{
    if (F < 1 || F > kMaxF)
        return TG_ERR_ARG;
    static LnsTables tables[kMaxF + 1];
    static int lens[kMaxF + 1];
    static std::once_flag once[kMaxF + 1];
    std::call_once(once[F], [F] { build_tables(F, tables[F], lens[F]); });   // host tables, once per F
    int Gp = 1;
    while (Gp < G)
        Gp *= 2;
    if (Gp > 32 * 128)   // a lane's run of groups is at most 128 (the run's eight tree levels)
        return TG_ERR_SHAPE;
    const size_t smem = (kLog8 + 2 * (size_t)lens[F]) * 2 + (size_t)128 * kBinStride + (size_t)G * kXStride;
    if (smem > 227 * 1024)
        return TG_ERR_SHAPE;
    cudaError_t e = cudaFuncSetAttribute(lns8_purelns_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return TG_ERR_CUDA;
    lns8_purelns_kernel<<<(N + kWarps - 1) / kWarps, kThreads, smem, s>>>(masks, codes, xa, A, S, N, G, Gp, F,
                                                                              lens[F], tables[F]);
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace tgi
