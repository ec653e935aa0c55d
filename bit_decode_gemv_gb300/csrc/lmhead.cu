// lmhead.cu -- vocab-scale lm_head over 8 base-3 planes with argmax and exact
// top-k (SKaiNET-transformers issue #337: BITNET_PLANES and
// BitNetTwoStageDecode; lowest-index tie-break from integer_engine.md §3.3).
//
// Weights arrive as two balanced base-3 digit groups per weight (tg.h):
// hi = planes 0-3 and lo = planes 4-7, both int8 in [-40, 40], W = 81 hi + lo,
// in rows of 2K bytes (the row's hi, then its lo; the pointers hi and lo below
// point at row 0's and advance by 2K per row). A row's dot products with x are
// plain signed-byte dp4a sums.
//
// Two-stage path (logits == NULL), all on one stream, no host round trip:
//   1. scan     every row: s1 = 81 * sum hi*x. Its planes 4-7 residual is at
//               most m[r] * sum|x| (m[r] = the row's max |lo| <= 40), so
//               lo_r = s*s1 - s*m*sum|x| <= exact_r <= s*s1 + s*m*sum|x| = hi_r.
//               Each warp counts the largest lo_r it saw in a histogram of
//               scores (below).
//   2. rescore  tau = the lower edge of the histogram bin that holds the k-th
//               largest of those per-warp maxima. They are lower bounds of k or
//               more distinct rows, so tau <= the k-th largest lower bound over
//               all rows <= the k-th largest exact logit; every row with
//               hi_r >= tau (this includes every row of the true top-k) is
//               rescored exactly with planes 4-7, appended as a key, and its
//               exact logit counted in a second histogram.
//   3. final    tau2 = the lower edge of the bin that holds the k-th largest
//               rescored logit; the candidates at or above it (about k) are
//               ranked against each other and written in order.
// Full path (logits != NULL): one scan over both digit groups writes every
// exact logit and counts each warp's largest; the rows at or above the k-th
// bin's edge are appended and step 3 runs on them.
//
// Score histogram. 6144 bins on a log scale: one bin for every score <= 0,
// one per integer for 1..63, then 64 bins per power of two (the leading bit's
// position and the next six bits), so a bin spans under 1/64 of its values.
// A bin's lower edge is a valid lower bound for every score in it.
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
constexpr int kSelThreads = 1024;   // threads of the final selection
constexpr int kHistBins = 6144;     // score histogram bins
constexpr int kFilterMax = 4096;    // candidates at or above tau2 ranked directly
constexpr uint64_t kSignBit = 0x8000000000000000ull;

// Workspace: a region cleared at the start of every call, then per-row data.
struct Ws {
    unsigned long long *count;   // candidates appended
    unsigned *hist_row;          // [kHistWords] scores of every row (fine bins, then coarse)
    unsigned *hist_cand;         // [kHistWords] exact scores of the candidates
    int64_t *s1;                 // [N] stage-1 sums (two-stage path)
    uint64_t *cand;              // [N] candidate keys, sign bit flipped (unsigned order)
};
constexpr int kCoarseBins = kHistBins / 64;   // coarse level: 64 fine bins each
constexpr int kHistWords = kHistBins + kCoarseBins;   // one histogram: fine bins, then coarse bins
constexpr size_t kClearedBytes = 256 + 2 * (size_t)kHistWords * sizeof(unsigned);

__device__ __forceinline__ uint64_t to_ordered(int64_t v) { return (uint64_t)v ^ kSignBit; }

// Byte offset of row r's digit group (hi or lo) from row 0's: rows of 2K bytes.
__device__ __forceinline__ size_t row_off(int r, int K) { return (size_t)r * 2 * (size_t)K; }
__device__ __forceinline__ int64_t from_ordered(uint64_t u) { return (int64_t)(u ^ kSignBit); }

__device__ __forceinline__ int score_bin(int64_t v)
{
    if (v <= 0)
        return 0;
    if (v < 64)
        return 2048 + (int)v;
    const int e = 63 - __clzll(v);                  // 6..62
    const int m = (int)((v >> (e - 6)) & 63);
    return 2048 + 64 * (e - 5) + m;                 // 2112..5759
}

__device__ __forceinline__ int64_t bin_edge(int b)
{
    if (b < 2048)
        return INT64_MIN;
    if (b < 2112)
        return (int64_t)(b - 2048);
    const int t = b - 2048;
    return (int64_t)(64 + (t & 63)) << (t / 64 - 1);
}

// Count one score: its fine bin and the coarse bin above it.
__device__ __forceinline__ void count_score(unsigned *hist, int64_t score)
{
    const int b = score_bin(score);
    atomicAdd(hist + b, 1u);
    atomicAdd(hist + kHistBins + (b >> 6), 1u);
}

// Lower edge of the bin that holds the k-th largest counted score, found by
// one warp from the top of the histogram in two levels -- the 96 coarse bins
// (three per lane), then the 64 fine bins of the chosen coarse bin (two per
// lane) -- each level one round of loads. The counts are read through L2,
// where other CTAs' atomics land. INT64_MIN if fewer than k scores were
// counted.
__device__ int64_t warp_kth_bin_edge(const unsigned *hist, int k)
{
    static_assert(kCoarseBins == 3 * 32, "three coarse bins per lane");
    const int lane = threadIdx.x & 31;
    const unsigned kk = (unsigned)k;

    // level 1: lane l owns coarse bins 95 - 3l, 94 - 3l, 93 - 3l (top down)
    unsigned c[3], mine = 0;
#pragma unroll
    for (int i = 0; i < 3; i++) {
        c[i] = __ldcg(hist + kHistBins + kCoarseBins - 1 - (3 * lane + i));
        mine += c[i];
    }
    unsigned incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    int cb = -1;               // coarse bin holding the k-th score
    unsigned before = 0;       // scores above that coarse bin
    if (incl - mine < kk && kk <= incl) {
        unsigned cum = incl - mine;
#pragma unroll
        for (int i = 0; i < 3; i++) {
            if (cb < 0 && cum + c[i] >= kk) {
                cb = kCoarseBins - 1 - (3 * lane + i);
                before = cum;
            }
            cum += c[i];
        }
    }
    unsigned owner = __ballot_sync(0xffffffffu, cb >= 0);
    if (!owner)
        return INT64_MIN;
    const int src = __ffs(owner) - 1;
    cb = __shfl_sync(0xffffffffu, cb, src);
    before = __shfl_sync(0xffffffffu, before, src);

    // level 2: lane l owns fine bins 64 cb + 63 - 2l and 64 cb + 62 - 2l (top down)
    const int top = 64 * cb + 63 - 2 * lane;
    const unsigned f0 = __ldcg(hist + top), f1 = __ldcg(hist + top - 1);
    const unsigned mine2 = f0 + f1;
    unsigned incl2 = mine2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned v = __shfl_up_sync(0xffffffffu, incl2, o);
        if (lane >= o)
            incl2 += v;
    }
    const unsigned start2 = before + incl2 - mine2;
    int found = -1;
    if (start2 < kk && kk <= before + incl2)
        found = start2 + f0 >= kk ? top : top - 1;
    owner = __ballot_sync(0xffffffffu, found >= 0);
    found = __shfl_sync(0xffffffffu, found, __ffs(owner) - 1);
    return bin_edge(found);
}

// sum_i |x_i| from the warp's register copy of x (chunk lane + 32 j in xr[j],
// zero past the end): |v| = v * (v < 0 ? -1 : 1) per byte in one dp4a.
template <int CPL>
__device__ __forceinline__ int64_t warp_sum_abs_regs(const uint4 (&xr)[CPL])
{
    int sa = 0;
#pragma unroll
    for (int j = 0; j < CPL; j++) {
        const uint32_t w[4] = {xr[j].x, xr[j].y, xr[j].z, xr[j].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t neg = (w[i] & 0x80808080u) >> 7;
            sa = dp4a_ss(w[i], (neg * 0xFEu) | 0x01010101u, sa);
        }
    }
    return (int64_t)tgi::warp_sum_i32(sa);
}

// The lane's CPL chunks of x (16 bytes each): chunk lane + 32 j.
template <int CPL>
__device__ __forceinline__ void load_x(const int8_t *x, int C16, int lane, uint4 (&xr)[CPL])
{
#pragma unroll
    for (int j = 0; j < CPL; j++) {
        const int c = lane + 32 * j;
        xr[j] = c < C16 ? __ldg(reinterpret_cast<const uint4 *>(x) + c) : make_uint4(0, 0, 0, 0);
    }
}

// One row's digit bytes against x. kEvictFirst: the row is read with the L2
// evict-first policy (stage 1: measured 67.4 -> 64.4 us per two-stage call on
// the vocabulary workload, the rescoring and selection kernels' code and data
// staying in L2; the full scan, which streams both digit groups, measured
// slower with it, 135 -> 156 us, and reads without it).
template <int CPL, bool kEvictFirst>
__device__ __forceinline__ int row_dot(const int8_t *row, int C16, int lane, const uint4 (&xr)[CPL])
{
    const uint64_t pol = kEvictFirst ? tgi::l2_evict_first_policy() : 0;
    uint4 h[CPL];
#pragma unroll
    for (int j = 0; j < CPL; j++) {
        const int c = lane + 32 * j;
        h[j] = c >= C16 ? make_uint4(0, 0, 0, 0)
                        : kEvictFirst ? tgi::ldg_stream(row + (size_t)c * 16, pol) : tgi::ldg_stream(row + (size_t)c * 16);
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

// 0. Zero the candidate count and both histograms. Launched as a programmatic
// dependent of whatever precedes the call on the stream, it waits for that
// work to finish (x may be its output), then lets the scan launch; the scan
// waits for the clearing before it touches the workspace.
__global__ void __launch_bounds__(256) lmh_clear_kernel(uint4 *__restrict__ p, int n16)
{
    tgi::pdl_wait();
    tgi::pdl_launch_dependents();
    for (int i = threadIdx.x; i < n16; i += blockDim.x)
        p[i] = make_uint4(0, 0, 0, 0);
}

// 1. Stage-1 scan over planes 0-3; two rows per warp iteration keep 2 * CPL
// 16-byte loads per lane in flight. Each warp counts its largest lower bound.
template <int CPL>
__global__ void __launch_bounds__(kScanWarps * 32)
lmh_stage1_kernel(const int8_t *__restrict__ hi, const int32_t *__restrict__ s,
                  const uint8_t *__restrict__ m, const int8_t *__restrict__ x, Ws ws, int N, int K)
{
    const int lane = threadIdx.x & 31;
    const int wg = blockIdx.x * kScanWarps + (threadIdx.x >> 5);
    const int NW = gridDim.x * kScanWarps;
    const int C16 = K / 16;
    // the rescoring kernel may launch now; it waits for this grid before it
    // reads anything this grid writes
    tgi::pdl_launch_dependents();
    uint4 xr[CPL];
    load_x<CPL>(x, C16, lane, xr);
    const int64_t sum_abs = warp_sum_abs_regs<CPL>(xr);
    // the clearing kernel (tiny) has long finished. Waiting for it here rather
    // than before the first count lets the rescoring CTAs launch while the scan
    // runs (measured: with the wait at the end they launched only as the scan's
    // CTAs exited).
    tgi::pdl_wait();

    int64_t best = INT64_MIN;
    for (int r = wg; r < N; r += 2 * NW) {
        const int r2 = r + NW;
        const int d1 = row_dot<CPL, true>(hi + row_off(r, K), C16, lane, xr);
        const int d2 = r2 < N ? row_dot<CPL, true>(hi + row_off(r2, K), C16, lane, xr) : 0;
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
    if (lane == 0 && best != INT64_MIN)
        count_score(ws.hist_row, best);
}

// Full path: exact logits from both digit groups; each warp counts its largest.
template <int CPL>
__global__ void __launch_bounds__(kScanWarps * 32)
lmh_full_kernel(const int8_t *__restrict__ hi, const int8_t *__restrict__ lo,
                const int32_t *__restrict__ s, const int8_t *__restrict__ x, int64_t *__restrict__ logits,
                Ws ws, int N, int K)
{
    const int lane = threadIdx.x & 31;
    const int wg = blockIdx.x * kScanWarps + (threadIdx.x >> 5);
    const int NW = gridDim.x * kScanWarps;
    const int C16 = K / 16;
    tgi::pdl_launch_dependents();   // the collecting kernel waits for this grid before it reads anything
    uint4 xr[CPL];
    load_x<CPL>(x, C16, lane, xr);
    tgi::pdl_wait();   // the clearing kernel (as in stage 1)

    int64_t best = INT64_MIN;
    for (int r = wg; r < N; r += NW) {
        const int dh = row_dot<CPL, false>(hi + row_off(r, K), C16, lane, xr);
        const int dl = row_dot<CPL, false>(lo + row_off(r, K), C16, lane, xr);
        const int th = tgi::warp_sum_i32(dh);
        const int tl = tgi::warp_sum_i32(dl);
        if (lane == 0) {
            const int64_t logit = (int64_t)__ldg(s + r) * (81 * (int64_t)th + (int64_t)tl);
            logits[r] = logit;
            best = max(best, logit);
        }
    }
    if (lane == 0 && best != INT64_MIN)
        count_score(ws.hist_row, best);
}

// Append this lane's key (if `take`) to the candidate list, one atomic per
// warp, and count the candidate's exact score.
__device__ __forceinline__ void append_key(Ws ws, bool take, uint64_t key, int64_t score)
{
    const unsigned mask = __ballot_sync(0xffffffffu, take);
    if (!mask)
        return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(mask) - 1;
    unsigned long long base = 0;
    if (lane == leader)
        base = atomicAdd(ws.count, (unsigned long long)__popc(mask));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (take) {
        ws.cand[base + __popc(mask & ((1u << lane) - 1))] = key;
        count_score(ws.hist_cand, score);
    }
}

// 2. Rescore every row whose upper bound reaches tau, exactly, with planes 4-7.
// Two CTAs per SM: at 64 registers one fits beside the scan's CTAs and can have
// read x before the scan ends, the other starts as the scan's CTAs exit. A CTA owns a
// contiguous range of rows and filters it in passes of kRescorePass rows (four
// per thread; the first pass's bounds load while one warp finds tau); the
// candidates of a pass are gathered in shared memory and shared out over the
// CTA's warps, two rows per warp at a time so that both rows' loads are in
// flight together.
constexpr int kRescorePass = kScanWarps * 32 * 4;

template <int CPL>
__global__ void __launch_bounds__(kScanWarps * 32, CPL <= 5 ? 4 : 1)
lmh_rescore_kernel(const int8_t *__restrict__ lo, const int32_t *__restrict__ s,
                   const uint8_t *__restrict__ m, const int8_t *__restrict__ x, Ws ws, int N, int K,
                   int k, int idx_bits)
{
    __shared__ int64_t sh_tau;
    __shared__ int sh_n;
    __shared__ unsigned long long sh_base;
    __shared__ int c_row[kRescorePass];
    __shared__ int c_sc[kRescorePass];
    __shared__ int64_t c_s1[kRescorePass];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int C16 = K / 16;
    uint4 xr[CPL];
    load_x<CPL>(x, C16, lane, xr);
    const int64_t sum_abs = warp_sum_abs_regs<CPL>(xr);
    // launched as a programmatic dependent of stage 1: x (complete before stage
    // 1 started) is read above; the histogram and the stage-1 sums only after
    // stage 1 has finished. The final selection may launch now.
    tgi::pdl_launch_dependents();
    tgi::pdl_wait();
    const int64_t low_mask = ((int64_t)1 << idx_bits) - 1;
    const uint64_t pol = tgi::l2_evict_first_policy();
    const int per = (N + (int)gridDim.x - 1) / (int)gridDim.x;
    const int r_begin = (int)blockIdx.x * per;
    const int r_end = min(N, r_begin + per);

    for (int c0 = r_begin; c0 < r_end; c0 += kRescorePass) {
        int scv[4];
        int64_t s1v[4], mv[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int r = c0 + (int)threadIdx.x + kScanWarps * 32 * i;
            const bool ok = r < r_end;
            scv[i] = ok ? __ldg(s + r) : 0;
            s1v[i] = ok ? __ldcg(ws.s1 + r) : 0;
            mv[i] = ok ? (int64_t)__ldg(m + r) : 0;
        }
        if (c0 == r_begin && warp == 0) {
            const int64_t t = warp_kth_bin_edge(ws.hist_row, k);
            if (lane == 0)
                sh_tau = t;
        }
        if (threadIdx.x == 0)
            sh_n = 0;
        __syncthreads();
        const int64_t tau = sh_tau;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int r = c0 + (int)threadIdx.x + kScanWarps * 32 * i;
            const int64_t sc = scv[i];
            if (r < r_end && sc * s1v[i] + sc * mv[i] * sum_abs >= tau) {
                const int slot = atomicAdd(&sh_n, 1);
                c_row[slot] = r;
                c_sc[slot] = scv[i];
                c_s1[slot] = s1v[i];
            }
        }
        __syncthreads();
        const int nc = sh_n;
        for (int i = 2 * warp; i < nc; i += 2 * kScanWarps) {
            const bool two = i + 1 < nc;
            const int r0 = c_row[i], r1 = two ? c_row[i + 1] : r0;
            uint4 h0[CPL], h1[CPL];
#pragma unroll
            for (int j = 0; j < CPL; j++) {
                const int c = lane + 32 * j;
                h0[j] = c < C16 ? tgi::ldg_stream(lo + row_off(r0, K) + (size_t)c * 16, pol)
                                : make_uint4(0, 0, 0, 0);
                h1[j] = (two && c < C16) ? tgi::ldg_stream(lo + row_off(r1, K) + (size_t)c * 16, pol)
                                         : make_uint4(0, 0, 0, 0);
            }
            int a0 = 0, a1 = 0;
#pragma unroll
            for (int j = 0; j < CPL; j++) {
                a0 = dp4a_ss(h0[j].x, xr[j].x, a0);
                a0 = dp4a_ss(h0[j].y, xr[j].y, a0);
                a0 = dp4a_ss(h0[j].z, xr[j].z, a0);
                a0 = dp4a_ss(h0[j].w, xr[j].w, a0);
                a1 = dp4a_ss(h1[j].x, xr[j].x, a1);
                a1 = dp4a_ss(h1[j].y, xr[j].y, a1);
                a1 = dp4a_ss(h1[j].z, xr[j].z, a1);
                a1 = dp4a_ss(h1[j].w, xr[j].w, a1);
            }
            const int t0 = tgi::warp_sum_i32(a0);
            const int t1 = tgi::warp_sum_i32(a1);
            // lane 0 finishes the first row, lane 1 the second: the exact logit is
            // counted, and its key replaces the row's stage-1 sum in the list
            if (lane == 0 || (two && lane == 1)) {
                const int src = i + lane;
                const int64_t e = (int64_t)c_sc[src] * (c_s1[src] + (int64_t)(lane == 1 ? t1 : t0));
                c_s1[src] = (int64_t)to_ordered(e * (low_mask + 1) + (low_mask - c_row[src]));
                count_score(ws.hist_cand, e);
            }
        }
        // the pass's keys go out together: one counter update per CTA
        __syncthreads();
        if (threadIdx.x == 0 && nc > 0)
            sh_base = atomicAdd(ws.count, (unsigned long long)nc);
        __syncthreads();
        for (int i = (int)threadIdx.x; i < nc; i += (int)blockDim.x)
            ws.cand[sh_base + i] = (uint64_t)c_s1[i];
        __syncthreads();   // the list is read before the next pass refills it
    }
}

// Full path, 2: append every row whose exact logit reaches the k-th bin's edge.
__global__ void __launch_bounds__(256)
lmh_collect_kernel(const int64_t *__restrict__ logits, Ws ws, int N, int k, int idx_bits)
{
    __shared__ int64_t sh_tau;
    tgi::pdl_launch_dependents();
    tgi::pdl_wait();   // launched as a programmatic dependent of the full scan
    if (threadIdx.x < 32) {
        const int64_t tau = warp_kth_bin_edge(ws.hist_row, k);
        if (threadIdx.x == 0)
            sh_tau = tau;
    }
    __syncthreads();
    const int64_t tau = sh_tau;
    const int64_t low_mask = ((int64_t)1 << idx_bits) - 1;
    const int stride = gridDim.x * blockDim.x;
    for (int base = blockIdx.x * blockDim.x; base < N; base += stride) {
        const int r = base + threadIdx.x;
        const int64_t logit = r < N ? logits[r] : INT64_MIN;
        append_key(ws, r < N && logit >= tau, to_ordered(logit * (low_mask + 1) + (low_mask - r)), logit);
    }
}

// k-th largest (1-based, counting duplicates) of n ordered keys, by radix
// select from the most significant byte (fallback of the final selection).
// Leading bytes shared by every key (from the block's min and max) are
// skipped. Each warp counts into its own histogram (lanes that share a bin are
// merged first); the 32 histograms are then summed. Called by all threads of
// the block; `key(i)` reads key i. Returns 0 (below every real key) if n < k.
struct RadixSmem {
    unsigned hist[32][256];
    unsigned total[256];
    uint64_t red_min[32], red_max[32];
    uint64_t bcast[2];
};

template <class KeyAt>
__device__ uint64_t block_kth_largest(KeyAt key, int n, int k, RadixSmem &sm)
{
    if (n < k)
        return 0ull;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;

    uint64_t lo = ~0ull, hi = 0ull;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const uint64_t u = key(i);
        lo = u < lo ? u : lo;
        hi = u > hi ? u : hi;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t a = __shfl_xor_sync(0xffffffffu, lo, o), b = __shfl_xor_sync(0xffffffffu, hi, o);
        lo = a < lo ? a : lo;
        hi = b > hi ? b : hi;
    }
    if (lane == 0) {
        sm.red_min[warp] = lo;
        sm.red_max[warp] = hi;
    }
    __syncthreads();
    lo = sm.red_min[0];
    hi = sm.red_max[0];
    for (int w = 1; w < nwarps; w++) {
        lo = sm.red_min[w] < lo ? sm.red_min[w] : lo;
        hi = sm.red_max[w] > hi ? sm.red_max[w] : hi;
    }
    if (lo == hi)
        return lo;
    int shift = 56;
    while (((lo ^ hi) >> shift) == 0)   // bytes above `shift` are common
        shift -= 8;
    uint64_t pmask = shift == 56 ? 0ull : (~0ull << (shift + 8));
    uint64_t prefix = lo & pmask;
    int kk = k;

    for (; shift >= 0; shift -= 8) {
        for (int i = lane; i < 256; i += 32)
            sm.hist[warp][i] = 0;
        __syncwarp();
        for (int base = 0; base < n; base += blockDim.x) {
            const int i = base + threadIdx.x;
            uint64_t u = 0;
            bool take = false;
            if (i < n) {
                u = key(i);
                take = (u & pmask) == prefix;
            }
            const unsigned active = __ballot_sync(0xffffffffu, take);
            if (take) {
                const unsigned bin = (unsigned)(u >> shift) & 255u;
                const unsigned peers = __match_any_sync(active, bin);
                if (lane == __ffs(peers) - 1)
                    sm.hist[warp][bin] += (unsigned)__popc(peers);
            }
            __syncwarp();
        }
        __syncthreads();
        if (threadIdx.x < 256) {
            unsigned t = 0;
            for (int w = 0; w < nwarps; w++)
                t += sm.hist[w][threadIdx.x];
            sm.total[threadIdx.x] = t;
        }
        __syncthreads();
        if (warp == 0) {
            unsigned cnt[8], mine = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                cnt[j] = sm.total[255 - 8 * lane - j];
                mine += cnt[j];
            }
            unsigned incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            const unsigned before = incl - mine;
            if (before < (unsigned)kk && (unsigned)kk <= incl) {
                unsigned cum = before;
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    if (cum < (unsigned)kk && (unsigned)kk <= cum + cnt[j]) {
                        sm.bcast[0] = (uint64_t)(255 - 8 * lane - j);
                        sm.bcast[1] = (uint64_t)cum;
                    }
                    cum += cnt[j];
                }
            }
        }
        __syncthreads();
        prefix |= sm.bcast[0] << shift;
        pmask |= 0xFFull << shift;
        kk -= (int)sm.bcast[1];
        __syncthreads();
    }
    return prefix;
}

// 3. Top-k of the candidate keys. The candidates whose exact score reaches
// the k-th candidate bin's edge (about k of them, and every one of the top k)
// are gathered and each is written at its rank among them. If a dense bin
// makes that set too large, the k-th largest key is found by radix select and
// the k keys at or above it are ranked instead.
__global__ void __launch_bounds__(kSelThreads)
lmh_final_kernel(Ws ws, int k, int idx_bits, int32_t *__restrict__ argmax, int32_t *__restrict__ ids,
                 int64_t *__restrict__ scores, int32_t *__restrict__ ncand)
{
    // the next kernel on the stream may launch now (it waits for this grid before
    // it touches anything this call reads or writes)
    tgi::pdl_launch_dependents();
    tgi::pdl_wait();   // launched as a programmatic dependent of the rescoring / collecting kernel
    extern __shared__ __align__(16) unsigned char dyn[];
    uint64_t *sel = reinterpret_cast<uint64_t *>(dyn);                                 // [kFilterMax]
    RadixSmem &rs = *reinterpret_cast<RadixSmem *>(dyn + kFilterMax * sizeof(uint64_t));
    __shared__ int64_t sh_tau;
    __shared__ int nsel;
    const int n = (int)*ws.count;
    const int64_t low_mask = ((int64_t)1 << idx_bits) - 1;
    // this thread's first two candidate keys load while warp 0 finds tau2
    const int i0 = (int)threadIdx.x, i1 = (int)threadIdx.x + kSelThreads;
    const uint64_t u0 = i0 < n ? __ldcg(ws.cand + i0) : 0ull;
    const uint64_t u1 = i1 < n ? __ldcg(ws.cand + i1) : 0ull;
    if (threadIdx.x < 32) {
        const int64_t tau = warp_kth_bin_edge(ws.hist_cand, k);
        if (threadIdx.x == 0) {
            sh_tau = tau;
            nsel = 0;
        }
    }
    __syncthreads();
    const int64_t tau = sh_tau;
    // warp-aggregated appends: one shared atomic per warp, not per key
    auto append_sel = [&](bool take, uint64_t u) {
        const unsigned mask = __ballot_sync(0xffffffffu, take);
        if (!mask)
            return;
        const int lane = threadIdx.x & 31;
        const int leader = __ffs(mask) - 1;
        int base = 0;
        if (lane == leader)
            base = atomicAdd(&nsel, __popc(mask));
        base = __shfl_sync(0xffffffffu, base, leader);
        const int slot = base + __popc(mask & ((1u << lane) - 1));
        if (take && slot < kFilterMax)
            sel[slot] = u;
    };
    append_sel(i0 < n && (from_ordered(u0) >> idx_bits) >= tau, u0);
    append_sel(i1 < n && (from_ordered(u1) >> idx_bits) >= tau, u1);
    for (int b = 2 * kSelThreads; b < n; b += kSelThreads) {   // uniform over the block: full warps in append_sel
        const int i = b + (int)threadIdx.x;
        const uint64_t u = i < n ? ws.cand[i] : 0ull;
        append_sel(i < n && (from_ordered(u) >> idx_bits) >= tau, u);
    }
    __syncthreads();
    int m = nsel;
    if (m > kFilterMax) {
        // dense bin: radix select over every candidate, keep the k at or above
        const uint64_t t = block_kth_largest([&](int i) { return ws.cand[i]; }, n, k, rs);
        if (threadIdx.x == 0)
            nsel = 0;
        __syncthreads();
        for (int b = 0; b < n; b += blockDim.x) {
            const int i = b + threadIdx.x;
            const uint64_t u = i < n ? ws.cand[i] : 0ull;
            append_sel(i < n && u >= t, u);
        }
        __syncthreads();
        m = nsel < kFilterMax ? nsel : kFilterMax;
    }
    const int kout = m < k ? m : k;
    // Rank of key i = the number of larger keys (all keys are distinct). Each
    // run of 32 keys is sorted (descending) by one warp, which gives every key
    // its count within its run; the counts in the other runs come from binary
    // searches, one (key, run) pair per thread, summed in shared memory (the
    // radix select's bins are free by now).
    unsigned *rank_of = &rs.hist[0][0];
    static_assert(sizeof(rs.hist) >= kFilterMax * sizeof(unsigned), "rank array");
    const int runs = (m + 31) >> 5;
    {
        const int warp = (int)threadIdx.x >> 5, lane = (int)threadIdx.x & 31;
        for (int rr = warp; rr < runs; rr += kSelThreads / 32) {
            const int i = rr * 32 + lane;
            uint64_t u = i < m ? sel[i] : 0ull;   // padding sorts below every key
#pragma unroll
            for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    const uint64_t o = __shfl_xor_sync(0xffffffffu, u, stride);
                    const bool lower = (lane & stride) == 0, rising = (lane & size) == 0;
                    u = (lower != rising) ? (u < o ? u : o) : (u > o ? u : o);
                }
            }
            sel[i] = u;
            rank_of[i] = (unsigned)lane;
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < m * runs; t += blockDim.x) {
        const int i = t / runs, rr = t - i * runs;
        if (rr == (i >> 5))
            continue;
        const uint64_t u = sel[i];
        const uint64_t *run = sel + rr * 32;
        int lo = 0, hi = m - rr * 32 < 32 ? m - rr * 32 : 32;
        while (lo < hi) {   // first position of the run holding a key below u
            const int mid = (lo + hi) >> 1;
            if (run[mid] > u)
                lo = mid + 1;
            else
                hi = mid;
        }
        if (lo)
            atomicAdd(rank_of + i, (unsigned)lo);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
        const uint64_t u = sel[i];
        const int rank = (int)rank_of[i];
        if (rank < kout) {
            const int64_t key = from_ordered(u);
            ids[rank] = (int32_t)(low_mask - (key & low_mask));
            scores[rank] = key >> idx_bits;
            if (rank == 0)
                argmax[0] = (int32_t)(low_mask - (key & low_mask));
        }
    }
    for (int i = kout + threadIdx.x; i < k; i += blockDim.x) {
        ids[i] = -1;
        scores[i] = INT64_MIN;
    }
    if (threadIdx.x == 0) {
        if (kout == 0)
            argmax[0] = -1;
        if (ncand)
            ncand[0] = n;
    }
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

Ws carve(void *ws, int64_t N)
{
    auto *p = static_cast<unsigned char *>(ws);
    Ws w;
    w.count = reinterpret_cast<unsigned long long *>(p);
    w.hist_row = reinterpret_cast<unsigned *>(p + 256);
    w.hist_cand = w.hist_row + kHistWords;
    size_t off = kClearedBytes;
    w.s1 = reinterpret_cast<int64_t *>(p + off);
    off += align256((size_t)N * 8);
    w.cand = reinterpret_cast<uint64_t *>(p + off);
    return w;
}

// Launch config of a programmatic dependent of the previous kernel on the stream.
struct PdlLaunch {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    PdlLaunch(int grid, int threads, size_t smem, cudaStream_t st)
    {
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
};

template <int CPL>
cudaError_t launch_scan(bool full, int grid, cudaStream_t st, const int8_t *hi, const int8_t *lo,
                        const int32_t *s, const uint8_t *m, const int8_t *x, int64_t *logits, Ws ws, int N, int K)
{
    // The scans use no shared memory; ask for an SM configuration with room for
    // the rescoring or collecting CTAs that launch beside them (set on every call:
    // a function attribute belongs to the current device).
    cudaError_t carve = cudaFuncSetAttribute(lmh_stage1_kernel<CPL>, cudaFuncAttributePreferredSharedMemoryCarveout, 25);
    if (carve == cudaSuccess)
        carve = cudaFuncSetAttribute(lmh_full_kernel<CPL>, cudaFuncAttributePreferredSharedMemoryCarveout, 25);
    if (carve != cudaSuccess)
        return carve;
    PdlLaunch l(grid, kScanWarps * 32, 0, st);
    if (full)
        return cudaLaunchKernelEx(&l.cfg, lmh_full_kernel<CPL>, hi, lo, s, x, logits, ws, N, K);
    return cudaLaunchKernelEx(&l.cfg, lmh_stage1_kernel<CPL>, hi, s, m, x, ws, N, K);
}

template <int CPL>
cudaError_t launch_rescore(int grid, cudaStream_t st, const int8_t *lo, const int32_t *s, const uint8_t *m,
                           const int8_t *x, Ws ws, int N, int K, int k, int idx_bits)
{
    PdlLaunch l(grid, kScanWarps * 32, 0, st);
    return cudaLaunchKernelEx(&l.cfg, lmh_rescore_kernel<CPL>, lo, s, m, x, ws, N, K, k, idx_bits);
}

}  // namespace

extern "C" size_t tg_lmhead_workspace_bytes(const tg_layout *L, int32_t k)
{
    if (!L || L->kind != TG_PLANES8 || L->N < 1 || k < 1)
        return 0;
    return kClearedBytes + align256((size_t)L->N * 8) + align256((size_t)L->N * 8);
}

namespace tgi {

int lmhead_check_args(const tg_layout *L, const void *w, const int8_t *x, int32_t k, const int64_t *logits,
                      const int32_t *argmax, const int32_t *ids, const int64_t *scores, const int32_t *ncand)
{
    if (!L || !w || !x || !argmax || !ids || !scores)
        return TG_ERR_ARG;
    if (L->kind != TG_PLANES8 || L->version != 1 || L->frac != 0)
        return TG_ERR_ARG;
    if (!tgi::aligned(w, 256) || !tgi::aligned(x, 16) || (logits && !tgi::aligned(logits, 8)) ||
        !tgi::aligned(argmax, 4) || !tgi::aligned(ids, 4) || !tgi::aligned(scores, 8) ||
        (ncand && !tgi::aligned(ncand, 4)))
        return TG_ERR_ARG;
    const int64_t N = L->N, K = L->K;
    if (N < 1 || K < TG_GROUP || K % TG_GROUP || k < 1 || k > TG_MAX_K || k > N)
        return TG_ERR_SHAPE;
    if ((K / 16 + 31) / 32 > 16)   // 16-byte chunks of a row per lane
        return TG_ERR_SHAPE;
    return TG_OK;
}

}  // namespace tgi

extern "C" int tg_lmhead_argmax_topk(const tg_layout *L, const void *w, const int8_t *x, int32_t k,
                                     int64_t *logits, int32_t *argmax, int32_t *ids, int64_t *scores,
                                     int32_t *ncand, void *ws, size_t ws_bytes, void *stream)
{
    const int bad = tgi::lmhead_check_args(L, w, x, k, logits, argmax, ids, scores, ncand);
    if (bad != TG_OK)
        return bad;
    const int64_t N = L->N, K = L->K;
    const int C16 = (int)(K / 16);
    const int cpl = (C16 + 31) / 32;
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
    const bool full = logits != nullptr;
    // scan CTAs per SM (measured on the vocabulary workload): the two-stage scan leaves
    // room for one rescoring CTA per SM beside its four (65.5 us per call; five: 78.5);
    // the full scan, followed only by the collecting kernel, is fastest with five
    // (111.4 us per call; four: 118.3)
    int grid = nsm * (full ? 5 : 4);
    const int need = (int)((N + kScanWarps - 1) / kScanWarps);
    if (grid > need)
        grid = need;
    const int n = (int)N, kk = (int)K;

    // the candidate count and both histograms start at zero every call
    static_assert(kClearedBytes % 16 == 0, "cleared region in 16-byte words");
    {
        PdlLaunch cl(1, 256, 0, st);
        if (cudaLaunchKernelEx(&cl.cfg, lmh_clear_kernel, static_cast<uint4 *>(ws), (int)(kClearedBytes / 16)) !=
            cudaSuccess)
            return TG_ERR_CUDA;
    }

    cudaError_t re = cudaSuccess;
#define TGI_CPL_CASE(C)                                                                            \
    case C:                                                                                        \
        re = launch_scan<C>(full, grid, st, hi, lo, s, m, x, logits, wsp, n, kk);                  \
        break;
    switch (cpl) {
        TGI_CPL_CASE(1) TGI_CPL_CASE(2) TGI_CPL_CASE(3) TGI_CPL_CASE(4) TGI_CPL_CASE(5)
        TGI_CPL_CASE(6) TGI_CPL_CASE(7) TGI_CPL_CASE(8)
    default:
        re = launch_scan<16>(full, grid, st, hi, lo, s, m, x, logits, wsp, n, kk);
        break;
    }
#undef TGI_CPL_CASE
    if (re != cudaSuccess)
        return TG_ERR_CUDA;

    if (full) {
        const int cgrid = (int)((N + 255) / 256 < nsm * 4 ? (N + 255) / 256 : nsm * 4);
        PdlLaunch cl(cgrid, 256, 0, st);
        re = cudaLaunchKernelEx(&cl.cfg, lmh_collect_kernel, static_cast<const int64_t *>(logits), wsp, n, (int)k,
                                idx_bits);
    } else {
        // two rescoring CTAs per SM (one fits beside the scan's CTAs, the other starts as
        // they exit; measured 66.3 -> 64.8 us per call against one per SM, and no better
        // with three or four), none without rows
        const int64_t rows_cta = kScanWarps * 32;
        const int rgrid = (int)((N + rows_cta - 1) / rows_cta < 2 * nsm ? (N + rows_cta - 1) / rows_cta : 2 * nsm);
#define TGI_CPL_CASE(C)                                                                            \
    case C:                                                                                        \
        re = launch_rescore<C>(rgrid, st, lo, s, m, x, wsp, n, kk, k, idx_bits);                   \
        break;
        switch (cpl) {
            TGI_CPL_CASE(1) TGI_CPL_CASE(2) TGI_CPL_CASE(3) TGI_CPL_CASE(4) TGI_CPL_CASE(5)
            TGI_CPL_CASE(6) TGI_CPL_CASE(7) TGI_CPL_CASE(8)
        default:
            re = launch_rescore<16>(rgrid, st, lo, s, m, x, wsp, n, kk, k, idx_bits);
            break;
        }
#undef TGI_CPL_CASE
    }
    if (re != cudaSuccess)
        return TG_ERR_CUDA;
    const size_t final_smem = kFilterMax * sizeof(uint64_t) + sizeof(RadixSmem);
    if (cudaFuncSetAttribute(lmh_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)final_smem) != cudaSuccess)
        return TG_ERR_CUDA;
    PdlLaunch fl(1, kSelThreads, final_smem, st);
    if (cudaLaunchKernelEx(&fl.cfg, lmh_final_kernel, wsp, k, idx_bits, argmax, ids, scores, ncand) != cudaSuccess)
        return TG_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

extern "C" int tg_device_error(void *stream, int32_t *code)
{
    if (!code)
        return TG_ERR_ARG;
    int worst = TG_OK;
    const int r[4] = {tgi::gemv_take_device_error(stream), tgi::gemv_mma_take_device_error(stream),
                      tgi::lns8_take_device_error(stream), tgi::lmhead_take_device_error(stream)};
    for (int v : r) {
        if (v == TG_ERR_CUDA)
            return TG_ERR_CUDA;
        if (v != TG_OK)
            worst = v;
    }
    *code = worst;
    return TG_OK;
}
