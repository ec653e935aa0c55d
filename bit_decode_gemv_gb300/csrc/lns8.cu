// lns8.cu -- LNS8 S1|E4|L3 eight-phase GEMV (BitState brief §3, §3.1, and the
// generic variant of §4, where the group's scale code is added before the
// L3/E4 split):
//
//   for every lane with t != 0 and activation code a != 0:
//     k = a + d[r][g] - 74;  k <= 0 -> exact zero;  k > 127 -> 127
//     A[r][k & 7] += (s_a XOR [t < 0]) ? -(1 << (k >> 3)) : (1 << (k >> 3))
//   S[r] = 2^-9 * sum_{p=0..7} A[r][p] * F[p],  F[p] = 2^((p - 2) / 8)
//
// Factorisation. Write the group's offset e = d - 74 = 8*beta + delta with
// delta = e & 7, and an activation code a = 8c + q. A lane then lands in phase
// (q + delta) & 7 with band c + beta + [q + delta >= 8]: the phase depends on
// the activation only through q, and the row only through delta and beta. So
// per (row, group) it is enough to form
//   G[q] = sum over lanes with a & 7 == q of  t * s_a * 2^c
// and add G[q] * 2^(beta + [q + delta >= 8]) into A[(q + delta) & 7]. This is
// exact when no lane of that (row, group) is clamped (k in 1..127 for every
// nonzero lane), which is checked per (row, group) from the group's smallest
// and largest nonzero activation code. In a (row, group) that can clamp, the
// lanes that do clamp -- found from a per-warp list of the group's lanes that
// can clamp for any of the warp's rows -- are taken back out of G, and their
// saturated value (+-2^15 in phase 7, or nothing for k <= 0) is added
// directly; the rest stays on the factorised path.
//
// G is a contraction t (rows x lanes) . V (lanes x 8) with V[i][q] = s_i 2^c_i
// when a_i & 7 == q, else 0. Every entry (+-1, +-2^c) is exact in bf16 and
// every partial sum is an integer below 2^23, so a bf16 tensor-core product
// with fp32 accumulation is exact. A 16x8x16 warp-level MMA takes 16 rows x 16
// lanes of t from registers (converted straight from the packed mask pair, two
// integer ops per weight) against the 16 x 8 slice of V, N = 8 = the phases.
// The tensor core here routes rather than multiplies: the work is the trit
// conversion, and the warp-level MMA, fed from registers, avoids staging the
// expanded weights anywhere.
//
// Mapping: a CTA owns 128 rows and a slice of the groups; a cluster of up to 8
// CTAs covers all groups of those rows. Two warps share each 16-row block
// (warps w and w + 8: rows 16(w % 8)..+15), each taking half of every chunk of
// four groups, so twice as many warps hide the MMA and conversion latency.
// Each CTA keeps int32 phase partials in shared memory, one array per group
// half; each CTA of the cluster then
// owns a slice of the rows, gathers their partials from the other CTAs through
// distributed shared memory, sums them into int64 A and materialises S with
// explicitly rounded fp64 multiplies and adds in the order p = 0..7.

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "device_common.cuh"
#include "tg.h"
#include "tg_internal.h"

TGI_DEFINE_DEVICE_ERROR(lns8_take_device_error)

namespace {

namespace cg = cooperative_groups;

constexpr int kRowWarps = 8;               // 16-row blocks per CTA
constexpr int kWarps = 2 * kRowWarps;      // warps per CTA: two per 16-row block, each half of a chunk's groups
constexpr int kRows = kRowWarps * 16;      // rows per CTA
constexpr int kChunkGroups = 4;            // groups per step: V fragments staged, weights in flight
constexpr int kMaxCluster = 8;

struct PhaseF {
    double f[8];
};

// bf16 bit pattern of (-1)^sign * 2^c.
__device__ __forceinline__ uint32_t bf16_pow2(uint32_t sign, uint32_t c) { return (sign << 15) | ((127u + c) << 7); }

// bf16x2 A register from pair rp of a packed word: W_nonzero bits at 7-rp and
// 23-rp become the bf16 one (0x3F80) of each half, W_negative bits at 15-rp and
// 31-rp its sign.
template <int RP>
__device__ __forceinline__ uint32_t frag_pair(uint32_t w)
{
    return ((w & (0x00800080u >> RP)) * (0x7Fu << RP)) | ((w << RP) & 0x80008000u);
}

// One V value: (a != 0 and a & 7 == q) ? bf16(+-2^(a >> 3)) : 0.
__device__ __forceinline__ uint32_t v_entry(uint32_t xab, uint32_t q)
{
    const uint32_t a = xab & 0x7fu;
    return (a != 0u && (a & 7u) == q) ? bf16_pow2(xab >> 7, a >> 3) : 0u;
}

// Exact correction of the lanes that clamp. A lane of a (row, group) clamps when
// its product code k = a + e leaves 1..127 (e = the row's scale code - 74):
// k <= 0 contributes nothing and k > 127 contributes +-2^15 in phase 7, but the
// factorised class sum G[a & 7] holds its +-2^(a >> 3) as if k were in range.
// For each group, every warp lists once the lanes that can clamp for ANY of its
// rows -- nonzero codes with a + min(e) <= 0 or a + max(e) > 127, over the
// warp's rows below N -- and the (row, group) that can clamp walks only that
// list: each listed lane whose weight is nonzero and that does clamp for the
// row has its term taken back out of its class sum (into gcorr, the row's class
// corrections) and its saturated value, if any, added to the phase-7 term. Every
// other lane stays on the factorised path, where it is exact. The list is split
// by the quad thread that holds the lane's mask bits (lane 16kc + o of the
// group: thread (o & 7) >> 1 of the quad, byte (o & 1) + 2 (o >> 3) of chunk kc).
// Entry: code a (bits 0-6), activation sign (bit 7), chunk kc (bits 8-10), byte
// bi (bits 11-12).
constexpr int kListMax = 32;   // lanes of a group one quad thread holds

// Build this warp's lists for one group (called by the whole warp): x4 = the
// group's activation bytes 4 lane .. 4 lane + 3; emin/emax = the warp's e range.
__device__ __forceinline__ void build_clamp_lists(uint32_t x4, int emin, int emax, uint16_t (*list)[kListMax],
                                                  int *cnt)
{
    const int lane = threadIdx.x & 31;
    if (lane < 4)
        cnt[lane] = 0;
    __syncwarp();
#pragma unroll
    for (int b = 0; b < 4; b++) {
        const uint32_t xab = (x4 >> (8 * b)) & 0xffu;
        const int a = (int)(xab & 0x7fu);
        if (a != 0 && (a + emin <= 0 || a + emax > 127)) {
            const int i = 4 * lane + b, o = i & 15;
            const int tq = (o & 7) >> 1;
            const int bi = (o & 1) + 2 * (o >> 3);
            const int slot = atomicAdd(cnt + tq, 1);
            list[tq][slot] = (uint16_t)(a | (int)(xab & 0x80u) | ((i >> 4) << 8) | (bi << 11));
        }
    }
    __syncwarp();
}

// Walk this quad thread's list for the rows (halves) that need it.
__device__ __forceinline__ void walk_clamp_list(const uint16_t *list, int n, const uint32_t (&w4)[4], const int (&e)[2],
                                                const bool (&need)[2], int *const (&gcorr)[2], int (&clamp)[2])
{
    clamp[0] = clamp[1] = 0;
    for (int j = 0; j < n; j++) {
        const uint32_t ent = list[j];
        const int a = (int)(ent & 0x7fu);
        const uint32_t sgn = (ent >> 7) & 1u;
        const int kc = (int)(ent >> 8) & 7, bi = (int)(ent >> 11) & 3;
        const int wi = kc >> 1;
        const uint32_t w = wi == 0 ? w4[0] : wi == 1 ? w4[1] : wi == 2 ? w4[2] : w4[3];
#pragma unroll
        for (int half = 0; half < 2; half++) {
            if (!need[half])
                continue;
            const int rp = 4 * (kc & 1) + half + 2 * (bi >> 1);
            const int h = bi & 1;
            if (((w >> (16 * h + 7 - rp)) & 1u) == 0u)
                continue;
            const int k = a + e[half];
            if (k > 0 && k <= 127)
                continue;
            const bool minus = (sgn ^ ((w >> (16 * h + 15 - rp)) & 1u)) != 0u;
            const int v = 1 << (a >> 3);
            atomicAdd(gcorr[half] + (a & 7), minus ? v : -v);
            if (k > 127)
                clamp[half] += minus ? -(1 << 15) : (1 << 15);
        }
    }
}

__global__ void __launch_bounds__(kWarps * 32, 2)
lns8_mma_kernel(const uint4 *__restrict__ masks, const uint8_t *__restrict__ codes,
                const uint8_t *__restrict__ xa, int64_t *__restrict__ A, double *__restrict__ S,
                const __grid_constant__ PhaseF F, const double *__restrict__ Fd, int N, int G, int gpc)
{
    __shared__ uint2 vfrag[kChunkGroups][8][32];   // V fragments (b0, b1) per group, chunk, lane
    __shared__ unsigned gmin[kChunkGroups], gmax[kChunkGroups];
    __shared__ int acc[2][kRows][8];               // int32 phase partials of this CTA's groups, per group half
    __shared__ int stage[kRows + kMaxCluster][8];  // partials of the rows this CTA owns, per source CTA
    __shared__ int gcorr[kWarps][16][8];           // class-sum corrections of clamped lanes, per warp row
    __shared__ int64_t arow[kRows][8];             // int64 A of the rows this CTA owns
    __shared__ uint16_t clist[kWarps][4][kListMax];  // per warp: the lanes of a group that can clamp, by quad thread
    __shared__ int ccnt[kWarps][4];

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int csize = (int)cluster.num_blocks();
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int rw = warp & (kRowWarps - 1);           // this warp's 16-row block of the CTA
    const int gh = warp / kRowWarps;                 // and its half of each chunk's groups
    const int rb = blockIdx.x * kRowWarps + rw;      // 16-row block of this warp in the matrix
    const int g_begin = rank * gpc;
    const int g_end = min(G, g_begin + gpc);

    // (acc needs no clearing where a warp has a group: its first group stores its
    // rows' partials; a warp whose half of the first chunk is empty clears them)
    for (int i = tid; i < kWarps * 16 * 8; i += blockDim.x)
        (&gcorr[0][0][0])[i] = 0;

    const bool active = rb * 16 < N;   // warp-uniform
    if (2 * gh >= min(kChunkGroups, g_end - g_begin))
        for (int i = lane; i < 16 * 8; i += 32)
            acc[gh][rw * 16 + (i >> 3)][i & 7] = 0;
    for (int c0 = g_begin; c0 < g_end; c0 += kChunkGroups) {
        const int ng = min(kChunkGroups, g_end - c0);
        // this warp's masks and scale codes for its half of the chunk (groups
        // 2 gh, 2 gh + 1), issued before the shared-memory set-up so the weight
        // stream overlaps it
        constexpr int kHalf = kChunkGroups / 2;
        uint4 wv[kHalf];
        int ec[kHalf][2];
        uint32_t xw[kChunkGroups];   // activation bytes 4 lane .. 4 lane + 3 of each group (range, clamp lists)
        uint32_t xb[kHalf][2];       // this thread's V entries' activation byte pairs
        static_assert(kRowWarps * 32 == 256 && kWarps == 2 * kRowWarps,
                      "one V entry (chunk, lane) per thread and group of its half");
        const int vkc = (tid >> 5) & 7, vln = tid & 31, vgh = tid >> 8;
#pragma unroll
        for (int j = 0; j < kHalf; j++) {
            const int gl = kHalf * gh + j;
            wv[j] = make_uint4(0, 0, 0, 0);
            ec[j][0] = ec[j][1] = 0;
            if (active && gl < ng) {
                const size_t unit = (size_t)rb * G + c0 + gl;
                wv[j] = tgi::ldg_stream(masks + unit * 32 + lane);
                ec[j][0] = (int)__ldg(codes + unit * 16 + gq) - 74;
                ec[j][1] = (int)__ldg(codes + unit * 16 + gq + 8) - 74;
            }
        }
        // the activations, for every warp (all threads build V): issued with the weights
#pragma unroll
        for (int gl = 0; gl < kChunkGroups; gl++) {
            const int gx = c0 + min(gl, ng - 1);
            xw[gl] = __ldg(reinterpret_cast<const uint32_t *>(xa + (size_t)gx * TG_GROUP) + lane);
        }
#pragma unroll
        for (int j = 0; j < kHalf; j++) {
            const int gx = c0 + min(kHalf * vgh + j, ng - 1);
            const uint16_t *xg = reinterpret_cast<const uint16_t *>(xa + (size_t)gx * TG_GROUP + 16 * vkc) + (vln & 3);
            xb[j][0] = __ldg(xg);
            xb[j][1] = __ldg(xg + 4);
        }
        __syncthreads();
        // V fragments: thread (q, j) of chunk kc holds V rows 2j, 2j+1 (b0) and
        // 2j+8, 2j+9 (b1) of column q; thread tid builds entry (kc, ln) =
        // ((tid / 32) % 8, tid % 32) of the groups of its half of the chunk from
        // the byte pairs it loaded above (lanes 16 kc + 2 (ln & 3) + {0, 1} and
        // + {8, 9})
        {
            const uint32_t q = (uint32_t)(vln >> 2);
#pragma unroll
            for (int j = 0; j < kHalf; j++) {
                const int gl = kHalf * vgh + j;
                if (gl < ng) {
                    const uint32_t p0 = xb[j][0], p1 = xb[j][1];
                    const uint32_t b0 = v_entry(p0 & 0xffu, q) | (v_entry(p0 >> 8, q) << 16);
                    const uint32_t b1 = v_entry(p1 & 0xffu, q) | (v_entry(p1 >> 8, q) << 16);
                    vfrag[gl][vkc][vln] = make_uint2(b0, b1);
                }
            }
        }
        // smallest and largest nonzero activation code of each group
        static_assert(kChunkGroups <= kWarps, "warp gl finds group gl's range");
        if (warp < ng) {
            const int gl = warp;
            const uint32_t v4 = gl == 0 ? xw[0] : gl == 1 ? xw[1] : gl == 2 ? xw[2] : xw[3];
            unsigned lo = 128u, hi = 0u;
#pragma unroll
            for (int b = 0; b < 4; b++) {
                const unsigned a = (v4 >> (8 * b)) & 0x7fu;
                if (a) {
                    lo = min(lo, a);
                    hi = max(hi, a);
                }
            }
            lo = __reduce_min_sync(0xffffffffu, lo);
            hi = __reduce_max_sync(0xffffffffu, hi);
            if (lane == 0) {
                gmin[gl] = lo;
                gmax[gl] = hi;
            }
        }
        __syncthreads();

        if (active) {
#pragma unroll
            for (int j = 0; j < kHalf; j++) {
                const int gl = kHalf * gh + j;
                if (gl >= ng)
                    break;
                const uint32_t w4[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
                const bool first = c0 == g_begin && j == 0;   // this warp's first group: store, not add
                // two independent accumulation chains (even and odd chunks);
                // each partial is an integer of magnitude below 2^23, so the
                // fp32 sums and their final sum are exact
                float d[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kc = 0; kc < 8; kc += 2) {
                    const uint32_t w = w4[kc >> 1];
                    const uint2 b0 = vfrag[gl][kc][lane], b1 = vfrag[gl][kc + 1][lane];
                    tgi::mma_bf16_16816(d, frag_pair<0>(w), frag_pair<1>(w), frag_pair<2>(w), frag_pair<3>(w), b0.x, b0.y);
                    tgi::mma_bf16_16816(d1, frag_pair<4>(w), frag_pair<5>(w), frag_pair<6>(w), frag_pair<7>(w), b1.x, b1.y);
                }
#pragma unroll
                for (int i = 0; i < 4; i++)
                    d[i] += d1[i];
                const int lo = (int)gmin[gl], hi = (int)gmax[gl];
                // quad-uniform: the four threads of a quad hold the same two rows.
                // Rows past N (zero weights, scale code 0) never need the clamp
                // correction.
                const int e[2] = {ec[j][0], ec[j][1]};
                bool need[2];
#pragma unroll
                for (int half = 0; half < 2; half++)
                    need[half] = !(lo > 127 || (lo + e[half] >= 1 && hi + e[half] <= 127) ||
                                   rb * 16 + gq + 8 * half >= N);
                int clamp[2] = {0, 0};
                if (__any_sync(0xffffffffu, need[0] || need[1])) {
                    // the warp's e range over its rows below N, then its lists for this group
                    int emin = 1 << 20, emax = -(1 << 20);
#pragma unroll
                    for (int half = 0; half < 2; half++)
                        if (rb * 16 + gq + 8 * half < N) {
                            emin = min(emin, e[half]);
                            emax = max(emax, e[half]);
                        }
                    emin = __reduce_min_sync(0xffffffffu, emin);
                    emax = __reduce_max_sync(0xffffffffu, emax);
                    build_clamp_lists(xw[gl], emin, emax, clist[warp], ccnt[warp]);
                }
                if (need[0] || need[1]) {
                    int *const gc[2] = {gcorr[warp][gq], gcorr[warp][gq + 8]};
                    const unsigned qmask = 0xfu << (lane & ~3);
                    walk_clamp_list(clist[warp][tq], ccnt[warp][tq], w4, e, need, gc, clamp);
                    __syncwarp(qmask);
#pragma unroll
                    for (int half = 0; half < 2; half++) {   // this thread's two classes of each row
                        d[2 * half] += (float)gc[half][2 * tq];
                        d[2 * half + 1] += (float)gc[half][2 * tq + 1];
                        gc[half][2 * tq] = 0;
                        gc[half][2 * tq + 1] = 0;
                        clamp[half] += __shfl_xor_sync(qmask, clamp[half], 1);
                        clamp[half] += __shfl_xor_sync(qmask, clamp[half], 2);
                    }
                }
#pragma unroll
                for (int half = 0; half < 2; half++) {
                    int *acc_row = acc[gh][rw * 16 + gq + 8 * half];
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        const int q = 2 * tq + c;
                        const int v = __float2int_rn(d[2 * half + c]);
                        const int sidx = q + (e[half] & 7);
                        const int sh = max(-31, min(31, (e[half] >> 3) + (sidx >> 3)));
                        int add = sh >= 0 ? (v << sh) : (v >> -sh);
                        if ((sidx & 7) == 7)
                            add += clamp[half];
                        // the quad's eight (thread, j) pairs cover the eight phases once per group
                        if (first)
                            acc_row[sidx & 7] = add;
                        else
                            acc_row[sidx & 7] += add;
                    }
                }
                __syncwarp();
            }
        }
    }
    // Cluster reduction: CTA `dst` of the cluster owns rows [dst * slice,
    // (dst + 1) * slice) of the 128; every CTA stores its partials of those rows
    // into the owner's staging area, one barrier makes them visible, and each
    // owner sums its slice in rank order.
    __syncthreads();
    const int slice = (kRows + csize - 1) / csize;
    for (int item = tid; item < kRows * 8; item += blockDim.x) {
        const int rl = item >> 3, p = item & 7;
        const int dst = rl / slice;
        int *remote = cluster.map_shared_rank(&stage[0][0], dst);
        remote[((rank * slice) + (rl - dst * slice)) * 8 + p] = acc[0][rl][p] + acc[1][rl][p];
    }
    cluster.sync();
    // A: the owner sums its slice's partials in rank order
    const int rows_here = min(slice, kRows - rank * slice);   // rows of this CTA's slice (last slice may be short)
    for (int item = tid; item < rows_here * 8; item += blockDim.x) {
        const int i = item >> 3, p = item & 7;
        const int row = blockIdx.x * kRows + rank * slice + i;
        int64_t a = 0;
#pragma unroll
        for (int src = 0; src < kMaxCluster; src++)
            if (src < csize)
                a += stage[src * slice + i][p];
        arow[i][p] = a;
        if (row < N)
            A[(size_t)row * 8 + p] = a;
    }
    if (S) {
        // S: the products A[p] * F[p], one thread per (row, phase), written over A
        // in shared memory (fp64 is slow on this part: a thread per row doing all
        // eight measured ~2000 cycles), then one thread per row adds the eight
        // terms in the order p = 0..7
        __syncthreads();
        double *prod = reinterpret_cast<double *>(&arow[0][0]);
        static_assert(kWarps * 32 % 8 == 0, "a thread's phase p = tid & 7 is the same for all its items");
        // the caller's F[p] (device memory) when given, else the built-in grid constant
        const double fp = Fd ? Fd[tid & 7] : F.f[tid & 7];
        for (int item = tid; item < rows_here * 8; item += blockDim.x)
            prod[item] = __dmul_rn((double)arow[item >> 3][item & 7], fp);
        __syncthreads();
        for (int i = tid; i < rows_here; i += blockDim.x) {
            const int row = blockIdx.x * kRows + rank * slice + i;
            if (row < N) {
                double sum = 0.0;
#pragma unroll
                for (int p = 0; p < 8; p++)
                    sum = __dadd_rn(sum, prod[i * 8 + p]);
                S[row] = __dmul_rn(sum, 0x1p-9);
            }
        }
    }
}

}  // namespace

extern "C" int tg_gemv_lns8_phase(const tg_layout *L, const void *w, const uint8_t *xa, const double *F_dev,
                                  int64_t *A, double *S, void *stream)
{
    if (!L || !w || !xa || !A)
        return TG_ERR_ARG;
    const bool pure = (L->flags & TG_FLAG_LNS8_PURE_LNS) != 0;
    if (L->kind != TG_TERNARY_LNS8 || L->version != 1)
        return TG_ERR_ARG;
    if (pure ? (L->frac < 1 || L->frac > 6 || (L->flags & TG_FLAG_LNS8_STATE_SET)) : L->frac != 0)
        return TG_ERR_ARG;   // frac is the pure route's internal precision, 0 otherwise
    if (pure && F_dev)
        return TG_ERR_ARG;   // the pure route's S is a log-domain value; it takes no F
    if (!tgi::aligned(w, 256) || !tgi::aligned(xa, 16) || !tgi::aligned(A, 8) ||
        (S && !tgi::aligned(S, 8)) || (F_dev && !tgi::aligned(F_dev, 8)))
        return TG_ERR_ARG;
    if (L->N < 1 || L->K < TG_GROUP || L->K % TG_GROUP)
        return TG_ERR_SHAPE;
    if (L->K >= 65536)   // int32 phase partials per CTA: |sum| <= K * 2^15 < 2^31
        return TG_ERR_BOUND;

    PhaseF F;
    for (int p = 0; p < 8; p++)
        F.f[p] = std::exp2((double)(p - 2) / 8.0);

    const auto *base = static_cast<const unsigned char *>(w);
    const uint4 *masks = reinterpret_cast<const uint4 *>(base + L->mask_off);
    const uint8_t *codes = base + L->scale_off;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int G = (int)L->G, N = (int)L->N;
    if (L->flags & TG_FLAG_LNS8_STATE_SET)
        return tgi::lns8_stateset(masks, codes, xa, A, S, F.f, F_dev, N, G, (int)L->tiles, s);
    if (pure)
        return tgi::lns8_purelns(masks, codes, xa, A, S, N, G, (int)L->frac, s);
    const int gpc = (G + kMaxCluster - 1) / kMaxCluster;   // groups per CTA
    const int csize = (G + gpc - 1) / gpc;                 // CTAs per cluster, <= 8

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + kRows - 1) / kRows), (unsigned)csize);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)csize;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, lns8_mma_kernel, masks, codes, xa, A, S, F, F_dev, N, G, gpc) != cudaSuccess)
        return TG_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}
