// lns8_stateset.cu -- LNS8 eight-phase GEMV by the signed state-population
// route (BitState brief §4 "W_nonzero / W_negative" with §6, the reuse rule,
// and §8, the state-set candidates): the same A[r][8] and S[r] as the direct
// route, reached through popcounts of activation state masks.
//
// In the generic variant every lane of a group shares the row's scale code d,
// so all lanes with the same activation code a share one product code
// k = a + d - 74. The activation state of a lane is its code. For a state a,
//   A_a  = lanes with code a,   M = A_a & W_nonzero,
//   PNEG = activation_sign XOR W_negative,
//   C_a  = popcount(M) - 2 * popcount(M & PNEG)
// is the signed population of that state, and the row gains C_a * 2^(k >> 3)
// in phase k & 7 (k <= 0: nothing; k > 127: k = 127).
//
// Sparse state sets. The brief lists sparse (state, lane mask) pairs for the
// active states only, and warp ballot / match-any instead of a bit transpose.
// A group's 128 lanes are split into four 32-lane words; per word, one warp
// builds the list of (code, lane mask) entries of the codes present in that
// word: lane l of the warp takes the activation at bit l of the word, and
// __match_any_sync on the code returns the entry's mask itself. A state pays
// only in the words where it has lanes: about 85 entries per group for
// normally distributed codes instead of 4 x 45 word-state pairs. Entries with
// several lanes come first in each word's list; a single-lane entry needs no
// popcount (popcount of a word with at most one bit set is a bit test), which
// keeps the popcount pipe (a quarter of the integer rate) for the others.
//
// Reuse. The lists depend only on the activations; they are built once per
// CTA and applied to its 128 rows: "encode once per activation tile,
// intersect and count per row".
//
// Class sums on the tensor core. With e = d - 74 = 8 beta + delta, a state
// a = 8c + q lands in phase (q + delta) & 7 with band c + beta + [q + delta >=
// 8], so per (row, group) it is enough to form the class sums
//   G[row][q] = sum over entries of class q of C[row][entry] * 2^c,
// a contraction of C (rows x entries) with V (entries x 8), V[entry][q] =
// 2^c where the entry's code has class q. A 16x8x16 bf16 MMA takes 16 rows x
// 16 entries: C is in [-32, 32] and V a power of two, both exact in bf16, and
// every partial sum is an integer of magnitude at most 128 * 2^15 = 2^22, so
// fp32 accumulation is exact. The lane layout is the LNS8 fragment layout
// itself: lane (g, t) of a warp holds rows g and g + 8 of a 16-row block at
// the 32 lanes of word t, exactly the A-fragment rows it feeds, so each lane
// computes C for four entries of its own word per 16-entry tile. G is then
// shifted by beta + carry (exact either way: each term of G[q] is a multiple
// of 2^-shift when the shift is negative) into A[(q + delta) & 7].
//
// Clamps. A (warp, group) whose rows could clamp (decided from the group's
// smallest and largest nonzero code and the warp's scale codes) takes a
// checked loop: C of a (row, entry) with k <= 0 is set to 0, and with k > 127
// it goes to 2^15 in phase 7 instead.
//
// Reduction: int32 phase partials per CTA in shared memory, then the cluster
// push reduction and the fixed-order fp64 S of the direct route.

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "tg.h"
#include "tg_internal.h"

namespace {

namespace cg = cooperative_groups;

constexpr int kWarps = 8;           // warps per CTA; warp w owns one 16-row block
constexpr int kRows = kWarps * 16;  // rows per CTA
constexpr int kChunk = 8;           // groups whose entry lists are staged at once (one builder warp each)
constexpr int kListStride = 36;     // entries per word list: 32 + 4, so the four lists of a tile
                                    // sit in different banks
constexpr int kMaxCluster = 8;
constexpr unsigned kFull = 0xffffffffu;

struct WordMeta {
    int n, n_multi;    // entries, and of them those with several lanes
    int amin, amax;    // smallest and largest nonzero code of the word (amax = 0: none)
    uint32_t sg;       // activation sign, compact word
    uint32_t pad[3];
};

// bf16 pair (lo, hi) of two integers of magnitude below 2^8: the fp32 value
// from the 1.5 * 2^23 magic number, whose low 16 mantissa bits are zero.
__device__ __forceinline__ uint32_t bf16x2_int(int lo, int hi)
{
    const float flo = __int_as_float(0x4B400000 + lo) - 12582912.0f;
    const float fhi = __int_as_float(0x4B400000 + hi) - 12582912.0f;
    return __byte_perm(__float_as_uint(flo), __float_as_uint(fhi), 0x7632);
}

// Signed population of an entry in one row. kSingle: the mask has one lane.
template <bool kSingle>
__device__ __forceinline__ int entry_pop(uint32_t nz, uint32_t ne, uint32_t m)
{
    if (kSingle)
        return (nz & m) ? ((ne & m) ? -1 : 1) : 0;
    return __popc(nz & m) - 2 * __popc(ne & m);
}

// V of an entry for class n: bf16 2^(code >> 3) (bits 16..31 of y) if the
// entry's code has class n, else 0; padding entries carry y = 0.
__device__ __forceinline__ uint32_t v_of(uint32_t y, uint32_t n) { return ((y & 7u) == n) ? (y >> 16) : 0u; }

// bf16 bits of the signed population of a single-lane entry: +1, -1 or 0.
__device__ __forceinline__ uint32_t single_bf16(uint32_t nz, uint32_t ne, uint32_t m)
{
    return (nz & m) ? ((ne & m) ? 0xBF80u : 0x3F80u) : 0u;
}

// One 16-entry tile: C of this lane's four entries in its two rows -> A
// fragment, their V for class gq -> B fragment, one MMA.
template <bool kSingle, bool kChecked>
__device__ __forceinline__ void tile_step(const uint2 *L, int t, uint32_t nz0, uint32_t ne0, uint32_t nz1,
                                          uint32_t ne1, int e0, int e1, uint32_t gq, float (&d)[4], int &hi0,
                                          int &hi1)
{
    const uint4 p01 = *reinterpret_cast<const uint4 *>(L + 4 * t);
    const uint4 p23 = *reinterpret_cast<const uint4 *>(L + 4 * t + 2);
    const uint32_t m[4] = {p01.x, p01.z, p23.x, p23.z};
    const uint32_t y[4] = {p01.y, p01.w, p23.y, p23.w};
    const uint32_t b0 = v_of(y[0], gq) | (v_of(y[1], gq) << 16);
    const uint32_t b1 = v_of(y[2], gq) | (v_of(y[3], gq) << 16);
    if constexpr (kSingle && !kChecked) {
        tgi::mma_bf16_16816(d, single_bf16(nz0, ne0, m[0]) | (single_bf16(nz0, ne0, m[1]) << 16),
                       single_bf16(nz1, ne1, m[0]) | (single_bf16(nz1, ne1, m[1]) << 16),
                       single_bf16(nz0, ne0, m[2]) | (single_bf16(nz0, ne0, m[3]) << 16),
                       single_bf16(nz1, ne1, m[2]) | (single_bf16(nz1, ne1, m[3]) << 16), b0, b1);
    } else {
        int c0[4], c1[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            c0[i] = entry_pop<kSingle>(nz0, ne0, m[i]);
            c1[i] = entry_pop<kSingle>(nz1, ne1, m[i]);
            if (kChecked) {
                const int code = (int)(y[i] & 0x7fu);
                const int k0 = code + e0, k1 = code + e1;
                if ((unsigned)(k0 - 1) >= 127u) {
                    hi0 += k0 > 127 ? c0[i] : 0;
                    c0[i] = 0;
                }
                if ((unsigned)(k1 - 1) >= 127u) {
                    hi1 += k1 > 127 ? c1[i] : 0;
                    c1[i] = 0;
                }
            }
        }
        tgi::mma_bf16_16816(d, bf16x2_int(c0[0], c0[1]), bf16x2_int(c1[0], c1[1]), bf16x2_int(c0[2], c0[3]),
                       bf16x2_int(c1[2], c1[3]), b0, b1);
    }
}

// All tiles of a group: the leading tiles with multi-lane entries by popcount,
// the rest by bit tests.
__device__ __forceinline__ void scan_group_fast(const uint2 *L, int tiles_multi, int tiles, uint32_t nz0,
                                                uint32_t ne0, uint32_t nz1, uint32_t ne1, uint32_t gq, float (&d)[4])
{
    int h0 = 0, h1 = 0;
    int t = 0;
    for (; t < tiles_multi; t++)
        tile_step<false, false>(L, t, nz0, ne0, nz1, ne1, 0, 0, gq, d, h0, h1);
    for (; t < tiles; t++)
        tile_step<true, false>(L, t, nz0, ne0, nz1, ne1, 0, 0, gq, d, h0, h1);
}

// The same with the per-row k range applied; rare, so kept out of line.
__device__ __noinline__ void scan_group_checked(const uint2 *L, int tiles, uint32_t nz0, uint32_t ne0, uint32_t nz1,
                                                uint32_t ne1, int e0, int e1, uint32_t gq, float (&d)[4], int &hi0,
                                                int &hi1)
{
    for (int t = 0; t < tiles; t++)
        tile_step<false, true>(L, t, nz0, ne0, nz1, ne1, e0, e1, gq, d, hi0, hi1);
}

// Entry list of word j of a group (warp-wide): the entries with several
// lanes first, then the single-lane ones, then zero padding up to 32.
__device__ __forceinline__ void build_word(unsigned a, int lane, uint2 *list, WordMeta &M)
{
    const unsigned lt = (1u << lane) - 1u;
    const unsigned code = a & 0x7fu;
    const uint32_t sg = __ballot_sync(kFull, a >> 7);
    const unsigned mm = __match_any_sync(kFull, code);
    const bool leader = code != 0 && (mm & lt) == 0;
    const bool multi = leader && (mm & (mm - 1)) != 0;
    const unsigned bm = __ballot_sync(kFull, multi);
    const unsigned bs = __ballot_sync(kFull, leader && !multi);
    const int nm = __popc(bm), n = nm + __popc(bs);
    if (leader) {
        const int slot = multi ? __popc(bm & lt) : nm + __popc(bs & lt);
        list[slot] = make_uint2(mm, code | ((127u + (code >> 3)) << 23));
    }
    if (lane >= n)
        list[lane] = make_uint2(0u, 0u);
    const unsigned amin = __reduce_min_sync(kFull, code ? code : 255u);
    const unsigned amax = __reduce_max_sync(kFull, code);
    if (lane == 0) {
        M.n = n;
        M.n_multi = nm;
        M.amin = (int)amin;
        M.amax = (int)amax;
        M.sg = sg;
    }
}

struct PhaseF {
    double f[8];
};

__global__ void __launch_bounds__(kWarps * 32)
lns8_stateset_kernel(const uint4 *__restrict__ masks, const uint8_t *__restrict__ codes,
                     const uint8_t *__restrict__ xa, int64_t *__restrict__ A, double *__restrict__ S,
                     const __grid_constant__ PhaseF F, const double *__restrict__ Fd, int N, int G, int tiles,
                     int gpc)
{
    __shared__ __align__(16) uint2 lists[kChunk][4][kListStride];
    __shared__ WordMeta meta[kChunk][4];
    __shared__ int acc[kRows][8];                     // int32 phase partials of this CTA's groups
    __shared__ int stage[kRows + kMaxCluster][8];     // partials of the rows this CTA owns, per source CTA
    __shared__ int64_t arow[kRows][8];                // int64 A of the rows this CTA owns

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int csize = (int)cluster.num_blocks();
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t gq = (uint32_t)lane >> 2, tq = (uint32_t)lane & 3u;
    const int blk = blockIdx.x * kWarps + warp;       // 16-row block of this warp
    const bool blk_ok = blk < tiles;
    const int rl0 = warp * 16 + (int)gq;              // CTA-local rows rl0 and rl0 + 8
    const int row0 = blockIdx.x * kRows + rl0;
    const bool v0 = row0 < N, v1 = row0 + 8 < N;
    const int g_begin = rank * gpc;
    const int g_end = min(G, g_begin + gpc);

    for (int i = tid; i < kRows * 8; i += blockDim.x)
        (&acc[0][0])[i] = 0;

    for (int c0 = g_begin; c0 < g_end; c0 += kChunk) {
        const int ng = min(kChunk, g_end - c0);
        // weights and scale codes of the chunk's first group, in flight during the build
        uint4 wn = make_uint4(0u, 0u, 0u, 0u);
        int dn = 0;
        if (blk_ok) {
            wn = tgi::ldg_stream(masks + ((size_t)blk * G + c0) * 32 + lane);
            const uint8_t *dc = codes + ((size_t)blk * G + c0) * 16;
            dn = dc[gq] | (dc[gq + 8] << 8);
        }
        // entry lists: one (group, word) item per warp at a time
        // (the warp's activation bytes are loaded first, so that they are in flight together)
        static_assert(4 * kChunk % kWarps == 0, "the same number of items per warp");
        constexpr int kItems = 4 * kChunk / kWarps;
        unsigned av[kItems];
#pragma unroll
        for (int u = 0; u < kItems; u++) {
            const int item = min(warp + u * kWarps, 4 * ng - 1);
            av[u] = xa[(size_t)(c0 + (item >> 2)) * TG_GROUP + tgi::lns8_lane_col(item & 3, lane)];
        }
#pragma unroll
        for (int u = 0; u < kItems; u++) {
            const int item = warp + u * kWarps;
            if (item < 4 * ng)
                build_word(av[u], lane, lists[item >> 2][item & 3], meta[item >> 2][item & 3]);
        }
        __syncthreads();
        for (int gl = 0; gl < ng; gl++) {
            const uint4 w = wn;
            const int d0 = dn & 0xff, d1 = dn >> 8;
            if (blk_ok && gl + 1 < ng) {   // the next group's weights are in flight during this one
                wn = tgi::ldg_stream(masks + ((size_t)blk * G + c0 + gl + 1) * 32 + lane);
                const uint8_t *dc = codes + ((size_t)blk * G + c0 + gl + 1) * 16;
                dn = dc[gq] | (dc[gq + 8] << 8);
            }
            const WordMeta *M = meta[gl];
            int maxn = M[0].n, maxm = M[0].n_multi, amin = M[0].amin, amax = M[0].amax;
#pragma unroll
            for (int j = 1; j < 4; j++) {
                maxn = max(maxn, M[j].n);
                maxm = max(maxm, M[j].n_multi);
                amin = min(amin, M[j].amin);
                amax = max(amax, M[j].amax);
            }
            uint32_t nz0, ng0, nz1, ng1;
            tgi::lns8_compact_words(w, nz0, ng0, nz1, ng1);
            const uint32_t sg = M[tq].sg;
            const uint32_t ne0 = nz0 & (ng0 ^ sg), ne1 = nz1 & (ng1 ^ sg);
            const int e0 = d0 - 74, e1 = d1 - 74;

            // can any row of this warp clamp in this group? (rows past N have
            // zero weights and are left out)
            const int emin = (int)__reduce_min_sync(
                                 kFull, min(v0 ? (unsigned)(e0 + 128) : 511u, v1 ? (unsigned)(e1 + 128) : 511u)) - 128;
            const int emax = (int)__reduce_max_sync(
                                 kFull, max(v0 ? (unsigned)(e0 + 128) : 0u, v1 ? (unsigned)(e1 + 128) : 0u)) - 128;
            const bool safe = amax == 0 || (amin + emin >= 1 && amax + emax <= 127);

            float d[4] = {0.f, 0.f, 0.f, 0.f};
            int hi0 = 0, hi1 = 0;
            const uint2 *L = lists[gl][tq];
            const int tiles_g = (maxn + 3) >> 2, tiles_m = (maxm + 3) >> 2;
            if (safe)
                scan_group_fast(L, tiles_m, tiles_g, nz0, ne0, nz1, ne1, gq, d);
            else
                scan_group_checked(L, tiles_g, nz0, ne0, nz1, ne1, e0, e1, gq, d, hi0, hi1);

            // d = G[gq][2tq], G[gq][2tq+1], G[gq+8][2tq], G[gq+8][2tq+1]
#pragma unroll
            for (int r = 0; r < 2; r++) {
                const int e = r ? e1 : e0;
                const int delta = e & 7, beta = e >> 3;
#pragma unroll
                for (int c = 0; c < 2; c++) {
                    const int v = tgi::int_of_f32(d[2 * r + c]);
                    if (v != 0) {
                        const int q = 2 * (int)tq + c;
                        const int sh = beta + ((q + delta) >> 3);
                        atomicAdd(&acc[rl0 + 8 * r][(q + delta) & 7], sh >= 0 ? v << sh : v >> -sh);
                    }
                }
                const int h = r ? hi1 : hi0;
                if (h != 0)
                    atomicAdd(&acc[rl0 + 8 * r][7], h << 15);
            }
        }
        __syncthreads();   // the lists are rebuilt for the next chunk
    }

    // Cluster reduction: CTA `dst` of the cluster owns rows [dst * slice,
    // (dst + 1) * slice) of the 128; every CTA stores its partials of those
    // rows into the owner's staging area, one barrier makes them visible, and
    // each owner sums its slice in rank order.
    const int slice = (kRows + csize - 1) / csize;
    for (int item = tid; item < kRows * 8; item += blockDim.x) {
        const int rl = item >> 3, p = item & 7;
        const int dst = rl / slice;
        int *remote = cluster.map_shared_rank(&stage[0][0], dst);
        remote[((rank * slice) + (rl - dst * slice)) * 8 + p] = acc[rl][p];
    }
    cluster.sync();
    const int rows_here = min(slice, kRows - rank * slice);
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
        // S: the products A[p] * F[p], one thread per (row, phase), written over A in
        // shared memory, then one thread per row adds the eight terms in the order
        // p = 0..7 (fp64 is slow on this part: eight products per thread serialise)
        __syncthreads();
        static_assert(kWarps * 32 % 8 == 0, "a thread's phase p = tid & 7 is the same for all its items");
        double *prod = reinterpret_cast<double *>(&arow[0][0]);
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

namespace tgi {

int lns8_stateset(const uint4 *masks, const uint8_t *codes, const uint8_t *xa, int64_t *A, double *S,
                  const double F[8], const double *F_dev, int N, int G, int tiles, cudaStream_t s)
{
    PhaseF f;
    for (int p = 0; p < 8; p++)
        f.f[p] = F[p];
    const int gpc = (G + kMaxCluster - 1) / kMaxCluster;   // groups per CTA
    const int cl = (G + gpc - 1) / gpc;                     // CTAs per cluster, <= 8

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + kRows - 1) / kRows), (unsigned)cl);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)cl;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, lns8_stateset_kernel, masks, codes, xa, A, S, f, F_dev, N, G, tiles, gpc) !=
        cudaSuccess)
        return TG_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace tgi
