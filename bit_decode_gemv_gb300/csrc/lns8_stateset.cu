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
// A group's 128 lanes are split into four 32-lane words; one warp builds, per
// word, the list of (code, lane mask) pairs of the codes present in that word:
// lane l of the warp takes the activation at bit l of the word, and
// __match_any_sync on the code returns the mask itself. Entries are stored
// sorted by (word, code & 7). A state contributes only in the words where it
// has lanes, so a row pays two popcounts per (row, entry) and about 85 entries
// per group on normally distributed codes, not 4 x 45 word-state pairs.
//
// Reuse. The entry list depends only on the activations: the warp that builds
// it applies it to 64 rows (lane = rows q and q + 8 of one of four 16-row
// blocks), which is the "encode once per activation tile, intersect and count
// per row" split of the brief.
//
// Bit order. The weight blob is the LNS8 fragment layout (16-row blocks; entry
// 4q + j of a group holds rows q and q + 8 at lanes 16c + {2j, 2j+1, 2j+8,
// 2j+9}). A lane converts its four entries j into one W_nonzero and one
// effective-negative word per row and j, with two byte permutes and two
// shift-and-merge steps per word pair; the activation masks use the bit order
// this conversion produces (lane_col below), so no bit transpose is needed.
//
// Phase factorisation, as in the direct route: with e = d - 74 = 8 beta +
// delta, a state a = 8c + q lands in phase (q + delta) & 7 with band c + beta +
// [q + delta >= 8]. Per (row, group) the kernel sums G[q] = sum C_a 2^c over
// the entries of phase class q (an unrolled loop per class, so the eight sums
// stay in registers) and adds G[q] * 2^(beta + carry) into A[(q + delta) & 7]
// (an exact shift either way: every term of G[q] is a multiple of 2^-shift
// when the shift is negative). Where a row can clamp in a group (decided from
// the group's smallest and largest nonzero code), the whole warp takes a
// checked loop that leaves out k <= 0 and sends k > 127 to 2^15 in phase 7.
//
// Cost. Popcount issues at a quarter of the integer rate per SM, and there
// are 4 popcounts per (lane, entry), so the route is popcount-bound. It beats
// the direct route only where activations have few distinct codes per group;
// the reuse and cardinality sweeps measure where.
//
// Reduction: int32 phase partials per CTA in shared memory, then the same
// cluster push reduction and fixed-order fp64 S as the direct route.

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "tg.h"
#include "tg_internal.h"

namespace {

namespace cg = cooperative_groups;

constexpr int kWarps = 8;          // warps per CTA; each owns whole groups
constexpr int kRows = 64;          // rows per CTA: four 16-row blocks
constexpr int kMaxCluster = 8;
constexpr int kMaxEntries = 128;   // (word, code) entries of a group: at most one per lane
constexpr unsigned kFull = 0xffffffffu;

// Group lane held at bit `bit` of compact word j (the order the weight
// conversion below produces for both rows of a lane).
__device__ __forceinline__ int lane_col(int j, int bit)
{
    const int x = 7 - (bit & 7);
    const int c = (x >> 2) + 2 * ((bit >> 3) & 1) + 4 * (x & 1);
    return 16 * c + 2 * j + 8 * ((x >> 1) & 1) + (bit >> 4);
}

struct RowWords {
    uint32_t nz[4];   // W_nonzero, compact word j
    uint32_t ng[4];   // W_negative, compact word j (activation sign applied later)
};

// One 16-byte LNS8 entry (words u = 0..3) -> compact word j of rows q and q+8.
__device__ __forceinline__ void convert_entry(uint4 w, int j, RowWords &rq, RowWords &rq8)
{
    const uint32_t nza0 = __byte_perm(w.x, w.y, 0x6240), nga0 = __byte_perm(w.x, w.y, 0x7351);
    const uint32_t nza1 = __byte_perm(w.z, w.w, 0x6240), nga1 = __byte_perm(w.z, w.w, 0x7351);
    rq.nz[j] = (nza0 & 0xAAAAAAAAu) | ((nza1 >> 1) & 0x55555555u);
    rq8.nz[j] = ((nza0 << 1) & 0xAAAAAAAAu) | (nza1 & 0x55555555u);
    rq.ng[j] = (nga0 & 0xAAAAAAAAu) | ((nga1 >> 1) & 0x55555555u);
    rq8.ng[j] = ((nga0 << 1) & 0xAAAAAAAAu) | (nga1 & 0x55555555u);
}

// Entry scan of one group for the two rows of a lane. kChecked: apply the
// per-row k range (k <= 0 dropped, k > 127 counted into hi).
template <bool kChecked>
__device__ __forceinline__ void scan_group(const uint2 *list, const int *offs, const uint32_t (&nz0)[4],
                                           const uint32_t (&ne0)[4], const uint32_t (&nz1)[4],
                                           const uint32_t (&ne1)[4], int e0, int e1, int (&g0)[8],
                                           int (&g1)[8], int &hi0, int &hi1)
{
#pragma unroll
    for (int j = 0; j < 4; j++) {
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const int b = offs[8 * j + q], end = offs[8 * j + q + 1];
            for (int e = b; e < end; e++) {
                const uint2 en = list[e];
                const int pw = (int)(en.y & 0xffffu);
                const int c0 = __popc(nz0[j] & en.x) - 2 * __popc(ne0[j] & en.x);
                const int c1 = __popc(nz1[j] & en.x) - 2 * __popc(ne1[j] & en.x);
                if (kChecked) {
                    const int code = (int)(en.y >> 16);
                    const int k0 = code + e0, k1 = code + e1;
                    g0[q] += ((unsigned)(k0 - 1) < 127u) ? c0 * pw : 0;
                    g1[q] += ((unsigned)(k1 - 1) < 127u) ? c1 * pw : 0;
                    hi0 += k0 > 127 ? c0 : 0;
                    hi1 += k1 > 127 ? c1 : 0;
                } else {
                    g0[q] += c0 * pw;
                    g1[q] += c1 * pw;
                }
            }
        }
    }
}

// G[q] * 2^(beta + carry) into phase (q + delta) & 7 of one row's partials.
__device__ __forceinline__ void route_row(int *acc_row, const int (&g)[8], int hi, int e)
{
    const int delta = e & 7, beta = e >> 3;
#pragma unroll
    for (int q = 0; q < 8; q++) {
        const int v = g[q];
        if (v != 0) {
            const int sh = beta + ((q + delta) >> 3);
            atomicAdd(&acc_row[(q + delta) & 7], sh >= 0 ? v << sh : v >> -sh);
        }
    }
    if (hi != 0)
        atomicAdd(&acc_row[7], hi << 15);
}

struct PhaseF {
    double f[8];
};

__global__ void __launch_bounds__(kWarps * 32)
lns8_stateset_kernel(const uint4 *__restrict__ masks, const uint8_t *__restrict__ codes,
                     const uint8_t *__restrict__ xa, int64_t *__restrict__ A, double *__restrict__ S,
                     PhaseF F, int N, int G, int tiles, int gpc)
{
    __shared__ uint2 list[kWarps][kMaxEntries];       // (lane mask, code << 16 | 2^(code >> 3))
    __shared__ int offs[kWarps][33];                  // entry offsets per (word, phase class)
    __shared__ int acc[kRows][8];                     // int32 phase partials of this CTA's groups
    __shared__ int stage[kRows + kMaxCluster][8];     // partials of the rows this CTA owns, per source CTA
    __shared__ int64_t arow[kRows][8];                // int64 A of the rows this CTA owns

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int csize = (int)cluster.num_blocks();
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int q = lane & 7;                               // rows q and q + 8 of ...
    const int blk = blockIdx.x * (kRows / 16) + (lane >> 3);   // ... this 16-row block
    const int rl0 = 16 * (lane >> 3) + q;                 // CTA-local row of the first of them
    const bool blk_ok = blk < tiles;
    const int g_begin = rank * gpc;
    const int g_end = min(G, g_begin + gpc);
    const unsigned lt = (1u << lane) - 1u;

    for (int i = tid; i < kRows * 8; i += blockDim.x)
        (&acc[0][0])[i] = 0;
    __syncthreads();

    for (int g = g_begin + warp; g < g_end; g += kWarps) {
        // weights of this lane's two rows (issued first, used after the build)
        uint4 wv[4] = {};
        int d0 = 0, d1 = 0;
        if (blk_ok) {
            const uint4 *src = masks + ((size_t)blk * G + g) * 32 + 4 * q;
#pragma unroll
            for (int j = 0; j < 4; j++)
                wv[j] = tgi::ldg_stream(src + j);
            const uint8_t *dc = codes + ((size_t)blk * G + g) * 16;
            d0 = dc[q];
            d1 = dc[q + 8];
        }

        // state sets of this group: per word, one entry per code present
        uint32_t sg[4];
        int base = 0;
        unsigned amin = 255u, amax = 0u;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const unsigned a = xa[(size_t)g * TG_GROUP + lane_col(j, lane)];
            const unsigned code = a & 0x7fu;
            sg[j] = __ballot_sync(kFull, a >> 7);
            amin = min(amin, code ? code : 255u);
            amax = max(amax, code);
            const unsigned mm = __match_any_sync(kFull, code);
            const bool leader = code != 0 && (mm & lt) == 0;
            int slot = 0;
#pragma unroll
            for (int c = 0; c < 8; c++) {
                const bool mine = leader && (int)(code & 7u) == c;
                const unsigned bal = __ballot_sync(kFull, mine);
                if (mine)
                    slot = base + __popc(bal & lt);
                if (lane == 0)
                    offs[warp][8 * j + c] = base;
                base += __popc(bal);
            }
            if (leader)
                list[warp][slot] = make_uint2(mm, (code << 16) | (1u << (code >> 3)));
        }
        if (lane == 0)
            offs[warp][32] = base;
        amin = __reduce_min_sync(kFull, amin);
        amax = __reduce_max_sync(kFull, amax);
        __syncwarp();

        // this lane's rows: compact W_nonzero and effective-negative words
        RowWords r0, r1;
#pragma unroll
        for (int j = 0; j < 4; j++)
            convert_entry(wv[j], j, r0, r1);
        uint32_t ne0[4], ne1[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            ne0[j] = r0.nz[j] & (r0.ng[j] ^ sg[j]);
            ne1[j] = r1.nz[j] & (r1.ng[j] ^ sg[j]);
        }

        const int e0 = d0 - 74, e1 = d1 - 74;
        const bool any = amax != 0;
        const bool fast = !any || ((int)amin + min(e0, e1) >= 1 && (int)amax + max(e0, e1) <= 127);
        int g0[8] = {0, 0, 0, 0, 0, 0, 0, 0}, g1[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        int hi0 = 0, hi1 = 0;
        if (__all_sync(kFull, fast))
            scan_group<false>(list[warp], offs[warp], r0.nz, ne0, r1.nz, ne1, e0, e1, g0, g1, hi0, hi1);
        else
            scan_group<true>(list[warp], offs[warp], r0.nz, ne0, r1.nz, ne1, e0, e1, g0, g1, hi0, hi1);
        route_row(acc[rl0], g0, hi0, e0);
        route_row(acc[rl0 + 8], g1, hi1, e1);
        __syncwarp();   // the list and offsets are rebuilt for the next group
    }

    // Cluster reduction: CTA `dst` of the cluster owns rows [dst * slice,
    // (dst + 1) * slice) of the 64; every CTA stores its partials of those rows
    // into the owner's staging area, one barrier makes them visible, and each
    // owner sums its slice in rank order.
    __syncthreads();
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
        __syncthreads();
        for (int i = tid; i < rows_here; i += blockDim.x) {
            const int row = blockIdx.x * kRows + rank * slice + i;
            if (row < N) {
                double sum = 0.0;
#pragma unroll
                for (int p = 0; p < 8; p++)
                    sum = __dadd_rn(sum, __dmul_rn((double)arow[i][p], F.f[p]));
                S[row] = __dmul_rn(sum, 0x1p-9);
            }
        }
    }
}

}  // namespace

namespace tgi {

int lns8_stateset(const uint4 *masks, const uint8_t *codes, const uint8_t *xa, int64_t *A, double *S,
                  const double F[8], int N, int G, int tiles, cudaStream_t s)
{
    PhaseF f;
    for (int p = 0; p < 8; p++)
        f.f[p] = F[p];
    const int csize = min(kMaxCluster, (G + kWarps - 1) / kWarps);   // one group per warp where possible
    const int gpc = (G + csize - 1) / csize;
    const int cl = (G + gpc - 1) / gpc;

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
    if (cudaLaunchKernelEx(&cfg, lns8_stateset_kernel, masks, codes, xa, A, S, f, N, G, tiles, gpc) !=
        cudaSuccess)
        return TG_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace tgi
