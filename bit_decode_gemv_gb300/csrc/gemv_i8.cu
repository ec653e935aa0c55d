// gemv_i8.cu -- exact ternary GEMV with int8 activations and per-group integer
// scales (integer_engine.md §4.2 "BitNet b1.58 ternary" with §4.4 int8
// activations; the row is held as the W_nonzero / W_negative mask pair of the
// BitState brief §4):
//
//     y[m][r] = sum_g d[r][g] * P[m][r][g],   P = sum_{i in g} t[r][i] * x[m][i]
//
// P is an int32 (|P| <= 128 * 128), the sum over groups an int64; every sum is
// an integer sum, so the result does not depend on the launch geometry.
//
// Lane arithmetic. One 32-bit mask word holds 16 lanes: lane 4j + b of the word
// sits at bits 8b + 2j (nonzero) and 8b + 2j + 1 (negative). For a canonical
// pair the 2-bit field f is 0 (t = 0), 1 (t = +1) or 3 (t = -1), so f ^ 2 =
// t + 2. Masking column j of the word in place and flipping its high bit,
// (w & (0x03030303 << 2j)) ^ (0x02020202 << 2j), gives four unsigned bytes
// (t + 2) * 4^j, and one dp4a against the four activations of that column
// accumulates 4^j * sum (t + 2) x. Per group the four column sums are shifted
// back (exactly: each is a multiple of 4^j) and 2 * sum_{i in g} x is
// subtracted (the block-total reuse of integer_engine.md §4.1, computed once
// per group and shared by every row). Cost: one LOP3 and one dp4a per four
// weights, plus one broadcast 16-byte shared-memory load per sixteen.
//
// Binary Q1_0 weights (integer_engine.md §4.1) take the same path with one
// sign bit per weight (see group_pos_q1). Each group's scaled sum is floored
// by 2^frac on its own (§4.1/§4.2 arshift) before the sum over groups.
//
// This file holds the kernel for one to four tokens and the entry point, which
// picks the kernel for more (see kFewMaxTokens below).

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "device_common.cuh"
#include "tg.h"
#include "tg_internal.h"

TGI_DEFINE_DEVICE_ERROR(gemv_take_device_error)

namespace {

using tgi::dp4a_us;
using tgi::kTileRows;

// (w & mask) ^ flip in one LOP3 (truth table 0x6A = (a & b) ^ c).
__device__ __forceinline__ uint32_t and_xor(uint32_t w, uint32_t mask, uint32_t flip)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(w), "r"(mask), "r"(flip));
    return r;
}

// Column sums of one 128-lane group for one row: w[0..7] are the row's eight
// mask words (half 0 then half 1), xg the group's 128 activations in shared
// memory. Returns sum_i (t_i + 2) x_i.
__device__ __forceinline__ int group_dot_t2(const uint32_t w[8], const int8_t *xg)
{
    int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
    for (int u = 0; u < 8; u++) {
        const uint4 xv = *reinterpret_cast<const uint4 *>(xg + 16 * u);
        a0 = dp4a_us(and_xor(w[u], 0x03030303u, 0x02020202u), xv.x, a0);
        a1 = dp4a_us(and_xor(w[u], 0x0C0C0C0Cu, 0x08080808u), xv.y, a1);
        a2 = dp4a_us(and_xor(w[u], 0x30303030u, 0x20202020u), xv.z, a2);
        a3 = dp4a_us(and_xor(w[u], 0xC0C0C0C0u, 0x80808080u), xv.w, a3);
    }
    return a0 + (a1 >> 2) + (a2 >> 4) + (a3 >> 6);
}

// Q1_0 (integer_engine.md §4.1): sum of x over the +1 weights of one 128-lane
// group for one row. w[0..3] are the row's four words; word u holds lanes
// 32u + 4j + b in bit 8b + j. Masking bit j of every byte in place,
// w & (0x01010101 << j), gives four unsigned bytes 2^j * [weight is +1], and
// one dp4a against the four activations 32u + 4j .. 32u + 4j + 3 accumulates
// 2^j times their positive part; each column sum is shifted back exactly.
__device__ __forceinline__ int group_pos_q1(const uint32_t w[4], const int8_t *xg)
{
    int a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const uint4 lo = *reinterpret_cast<const uint4 *>(xg + 32 * u);
        const uint4 hi = *reinterpret_cast<const uint4 *>(xg + 32 * u + 16);
        const uint32_t xv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int j = 0; j < 8; j++)
            a[j] = dp4a_us(w[u] & (0x01010101u << j), xv[j], a[j]);
    }
    int pos = 0;
#pragma unroll
    for (int j = 0; j < 8; j++)
        pos += a[j] >> j;
    return pos;
}

// Several tokens (TB of them, their activations `stride` bytes apart in shared
// memory from xg). The masked words depend on the weights only, so each is
// formed once and fed to every token's dp4a. Ternary: out[t] = sum (t_i + 2) x_i.
template <int TB>
__device__ __forceinline__ void group_dot_t2_tokens(const uint32_t w[8], const int8_t *xg, int stride, int out[TB])
{
    int a[TB][4];
#pragma unroll
    for (int t = 0; t < TB; t++)
        a[t][0] = a[t][1] = a[t][2] = a[t][3] = 0;
#pragma unroll
    for (int u = 0; u < 8; u++) {
        const uint32_t c0 = and_xor(w[u], 0x03030303u, 0x02020202u);
        const uint32_t c1 = and_xor(w[u], 0x0C0C0C0Cu, 0x08080808u);
        const uint32_t c2 = and_xor(w[u], 0x30303030u, 0x20202020u);
        const uint32_t c3 = and_xor(w[u], 0xC0C0C0C0u, 0x80808080u);
#pragma unroll
        for (int t = 0; t < TB; t++) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(xg + t * stride + 16 * u);
            a[t][0] = dp4a_us(c0, xv.x, a[t][0]);
            a[t][1] = dp4a_us(c1, xv.y, a[t][1]);
            a[t][2] = dp4a_us(c2, xv.z, a[t][2]);
            a[t][3] = dp4a_us(c3, xv.w, a[t][3]);
        }
    }
#pragma unroll
    for (int t = 0; t < TB; t++)
        out[t] = a[t][0] + (a[t][1] >> 2) + (a[t][2] >> 4) + (a[t][3] >> 6);
}

// Q1_0 for several tokens: out[t] = sum of x over the +1 weights. Bit j of every
// byte is moved down to bit 0 ((w >> j) & 0x01010101), so all eight columns of
// a word accumulate into one sum per token without a shift back.
template <int TB>
__device__ __forceinline__ void group_pos_q1_tokens(const uint32_t w[4], const int8_t *xg, int stride, int out[TB])
{
    int a[TB][2];
#pragma unroll
    for (int t = 0; t < TB; t++)
        a[t][0] = a[t][1] = 0;
#pragma unroll
    for (int u = 0; u < 4; u++) {
        uint32_t c[8];
#pragma unroll
        for (int j = 0; j < 8; j++)
            c[j] = (w[u] >> j) & 0x01010101u;
#pragma unroll
        for (int t = 0; t < TB; t++) {
            const uint4 lo = *reinterpret_cast<const uint4 *>(xg + t * stride + 32 * u);
            const uint4 hi = *reinterpret_cast<const uint4 *>(xg + t * stride + 32 * u + 16);
            const uint32_t xv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int j = 0; j < 8; j++)
                a[t][j & 1] = dp4a_us(c[j], xv[j], a[t][j & 1]);
        }
    }
#pragma unroll
    for (int t = 0; t < TB; t++)
        out[t] = a[t][0] + a[t][1];
}

// A thread's int64 row sums of MT tokens: in registers up to four tokens; above
// that in the thread's own shared-memory slots (32 apart), where eight tokens'
// sums held in registers spilled (and sums in shared memory were slower at
// four tokens: 13824 x 5120 at M = 4, 11.1 -> 13.3 us).
template <int MT, bool kInSmem = (MT > 4)>
struct RowSums {
    int64_t v[MT];
    __device__ __forceinline__ void init(int64_t *)
    {
#pragma unroll
        for (int t = 0; t < MT; t++)
            v[t] = 0;
    }
    __device__ __forceinline__ void add(int t, int64_t a) { v[t] += a; }
    __device__ __forceinline__ void store(int64_t *slot)
    {
#pragma unroll
        for (int t = 0; t < MT; t++)
            slot[32 * t] = v[t];
    }
};

template <int MT>
struct RowSums<MT, true> {
    int64_t *p;
    __device__ __forceinline__ void init(int64_t *slot)
    {
        p = slot;
#pragma unroll
        for (int t = 0; t < MT; t++)
            p[32 * t] = 0;
    }
    __device__ __forceinline__ void add(int t, int64_t a) { p[32 * t] += a; }
    __device__ __forceinline__ void store(int64_t *) {}
};

// One group of one row for tokens T0..MT-1 in passes of up to four: P of each
// token from the masked words (formed once per pass), minus the block-total
// term, scaled by d, floored by 2^frac and added to the token's int64 sum.
// tsum_g[t * G] is token t's activation sum over the group.
template <int MT, int T0, bool kQ1>
__device__ __forceinline__ void tokens_pass(const uint4 &m0, const uint4 &m1, int32_t d, const int8_t *xg, int stride,
                                            const int *tsum_g, int G, int frac, RowSums<MT> &acc)
{
    constexpr int TB = MT - T0 < 4 ? MT - T0 : 4;
    int P[TB];
    if constexpr (kQ1) {
        const uint32_t w[4] = {m0.x, m0.y, m0.z, m0.w};
        group_pos_q1_tokens<TB>(w, xg + T0 * stride, stride, P);
#pragma unroll
        for (int t = 0; t < TB; t++)
            P[t] = 2 * P[t] - tsum_g[(T0 + t) * G];   // 2 * pos_sum - block_total
    } else {
        const uint32_t w[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        group_dot_t2_tokens<TB>(w, xg + T0 * stride, stride, P);
#pragma unroll
        for (int t = 0; t < TB; t++)
            P[t] -= 2 * tsum_g[(T0 + t) * G];
    }
#pragma unroll
    for (int t = 0; t < TB; t++)
        acc.add(T0 + t, ((int64_t)d * (int64_t)P[t]) >> frac);   // the group's floor (arithmetic shift)
    if constexpr (T0 + TB < MT)
        tokens_pass<MT, T0 + TB, kQ1>(m0, m1, d, xg, stride, tsum_g, G, frac, acc);
}

// Where a CTA, launched as a programmatic dependent, lets the next kernel on
// the stream launch: right after issuing its first weight loads, right after
// its wait for the previous kernel, or once its activations are staged.
constexpr int kTrigAfterLoads = 0, kTrigAfterWait = 1, kTrigAfterStage = 2;

// ---------------------------------------------------------------------------
// Batch 1 and a few tokens. One CTA per tile of 32 rows; lane l of every warp
// owns row 32T + l; the CTA's W warps split the row's groups (warp w takes
// g = w, w + W, ...; W = ceil(G / GPW), so each thread holds at most GPW
// groups), and the per-warp int64 partials are summed through shared memory at
// the end. Every weight load of the CTA is issued first, so a whole tile is in
// flight at once. Launched as a programmatic dependent (constant weights), the
// kernel issues its weight loads, lets the next kernel on the stream launch,
// and only then waits for the previous one and stages x: the next GEMV's weight
// stream starts while this one computes. (Measured on ffn_up: triggering right
// after the loads beats triggering at the start, which floods the memory
// system with several GEMVs' loads, and triggering after the compute, which
// leaves the memory idle between GEMVs.)
//
// MT tokens (1..kFewMaxTokens): the weights are read once; each thread keeps MT
// int64 row sums, and with MT > 1 a group's masked words are formed once per
// word and fed to every token (group_dot_t2_tokens), four tokens at a time,
// and each thread's per-token int64 sums live in its own shared-memory slots.
// ---------------------------------------------------------------------------
template <int GPW, bool kQ1, int MT>
__global__ void __launch_bounds__(GPW >= 4 ? 512 : 1024)
gemv_i8_m1_kernel(const uint4 *__restrict__ masks, const int32_t *__restrict__ scales,
                  const int8_t *__restrict__ x, int64_t *__restrict__ y, int N, int G, int frac, int trigger)
{
    constexpr int kChunks = kQ1 ? 32 : 64;   // uint4 per (tile, group): one or two per row
    extern __shared__ __align__(16) unsigned char smem[];
    const int K = G * 128;
    int8_t *xs = reinterpret_cast<int8_t *>(smem);                                        // [MT][K]
    int *tsum = reinterpret_cast<int *>(smem + MT * K);                                   // [MT][G]
    int64_t *red = reinterpret_cast<int64_t *>(smem + MT * K + ((MT * G * 4 + 15) & ~15));  // [W][MT][32]

    const int tile = blockIdx.x;
    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint4 *tmask = masks + (size_t)tile * G * kChunks;
    const int32_t *tscale = scales + (size_t)tile * G * kTileRows;

    uint4 m0[GPW], m1[GPW];
    int32_t dg[GPW];
    auto load_batch = [&](int g0) {
#pragma unroll
        for (int j = 0; j < GPW; j++) {
            const int g = g0 + j * nwarps;
            if (g < G) {
                m0[j] = tgi::ldg_stream(tmask + g * kChunks + lane);
                m1[j] = kQ1 ? make_uint4(0, 0, 0, 0) : tgi::ldg_stream(tmask + g * kChunks + 32 + lane);
                dg[j] = __ldg(tscale + g * kTileRows + lane);
            } else {
                m0[j] = m1[j] = make_uint4(0, 0, 0, 0);
                dg[j] = 0;
            }
        }
    };
    load_batch(warp);
    if (trigger == kTrigAfterLoads)
        tgi::pdl_launch_dependents();   // this CTA's first weights are in flight
    tgi::pdl_wait();
    if (trigger == kTrigAfterWait)
        tgi::pdl_launch_dependents();

    // Stage x and the per-group activation totals. With one group per warp each
    // warp stages only its own group's activations behind a warp barrier instead
    // of all of x behind a CTA barrier (measured on ffn_up: 2.19 -> 2.03 us per
    // call with constant weights, 2.95 -> 2.67 us without).
    if (GPW == 1) {
        // one group per warp (warp w owns group w): the warp stages its own
        // group's activations from the loads that also give the group's sum
        if (warp < G) {
            uint32_t v[MT];
#pragma unroll
            for (int t = 0; t < MT; t++)
                v[t] = __ldg(reinterpret_cast<const uint32_t *>(x + t * K + warp * 128) + lane);
#pragma unroll
            for (int t = 0; t < MT; t++) {
                reinterpret_cast<uint32_t *>(xs + t * K + warp * 128)[lane] = v[t];
                const int s = tgi::warp_sum_i32(tgi::byte_sum_s8(v[t]));
                if (lane == 0)
                    tsum[t * G + warp] = s;
            }
        }
        __syncwarp();
    } else {
        for (int i = threadIdx.x; i < MT * K / 16; i += blockDim.x)
            reinterpret_cast<uint4 *>(xs)[i] = __ldg(reinterpret_cast<const uint4 *>(x) + i);
        for (int tg = warp; tg < MT * G; tg += nwarps) {
            const uint32_t v = __ldg(reinterpret_cast<const uint32_t *>(x + tg * 128) + lane);
            const int s = tgi::warp_sum_i32(tgi::byte_sum_s8(v));
            if (lane == 0)
                tsum[tg] = s;
        }
        __syncthreads();
    }

    if (trigger == kTrigAfterStage)
        tgi::pdl_launch_dependents();
    // one token: the row sum in a register; several: RowSums (this thread's
    // slots of red, token t at [32 t], at the end or throughout)
    int64_t acc = 0;
    int64_t *const slot = red + warp * MT * 32 + lane;
    RowSums<MT> sums;
    if (MT > 1)
        sums.init(slot);
    for (int g0 = warp;;) {
#pragma unroll
        for (int j = 0; j < GPW; j++) {
            const int g = g0 + j * nwarps;
            if (g < G) {
                if constexpr (MT == 1) {
                    int P;
                    if (kQ1) {
                        // 2 * pos_sum - block_total
                        const uint32_t w[4] = {m0[j].x, m0[j].y, m0[j].z, m0[j].w};
                        P = 2 * group_pos_q1(w, xs + g * 128) - tsum[g];
                    } else {
                        const uint32_t w[8] = {m0[j].x, m0[j].y, m0[j].z, m0[j].w,
                                               m1[j].x, m1[j].y, m1[j].z, m1[j].w};
                        P = group_dot_t2(w, xs + g * 128) - 2 * tsum[g];
                    }
                    acc += ((int64_t)dg[j] * (int64_t)P) >> frac;   // the group's floor (arithmetic shift)
                } else {
                    tokens_pass<MT, 0, kQ1>(m0[j], m1[j], dg[j], xs + g * 128, K, tsum + g, G, frac, sums);
                }
            }
        }
        g0 += nwarps * GPW;
        if (g0 >= G)
            break;
        load_batch(g0);
    }

    if (MT == 1)
        red[warp * 32 + lane] = acc;
    else
        sums.store(slot);
    __syncthreads();
    const int row = tile * kTileRows + lane;
    for (int t = warp; t < MT; t += nwarps) {
        int64_t sum = 0;
        for (int w = 0; w < nwarps; w++)
            sum += red[(w * MT + t) * 32 + lane];
        if (row < N)
            y[(size_t)t * N + row] = sum;
    }
}

// ---------------------------------------------------------------------------
// Half-tile mapping of the same arithmetic. CTA c takes rows 16 (c & 1) ..
// 16 (c & 1) + 15 of tile c >> 1 for all groups; lane l owns row 16 (c & 1) +
// (l & 15), and its half of the warp, s = l >> 4, picks one group of a pair:
// warp w takes the pairs p = w, w + W, ... and half s group 2p + s. A warp
// instruction still covers 32 (row, group) lanes, but a CTA holds half as
// many, so twice as many CTAs spread the same work more evenly over the SMs
// (ffn_up: 432 CTAs of 10 warps, at most three per SM, instead of 216 of 20
// with 64 SMs holding two: at most 30 warp-groups of arithmetic per SM after
// the dependent-launch wait instead of 40). The two halves' sums of a row meet
// by one shuffle, the warps' through shared memory. Staged activations take
// kXStride bytes per group, so that the two groups a warp reads with one
// broadcast load sit in different banks.
// ---------------------------------------------------------------------------
constexpr int kXStride = 144;

template <int GPW, bool kQ1, int MT>
__device__ __forceinline__ void gemv_i8_half(const uint4 *__restrict__ masks, const int32_t *__restrict__ scales,
                                             const int8_t *__restrict__ x, int64_t *__restrict__ y, int N, int G,
                                             int frac, int trigger)
{
    constexpr int kChunks = kQ1 ? 32 : 64;   // uint4 per (tile, group): one or two per row
    extern __shared__ __align__(16) unsigned char smem[];
    const int K = G * 128;
    const int XS = G * kXStride;   // staged bytes per token
    int8_t *xs = reinterpret_cast<int8_t *>(smem);                                          // [MT][G][kXStride]
    int *tsum = reinterpret_cast<int *>(smem + MT * XS);                                    // [MT][G]
    int64_t *red = reinterpret_cast<int64_t *>(smem + MT * XS + ((MT * G * 4 + 15) & ~15));  // [W][MT][32]

    const int tile = blockIdx.x >> 1;
    const int half = (blockIdx.x & 1) * 16;
    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int side = lane >> 4, r16 = lane & 15;
    const uint4 *tmask = masks + (size_t)tile * G * kChunks + half + r16;
    const int32_t *tscale = scales + (size_t)tile * G * kTileRows + half + r16;

    uint4 m0[GPW], m1[GPW];
    int32_t dg[GPW];
    auto load_batch = [&](int p0) {
#pragma unroll
        for (int j = 0; j < GPW; j++) {
            const int g = 2 * (p0 + j * nwarps) + side;
            if (g < G) {
                m0[j] = tgi::ldg_stream(tmask + g * kChunks);
                m1[j] = kQ1 ? make_uint4(0, 0, 0, 0) : tgi::ldg_stream(tmask + g * kChunks + 32);
                dg[j] = __ldg(tscale + g * kTileRows);
            } else {
                m0[j] = m1[j] = make_uint4(0, 0, 0, 0);
                dg[j] = 0;
            }
        }
    };
    load_batch(warp);
    if (trigger == kTrigAfterLoads)
        tgi::pdl_launch_dependents();   // this CTA's first weights are in flight
    tgi::pdl_wait();
    if (trigger == kTrigAfterWait)
        tgi::pdl_launch_dependents();

    if (GPW == 1) {
        // warp w owns pair w: each half stages its group's 128 activations (8 bytes
        // a lane) and their sum, behind a warp barrier only
        const int g = 2 * warp + side;
        uint2 v[MT];
#pragma unroll
        for (int t = 0; t < MT; t++)
            v[t] = g < G ? __ldg(reinterpret_cast<const uint2 *>(x + t * K + g * 128) + r16) : make_uint2(0, 0);
#pragma unroll
        for (int t = 0; t < MT; t++) {
            int s = tgi::byte_sum_s8(v[t].x) + tgi::byte_sum_s8(v[t].y);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                s += __shfl_xor_sync(0xffffffffu, s, o);   // within the half
            if (g < G) {
                reinterpret_cast<uint2 *>(xs + t * XS + g * kXStride)[r16] = v[t];
                if (r16 == 0)
                    tsum[t * G + g] = s;
            }
        }
        __syncwarp();
    } else {
        for (int i = threadIdx.x; i < MT * G * 8; i += blockDim.x) {
            const int tg = i >> 3, c = i & 7;   // (token, group) tg = t * G + g, 16-byte chunk c
            reinterpret_cast<uint4 *>(xs + (tg / G) * XS + (tg % G) * kXStride)[c] =
                __ldg(reinterpret_cast<const uint4 *>(x + tg * 128) + c);
        }
        for (int tg = warp; tg < MT * G; tg += nwarps) {
            const uint32_t v = __ldg(reinterpret_cast<const uint32_t *>(x + tg * 128) + lane);
            const int s = tgi::warp_sum_i32(tgi::byte_sum_s8(v));
            if (lane == 0)
                tsum[tg] = s;
        }
        __syncthreads();
    }

    if (trigger == kTrigAfterStage)
        tgi::pdl_launch_dependents();
    // one token: the row sum in a register; several: RowSums (this thread's
    // slots of red, [W][MT][32]: both halves of the warp, summed at the end)
    int64_t acc = 0;
    int64_t *const slot = red + warp * MT * 32 + lane;
    RowSums<MT> sums;
    if (MT > 1)
        sums.init(slot);
    for (int p0 = warp;;) {
#pragma unroll
        for (int j = 0; j < GPW; j++) {
            const int g = 2 * (p0 + j * nwarps) + side;
            if (g < G) {
                const int8_t *xg = xs + g * kXStride;
                if constexpr (MT == 1) {
                    int P;
                    if (kQ1) {
                        const uint32_t w[4] = {m0[j].x, m0[j].y, m0[j].z, m0[j].w};
                        P = 2 * group_pos_q1(w, xg) - tsum[g];
                    } else {
                        const uint32_t w[8] = {m0[j].x, m0[j].y, m0[j].z, m0[j].w,
                                               m1[j].x, m1[j].y, m1[j].z, m1[j].w};
                        P = group_dot_t2(w, xg) - 2 * tsum[g];
                    }
                    acc += ((int64_t)dg[j] * (int64_t)P) >> frac;   // the group's floor (arithmetic shift)
                } else {
                    tokens_pass<MT, 0, kQ1>(m0[j], m1[j], dg[j], xg, XS, tsum + g, G, frac, sums);
                }
            }
        }
        p0 += nwarps * GPW;
        if (2 * p0 >= G)
            break;
        load_batch(p0);
    }

    // the two halves' sums of each row, then the warps'
    if (MT == 1) {
        acc += __shfl_xor_sync(0xffffffffu, acc, 16);
        if (side == 0)
            red[warp * 32 + r16] = acc;
    } else {
        sums.store(slot);
    }
    __syncthreads();
    const int row = tile * kTileRows + half + r16;
    if (lane < 16)
        for (int t = warp; t < MT; t += nwarps) {
            int64_t sum = 0;
            for (int w = 0; w < nwarps; w++)
                sum += MT == 1 ? red[w * 32 + r16] : red[(w * MT + t) * 32 + r16] + red[(w * MT + t) * 32 + 16 + r16];
            if (row < N)
                y[(size_t)t * N + row] = sum;
        }
}

template <int GPW, bool kQ1, int MT>
__global__ void __launch_bounds__(GPW >= 4 ? 512 : 1024)
gemv_i8_half_kernel(const uint4 *__restrict__ masks, const int32_t *__restrict__ scales,
                    const int8_t *__restrict__ x, int64_t *__restrict__ y, int N, int G, int frac, int trigger)
{
    gemv_i8_half<GPW, kQ1, MT>(masks, scales, x, y, N, G, frac, trigger);
}

// One token, one pair per warp: held to 32 registers a thread (two resident
// 1024-thread CTAs), so that an SM holds its three CTAs of one call and three
// of the next, launched as a programmatic dependent, at once (without the
// minimum the compiler took 50).
template <bool kQ1>
__global__ void __launch_bounds__(1024, 2)
gemv_i8_half1_kernel(const uint4 *__restrict__ masks, const int32_t *__restrict__ scales,
                     const int8_t *__restrict__ x, int64_t *__restrict__ y, int N, int G, int frac, int trigger)
{
    gemv_i8_half<1, kQ1, 1>(masks, scales, x, y, N, G, frac, trigger);
}

// ---------------------------------------------------------------------------
// One token of int64 fixed-point activations (integer engine §4.4; exact
// modulo 2^64, §5) on the whole-tile mapping. Each x is split into signed
// base-256 digits s_0..s_7 in [-128, 127] with x = sum_l 256^l s_l (mod 2^64)
// -- the bytes of (x + 0x8080...80) XOR 0x8080...80 -- and every digit plane is
// an int8 activation vector for the lane arithmetic above, four planes to a
// pass over the group's masked words (as four tokens). Per group the planes'
// P_l are recombined as sum_l P_l 2^(8l) in wrapping 64-bit arithmetic,
// multiplied by d, floored and summed, all modulo 2^64. A warp stages exactly
// the groups it computes, and only as many planes as the group's largest
// digit needs, rounded up to a pass (a group of zeros takes none): four for
// magnitudes below 2^31, eight beyond. Planes above a value's top digit are
// zero bytes, so staging a whole pass changes nothing.
// ---------------------------------------------------------------------------
template <int GPW, bool kQ1>
__global__ void __launch_bounds__(GPW >= 4 ? 512 : 1024)
gemv_x64_m1_kernel(const uint4 *__restrict__ masks, const int32_t *__restrict__ scales,
                   const int8_t *__restrict__ xv, int64_t *__restrict__ y, int N, int G, int frac, int trigger)
{
    constexpr int kChunks = kQ1 ? 32 : 64;
    extern __shared__ __align__(16) unsigned char smem[];
    const int K = G * 128;
    int8_t *xs = reinterpret_cast<int8_t *>(smem);                         // [8 planes][K]
    int *tsum = reinterpret_cast<int *>(smem + 8 * K);                     // [8][G]
    int *npl = tsum + 8 * G;                                               // [G] planes staged (0, 4 or 8)
    uint64_t *red = reinterpret_cast<uint64_t *>(smem + 8 * K + ((9 * G * 4 + 15) & ~15));   // [W][32]
    const uint64_t *x = reinterpret_cast<const uint64_t *>(xv);

    const int tile = blockIdx.x;
    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint4 *tmask = masks + (size_t)tile * G * kChunks;
    const int32_t *tscale = scales + (size_t)tile * G * kTileRows;

    uint4 m0[GPW], m1[GPW];
    int32_t dg[GPW];
    auto load_batch = [&](int g0) {
#pragma unroll
        for (int j = 0; j < GPW; j++) {
            const int g = g0 + j * nwarps;
            if (g < G) {
                m0[j] = tgi::ldg_stream(tmask + g * kChunks + lane);
                m1[j] = kQ1 ? make_uint4(0, 0, 0, 0) : tgi::ldg_stream(tmask + g * kChunks + 32 + lane);
                dg[j] = __ldg(tscale + g * kTileRows + lane);
            } else {
                m0[j] = m1[j] = make_uint4(0, 0, 0, 0);
                dg[j] = 0;
            }
        }
    };
    load_batch(warp);
    if (trigger == kTrigAfterLoads)
        tgi::pdl_launch_dependents();
    tgi::pdl_wait();
    if (trigger == kTrigAfterWait)
        tgi::pdl_launch_dependents();

    // the digit planes of this warp's groups (the groups it computes below):
    // lane l holds values 4l .. 4l + 3 of the group
    for (int g = warp; g < G; g += nwarps) {
        const ulonglong2 *src = reinterpret_cast<const ulonglong2 *>(x + (size_t)g * 128 + 4 * lane);
        const ulonglong2 v01 = __ldg(src), v23 = __ldg(src + 1);
        const uint64_t dv[4] = {(v01.x + 0x8080808080808080ull) ^ 0x8080808080808080ull,
                                (v01.y + 0x8080808080808080ull) ^ 0x8080808080808080ull,
                                (v23.x + 0x8080808080808080ull) ^ 0x8080808080808080ull,
                                (v23.y + 0x8080808080808080ull) ^ 0x8080808080808080ull};
        int top = -1;   // highest nonzero digit of the lane's values
#pragma unroll
        for (int b = 0; b < 4; b++)
            if (dv[b])
                top = max(top, (63 - __clzll((long long)dv[b])) >> 3);
        top = __reduce_max_sync(0xffffffffu, top);
        const int np = top < 0 ? 0 : top < 4 ? 4 : 8;
        for (int l = 0; l < np; l++) {
            const uint32_t word = (uint32_t)((dv[0] >> (8 * l)) & 0xFF) | ((uint32_t)((dv[1] >> (8 * l)) & 0xFF) << 8) |
                                  ((uint32_t)((dv[2] >> (8 * l)) & 0xFF) << 16) |
                                  ((uint32_t)((dv[3] >> (8 * l)) & 0xFF) << 24);
            reinterpret_cast<uint32_t *>(xs + (size_t)l * K + g * 128)[lane] = word;
            const int sum = tgi::warp_sum_i32(tgi::byte_sum_s8(word));
            if (lane == 0)
                tsum[l * G + g] = sum;
        }
        if (lane == 0)
            npl[g] = np;
    }
    __syncwarp();
    if (trigger == kTrigAfterStage)
        tgi::pdl_launch_dependents();

    uint64_t acc = 0;   // wrapping
    for (int g0 = warp;;) {
#pragma unroll
        for (int j = 0; j < GPW; j++) {
            const int g = g0 + j * nwarps;
            if (g < G && npl[g] > 0) {
                // sum_l P_l 2^(8l), one pass of four planes at a time, then times
                // d and floored: all modulo 2^64
                const int passes = npl[g] > 4 ? 2 : 1;
                uint64_t p64 = 0;
#pragma unroll 1
                for (int h = 0; h < passes; h++) {   // planes 4h .. 4h + 3
                    const int8_t *xg = xs + (size_t)(4 * h) * K + g * 128;
                    int P[4];
                    if (kQ1) {
                        const uint32_t w[4] = {m0[j].x, m0[j].y, m0[j].z, m0[j].w};
                        group_pos_q1_tokens<4>(w, xg, K, P);
#pragma unroll
                        for (int l = 0; l < 4; l++)
                            P[l] = 2 * P[l] - tsum[(4 * h + l) * G + g];
                    } else {
                        const uint32_t w[8] = {m0[j].x, m0[j].y, m0[j].z, m0[j].w,
                                               m1[j].x, m1[j].y, m1[j].z, m1[j].w};
                        group_dot_t2_tokens<4>(w, xg, K, P);
#pragma unroll
                        for (int l = 0; l < 4; l++)
                            P[l] -= 2 * tsum[(4 * h + l) * G + g];
                    }
#pragma unroll
                    for (int l = 0; l < 4; l++)
                        p64 += (uint64_t)(int64_t)P[l] << (32 * h + 8 * l);
                }
                const int64_t v = (int64_t)(p64 * (uint64_t)(int64_t)dg[j]);
                acc += (uint64_t)(v >> frac);
            }
        }
        g0 += nwarps * GPW;
        if (g0 >= G)
            break;
        load_batch(g0);
    }

    red[warp * 32 + lane] = acc;
    __syncthreads();
    if (warp == 0) {
        uint64_t sum = 0;
        for (int w = 0; w < nwarps; w++)
            sum += red[w * 32 + lane];
        const int row = tile * kTileRows + lane;
        if (row < N)
            y[row] = (int64_t)sum;
    }
}

// Kernel per token count: M = 1..kFewMaxTokens the two kernels above (the
// mapping, trigger position and resident-CTA cap from few_plan); then the
// warp-MMA kernel (gemv_i8_hmma.cu) for one token tile, or two when K is at
// most kHmmaTwoTileMaxK; above that the tensor-memory kernel (gemv_i8_mma.cu),
// whose cost hardly grows with M up to 64. The CUDA-core dp4a kernel
// (gemv_i8_mt.cu) takes int64 activations at every M, and int8 ones at
// 2..kDp4aMaxTokens when the activations do not fit the shared memory of the
// kernels above (it stages the tokens in chunks).
constexpr int kFewMaxTokens = 8;
constexpr int kDp4aMaxTokens = 4;
constexpr int kHmmaMaxTokens = 16;
constexpr int kHmmaTwoTileMaxK = 4096;
constexpr size_t kM1SmemMax = 200 * 1024;

size_t m1_smem_bytes(int G, int warps, int MT)
{
    return (size_t)MT * G * 128 + (((size_t)MT * G * 4 + 15) & ~(size_t)15) + (size_t)warps * MT * 32 * 8;
}

size_t half_smem_bytes(int G, int warps, int MT)
{
    return (size_t)MT * G * kXStride + (((size_t)MT * G * 4 + 15) & ~(size_t)15) + (size_t)warps * MT * 32 * 8;
}

// The launch of one of the kernels above: grid, warps, dynamic shared memory
// (at least min_smem: a larger reservation caps the CTAs resident on an SM),
// programmatic dependent launch when the weights are constant. A kernel's
// dynamic shared-memory limit is raised to the device's opt-in maximum on its
// first launch there (attr_set: one bit per device), not on every call.
using FewKernel = void (*)(const uint4 *, const int32_t *, const int8_t *, int64_t *, int, int, int, int);

cudaError_t launch_one(FewKernel kern, std::atomic<uint64_t> &attr_set, int smem_optin, int grid, int warps,
                       size_t smem, size_t min_smem, const uint4 *masks, const int32_t *scales, const int8_t *x,
                       int64_t *y, int N, int G, int frac, int trigger, bool pdl, cudaStream_t s)
{
    if (smem < min_smem)
        smem = min_smem;
    if (smem > 48 * 1024) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess)
            return cudaErrorInvalidDevice;
        const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;   // (devices past 64: set every call)
        if (!(attr_set.load(std::memory_order_acquire) & bit)) {
            const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
            if (e != cudaSuccess)
                return e;
            attr_set.fetch_or(bit, std::memory_order_acq_rel);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(warps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, masks, scales, x, y, N, G, frac, trigger);
}

struct FewLaunch {
    int smem_optin;   // the device's opt-in shared memory per CTA
    const uint4 *masks;
    const int32_t *scales;
    const int8_t *x;
    int64_t *y;
    int N, G, tiles, frac, trigger;
    size_t min_smem;
    bool pdl;
    cudaStream_t s;
};

template <int GPW, bool kQ1, int MT>
cudaError_t launch_whole(const FewLaunch &l)
{
    const int max_warps = GPW >= 4 ? 16 : 32;
    const int warps = min((l.G + GPW - 1) / GPW, max_warps);
    static std::atomic<uint64_t> attr_set{0};
    return launch_one(gemv_i8_m1_kernel<GPW, kQ1, MT>, attr_set, l.smem_optin, l.tiles, warps,
                      m1_smem_bytes(l.G, warps, MT), l.min_smem, l.masks, l.scales, l.x, l.y, l.N, l.G, l.frac,
                      l.trigger, l.pdl, l.s);
}

template <int GPW, bool kQ1, int MT>
cudaError_t launch_half(const FewLaunch &l)
{
    FewKernel kern;
    if constexpr (GPW == 1 && MT == 1)
        kern = gemv_i8_half1_kernel<kQ1>;
    else
        kern = gemv_i8_half_kernel<GPW, kQ1, MT>;
    const int max_warps = GPW >= 4 ? 16 : 32;
    const int warps = min(((l.G + 1) / 2 + GPW - 1) / GPW, max_warps);
    static std::atomic<uint64_t> attr_set{0};
    return launch_one(kern, attr_set, l.smem_optin, 2 * l.tiles, warps, half_smem_bytes(l.G, warps, MT), l.min_smem,
                      l.masks, l.scales, l.x, l.y, l.N, l.G, l.frac, l.trigger, l.pdl, l.s);
}

size_t x64_smem_bytes(int G, int warps)
{
    return (size_t)8 * G * 128 + (((size_t)9 * G * 4 + 15) & ~(size_t)15) + (size_t)warps * 32 * 8;
}

template <int GPW, bool kQ1>
cudaError_t launch_x64(const FewLaunch &l)
{
    const int max_warps = GPW >= 4 ? 16 : 32;
    const int warps = min((l.G + GPW - 1) / GPW, max_warps);
    static std::atomic<uint64_t> attr_set{0};
    return launch_one(gemv_x64_m1_kernel<GPW, kQ1>, attr_set, l.smem_optin, l.tiles, warps,
                      x64_smem_bytes(l.G, warps), l.min_smem, l.masks, l.scales, l.x, l.y, l.N, l.G, l.frac,
                      l.trigger, l.pdl, l.s);
}

template <bool kQ1>
cudaError_t launch_x64_m1(const FewLaunch &l)
{
    if (l.G <= 32)
        return launch_x64<1, kQ1>(l);
    if (l.G <= 64)
        return launch_x64<2, kQ1>(l);
    return launch_x64<4, kQ1>(l);
}

// Groups per warp. Whole tiles, one token: one group per warp up to K = 4096
// (32 warps), then two up to K = 8192; several tokens: two up to K = 8192
// (measured faster than one on ffn_up at M = 3, 4 and on 13824 x 5120); beyond
// that 16 warps loop over batches of four. Half tiles (a warp covers a pair of
// groups): one pair per warp up to K = 8192, two up to K = 16384, then four.
template <int MT, bool kQ1>
cudaError_t launch_tokens(bool half, const FewLaunch &l)
{
    if (half) {
        if (l.G <= 64)
            return launch_half<1, kQ1, MT>(l);
        if (l.G <= 128)
            return launch_half<2, kQ1, MT>(l);
        return launch_half<4, kQ1, MT>(l);
    }
    if constexpr (MT == 1) {
        if (l.G <= 32)
            return launch_whole<1, kQ1, 1>(l);
    }
    if (l.G <= 64)
        return launch_whole<2, kQ1, MT>(l);
    return launch_whole<4, kQ1, MT>(l);
}

template <bool kQ1>
cudaError_t launch_few(int M, bool half, const FewLaunch &l)
{
    static_assert(kFewMaxTokens == 8, "one instance per token count");
    switch (M) {
    case 1: return launch_tokens<1, kQ1>(half, l);
    case 2: return launch_tokens<2, kQ1>(half, l);
    case 3: return launch_tokens<3, kQ1>(half, l);
    case 4: return launch_tokens<4, kQ1>(half, l);
    case 5: return launch_tokens<5, kQ1>(half, l);
    case 6: return launch_tokens<6, kQ1>(half, l);
    case 7: return launch_tokens<7, kQ1>(half, l);
    default: return launch_tokens<8, kQ1>(half, l);
    }
}

// The device's SM count and shared memory per SM (and per CTA reserved by the
// system), looked up once per device.
struct DeviceShape {
    int nsm, smem_sm, smem_reserved, smem_optin;
};

bool device_shape(DeviceShape &d)
{
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cache[kMaxDevices][4];
    static std::atomic<bool> have[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    if (dev >= 0 && dev < kMaxDevices && have[dev].load(std::memory_order_acquire)) {
        d = {cache[dev][0].load(std::memory_order_relaxed), cache[dev][1].load(std::memory_order_relaxed),
             cache[dev][2].load(std::memory_order_relaxed), cache[dev][3].load(std::memory_order_relaxed)};
        return true;
    }
    if (cudaDeviceGetAttribute(&d.nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return false;
    if (dev >= 0 && dev < kMaxDevices) {
        cache[dev][0].store(d.nsm, std::memory_order_relaxed);
        cache[dev][1].store(d.smem_sm, std::memory_order_relaxed);
        cache[dev][2].store(d.smem_reserved, std::memory_order_relaxed);
        cache[dev][3].store(d.smem_optin, std::memory_order_relaxed);
        have[dev].store(true, std::memory_order_release);
    }
    return true;
}

// Launch plan of the one-to-four-token kernels: whole or half tiles, where a
// CTA lets the next call launch, and at most how many CTAs an SM holds (0 = no
// cap). Chosen from a sweep of per-call times with constant weights, back to
// back (N x K = 2560 x 2560, 2560 x 6912, 6912 x 2560, 5120 x 5120,
// 13824 x 5120, 32000 x 2560; M = 1..4), where each rule below was within a
// few percent of the fastest of 2 mappings x 3 trigger positions x 5 caps:
//   - one token, one group per warp (K <= 4096): whole tiles, next call
//     launched after the wait; when a call has at most two tiles per SM, at
//     most two CTAs per SM (ffn_up 2.13 -> 1.80 us, 2560 x 2560 1.85 -> 1.46):
//     fewer calls then prefetch weights at once, which otherwise delays the
//     running call's activation reads, output writes and completion (one
//     group per warp beat two on every one-token shape measured);
//   - one token, longer rows: half tiles (5120 x 5120 3.77 -> 2.68 us,
//     13824 x 5120 6.38 -> 5.03);
//   - several tokens: half tiles when K <= 4096 and a call has at most two
//     tiles per SM, the next call launched after the wait; else whole tiles,
//     the next call launched once the activations are staged (13824 x 5120 at
//     M = 4: 12.1 -> 11.1 us, 2560 x 2560 at M = 4: 4.7 -> 2.6). Checked on seven
//     more shapes (4096 x 1024, 4096 x 2048, 1024 x 4096, 2048 x 3072,
//     11008 x 4096, 4096 x 11008, 8192 x 8192): for half tiles the release
//     after the wait was as fast as after staging at M = 5..8 and up to 25 %
//     faster at M = 2..4 (4096 x 2048 at M = 4: 3.23 -> 2.44 us).
struct FewPlan {
    bool half;
    int trigger;
    int cap;
};

FewPlan few_plan(int M, int G, int tiles, int nsm)
{
    const bool few_tiles = tiles <= 2 * nsm;
    if (M == 1) {
        if (G <= 32) {
            // whole tiles of G warps: threads alone hold an SM to 64 / G CTAs;
            // where that is three or fewer, reserving shared memory for exactly
            // that many (no fewer CTAs, a larger shared-memory carveout) was
            // faster too (32000 x 2560: 5.76 -> 5.55 us)
            const int by_threads = 64 / G;
            return {false, kTrigAfterWait, few_tiles ? 2 : by_threads <= 3 ? by_threads : 0};
        }
        return {true, kTrigAfterLoads, 0};
    }
    if (G <= 32 && few_tiles)
        return {true, kTrigAfterWait, 0};
    return {false, kTrigAfterStage, 0};
}

// Whether M tokens go to the few-token kernels rather than the warp-MMA one:
// up to six always (per call on 2560 x 2560 / 6912 x 2560 / 13824 x 5120 /
// 32000 x 2560 at M = 5: 3.37 / 4.46 / 14.0 / 14.5 us against 6.02 / 6.22 /
// 18.0 / 20.8); seven or eight where a call has at most one tile per SM, or
// K <= 4096 and at most two (at M = 8: 2560 x 6912 9.4 against 13.5 us, 6912 x
// 2560 6.2 against 6.3; with more tiles the warp-MMA kernel was faster:
// 5120 x 5120 10.9 against 13.9, 13824 x 5120 18.4 against 21.3).
bool few_takes(int M, int G, int tiles, int nsm)
{
    if (M > kFewMaxTokens)
        return false;
    if (M <= 6)
        return true;
    return tiles <= nsm || (G <= 32 && tiles <= 2 * nsm);
}

// Dynamic shared memory that holds an SM to `cap` resident CTAs: the smallest
// reservation above a (cap + 1)-th share of the SM's shared memory, plus a
// third of the range that still fits cap of them (measured: on ffn_up at one
// token 89.8 KB, in the range 76.8..115.7 KB, gave 1.79 us and 104 KB 1.86).
size_t cap_smem(const DeviceShape &d, int cap)
{
    if (cap <= 0)
        return 0;
    const size_t lo = (size_t)d.smem_sm / (cap + 1) - d.smem_reserved + 1;   // cap + 1 no longer fit
    const size_t hi = (size_t)d.smem_sm / cap - d.smem_reserved;             // cap still fit
    return lo + (hi - lo) / 3;
}

}  // namespace

extern "C" int tg_gemv_i8(const tg_layout *L, const void *w, const int8_t *x, int64_t M,
                          int64_t *y, void *stream)
{
    if (!L || !w || !x || !y)
        return TG_ERR_ARG;
    if ((L->kind != TG_TERNARY_I8 && L->kind != TG_BINARY_Q1) || L->version != 1)
        return TG_ERR_ARG;
    if (L->frac < 0 || L->frac > 62 || L->wait_limit < 0)
        return TG_ERR_ARG;
    if (!tgi::aligned(w, 256) || !tgi::aligned(x, 16) || !tgi::aligned(y, 8))
        return TG_ERR_ARG;
    if (L->N < 1 || L->K < TG_GROUP || L->K % TG_GROUP || M < 1 || M > TG_MAX_M)
        return TG_ERR_SHAPE;
    const bool x64 = (L->flags & TG_FLAG_X_INT64) != 0;
    // int8 activations: |y| <= G * 128 * 128 * max|d| must stay well inside
    // int64 (int64 activations wrap modulo 2^64 by definition).
    if (!x64 && (double)L->G * 16384.0 * (double)L->max_abs_scale >= 4.0e18)
        return TG_ERR_BOUND;

    const auto *base = static_cast<const unsigned char *>(w);
    const uint4 *masks = reinterpret_cast<const uint4 *>(base + L->mask_off);
    const int32_t *scales = reinterpret_cast<const int32_t *>(base + L->scale_off);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int G = (int)L->G, N = (int)L->N;
    const int tiles = (int)L->tiles;

    const bool pdl = (L->flags & TG_FLAG_CONST_WEIGHTS) != 0;
    const bool q1 = L->kind == TG_BINARY_Q1;
    // shapes no kernel takes are refused before any device query or launch
    DeviceShape d;
    if (x64) {
        // int64 activations: one token on the whole-tile digit-plane kernel
        // (launched like the one-token int8 plan for K <= 4096), else the
        // chunked dp4a kernel for every M (which refuses what it cannot stage)
        if (M == 1 && x64_smem_bytes(G, 32) <= kM1SmemMax) {
            if (!device_shape(d))
                return TG_ERR_CUDA;
            const bool few_tiles = tiles <= 2 * d.nsm;
            const FewLaunch l = {d.smem_optin, masks, scales, x, y, N, G, tiles, (int)L->frac, kTrigAfterWait,
                                 cap_smem(d, G <= 32 && few_tiles ? 2 : 0), pdl, s};
            const cudaError_t e = q1 ? launch_x64_m1<true>(l) : launch_x64_m1<false>(l);
            return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
        }
        return tgi::gemv_i8_mt(masks, scales, x, y, N, G, tiles, (int)M, q1, true, (int)L->frac, pdl, s);
    }

    const bool few_fit = M <= kFewMaxTokens && m1_smem_bytes(G, 32, (int)M) <= kM1SmemMax;
    if (M == 1 && !few_fit)
        return TG_ERR_SHAPE;
    if (few_fit) {
        if (!device_shape(d))
            return TG_ERR_CUDA;
        if (few_takes((int)M, G, tiles, d.nsm)) {
            FewPlan plan = few_plan((int)M, G, tiles, d.nsm);
            if (plan.half && half_smem_bytes(G, 32, (int)M) > kM1SmemMax)
                plan = {false, kTrigAfterLoads, 0};
            const FewLaunch l = {d.smem_optin, masks, scales, x, y, N, G, tiles, (int)L->frac, plan.trigger,
                                 cap_smem(d, plan.cap), pdl, s};
            const cudaError_t e =
                q1 ? launch_few<true>((int)M, plan.half, l) : launch_few<false>((int)M, plan.half, l);
            return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
        }
    }
    if (M <= kDp4aMaxTokens)
        return tgi::gemv_i8_mt(masks, scales, x, y, N, G, tiles, (int)M, q1, false, (int)L->frac, pdl, s);
    if ((M <= 8 || (M <= kHmmaMaxTokens && L->K <= kHmmaTwoTileMaxK)) && tgi::gemv_i8_hmma_fits(G))
        return tgi::gemv_i8_hmma(masks, scales, x, y, N, G, tiles, (int)M, q1, (int)L->frac, pdl, s);
    return tgi::gemv_i8_mma(masks, scales, x, y, N, G, tiles, (int)M, L->max_abs_scale, q1, (int)L->frac,
                            L->wait_limit, s);
}
