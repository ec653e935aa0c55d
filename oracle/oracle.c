/*
 * oracle.c -- plain, slow CPU reference for the exact ternary weight apply.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the bench's CPU
 * baseline leg are the only callers. The CUDA path never includes, links or
 * loads this file, and this file shares no code, header, table or constant
 * with it. Inputs come from the seeded generators; nothing here is computed
 * from a GPU result.
 *
 * Every function is the plain definition, written as naive loops in int64 (and
 * fp64 / long double where a real number is materialised). Sources, by page:
 *
 *   [BitState]  "BitState / HSDR PoC Technical Brief v0.5"
 *               (huggingface.co/datasets/mktnhr/BitState)
 *   [SKaiNET]   SKaiNET-transformers issue #337, "[bitnet] T2: lm_head via
 *               BITNET_PLANES weight format (WeightForm) + two-stage top-k decode"
 *   [IntEngine] integer_engine.md, "A standalone deterministic integer inference
 *               engine for BitNet-style LLMs, with Ollama interop"
 *
 * Readings taken where the pages leave a step open (each is listed with its
 * reason in the design notes):
 *   - per-group arshift(., frac) of [IntEngine] §4.1/§4.2 is floor division by
 *     2^frac of each group's scaled sum; the main apply functions take frac = 0
 *     and the *_frac functions take it as an argument;
 *   - K must be a multiple of 128 (the group size); other K is rejected;
 *   - LNS8 product code k = a + d - 74: k <= 0 is exact zero, k > 127 saturates
 *     to 127; an activation with code 0 is zero whatever its sign bit;
 *   - lm_head plane p carries the integer weight 3^(7-p) (the pages' 3^-p
 *     scaled by 3^7), so the planes 4..7 truncation bound is 40 = 27+9+3+1;
 *   - top-k order is (score descending, row index ascending), which makes the
 *     argmax the lowest index among equal maxima.
 *
 * All functions return 0 on success and -1 on an invalid argument.
 */

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_GROUP 128

/* Population count of a 64-bit word by clearing the lowest set bit. */
static int oracle_popcount64(uint64_t v)
{
    int n = 0;
    while (v) {
        v &= v - 1;
        n++;
    }
    return n;
}

/* ------------------------------------------------------------------------- */
/* 1. Ternary GEMV with int8 activations and per-group integer scales.       */
/* ------------------------------------------------------------------------- */

/*
 * y[m][r] = sum_g d[r][g] * ( sum_{i in group g} t[r][i] * x[m][i] )
 *
 * [IntEngine] §4.2 (BitNet b1.58 ternary): the per-group signed sum is the sum
 * of x over the +1 weights minus the sum over the -1 weights (zeros drop out);
 * it is multiplied by the per-group integer scale and summed over groups
 * (§4.1/§4.2 "out_o", frac = 0). §4.4 fixes int8 activations with integer
 * accumulation. Layouts: t [N][K] int8 in {-1,0,1}; d [N][K/128] int32;
 * x [M][K] int8; y [M][N] int64.
 */
int oracle_gemv_i8(int64_t M, int64_t N, int64_t K, const int8_t *t,
                   const int32_t *d, const int8_t *x, int64_t *y)
{
    if (M < 1 || N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t r = 0; r < N; r++) {
            int64_t out = 0;
            for (int64_t g = 0; g < G; g++) {
                int64_t signed_sum = 0;
                for (int64_t i = g * ORACLE_GROUP; i < (g + 1) * ORACLE_GROUP; i++)
                    signed_sum += (int64_t)t[r * K + i] * (int64_t)x[m * K + i];
                out += (int64_t)d[r * G + g] * signed_sum;
            }
            y[m * N + r] = out;
        }
    }
    return 0;
}

/*
 * arshift(v, s) of [IntEngine] §4.1: an arithmetic right shift, i.e. floor
 * division by 2^s (rounding toward minus infinity), written with C's
 * truncating division so that it does not rest on how the compiler shifts a
 * negative number. 0 <= s <= 62.
 */
static int64_t oracle_arshift(int64_t v, int s)
{
    const int64_t p = (int64_t)1 << s;
    int64_t q = v / p;
    if (v % p != 0 && v < 0)
        q -= 1;
    return q;
}

/*
 * [IntEngine] §4.2 with the per-group floor: for every output o
 *   out_o = sum_b arshift( signed_sum_b * scale[o][b], frac ),
 *   signed_sum_b = (sum over the +1 weights of x) - (sum over the -1 weights of x).
 * t in {-1, 0, 1}; layouts as oracle_gemv_i8.
 */
int oracle_gemv_i8_frac(int64_t M, int64_t N, int64_t K, const int8_t *t,
                        const int32_t *d, const int8_t *x, int frac, int64_t *y)
{
    if (M < 1 || N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0 || frac < 0 || frac > 62)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t r = 0; r < N; r++) {
            int64_t out = 0;
            for (int64_t g = 0; g < G; g++) {
                int64_t plus = 0, minus = 0;
                for (int64_t i = g * ORACLE_GROUP; i < (g + 1) * ORACLE_GROUP; i++) {
                    if (t[r * K + i] == 1)
                        plus += x[m * K + i];
                    else if (t[r * K + i] == -1)
                        minus += x[m * K + i];
                    else if (t[r * K + i] != 0)
                        return -1;
                }
                out += oracle_arshift((plus - minus) * (int64_t)d[r * G + g], frac);
            }
            y[m * N + r] = out;
        }
    }
    return 0;
}

/* The int64 value of a 64-bit two's-complement pattern (no implementation-defined conversion). */
static int64_t oracle_signed64(uint64_t v)
{
    if (v <= (uint64_t)INT64_MAX)
        return (int64_t)v;
    return -(int64_t)(~v) - 1;
}

/*
 * [IntEngine] §4.4 fixed-point int64 activations, with §5's statement that the
 * limb-decomposed apply is exact modulo 2^64: for every output o
 *   out_o = sum_b arshift( signed_sum_b * scale[o][b], frac ),
 *   signed_sum_b = sum_i t_i x_i,
 * with x int64 and every sum and product taken modulo 2^64 (two's-complement
 * wrapping); arshift acts on the int64 value of each group's wrapped product.
 * Where no step leaves the int64 range this is the exact integer result.
 * t in {-1, 0, 1} (a Q1_0 row is the case t in {-1, 1}); x [M][K] int64.
 */
int oracle_gemv_x64(int64_t M, int64_t N, int64_t K, const int8_t *t,
                    const int32_t *d, const int64_t *x, int frac, int64_t *y)
{
    if (M < 1 || N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0 || frac < 0 || frac > 62)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t r = 0; r < N; r++) {
            uint64_t out = 0;
            for (int64_t g = 0; g < G; g++) {
                uint64_t s = 0;
                for (int64_t i = g * ORACLE_GROUP; i < (g + 1) * ORACLE_GROUP; i++) {
                    if (t[r * K + i] == 1)
                        s += (uint64_t)x[m * K + i];
                    else if (t[r * K + i] == -1)
                        s -= (uint64_t)x[m * K + i];
                    else if (t[r * K + i] != 0)
                        return -1;
                }
                const uint64_t v = s * (uint64_t)(int64_t)d[r * G + g];
                out += (uint64_t)oracle_arshift(oracle_signed64(v), frac);
            }
            y[m * N + r] = oracle_signed64(out);
        }
    }
    return 0;
}

/*
 * [IntEngine] §4.1 Q1_0: 1-bit weights, bit[r][i] in {0, 1} standing for
 * sign -1 / +1, and for every output o
 *   signed_sum_b = 2 * pos_sum_b - block_total_b,
 *   pos_sum_b = sum of x over the weights whose bit is 1,
 *   block_total_b = sum of x over the group (the same for every output),
 *   out_o = sum_b arshift( signed_sum_b * scale[o][b], frac ).
 * Layouts: bits [N][K] uint8 in {0, 1}; d [N][K/128] int32; x [M][K] int8.
 */
int oracle_gemv_q1(int64_t M, int64_t N, int64_t K, const uint8_t *bits,
                   const int32_t *d, const int8_t *x, int frac, int64_t *y)
{
    if (M < 1 || N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0 || frac < 0 || frac > 62)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t r = 0; r < N; r++) {
            int64_t out = 0;
            for (int64_t g = 0; g < G; g++) {
                int64_t pos_sum = 0, block_total = 0;
                for (int64_t i = g * ORACLE_GROUP; i < (g + 1) * ORACLE_GROUP; i++) {
                    if (bits[r * K + i] > 1)
                        return -1;
                    block_total += x[m * K + i];
                    if (bits[r * K + i] == 1)
                        pos_sum += x[m * K + i];
                }
                out += oracle_arshift((2 * pos_sum - block_total) * (int64_t)d[r * G + g], frac);
            }
            y[m * N + r] = out;
        }
    }
    return 0;
}

/* Build the W_nonzero / W_negative bitmask pair of one 128-weight group. */
static void oracle_group_masks(const int8_t *trow, int64_t g, uint64_t nz[2], uint64_t neg[2])
{
    nz[0] = nz[1] = neg[0] = neg[1] = 0;
    for (int j = 0; j < ORACLE_GROUP; j++) {
        int8_t v = trow[g * ORACLE_GROUP + j];
        if (v != 0)
            nz[j >> 6] |= (uint64_t)1 << (j & 63);
        if (v < 0)
            neg[j >> 6] |= (uint64_t)1 << (j & 63);
    }
}

/*
 * The same GEMV through the two-bitmask masked sum: per group the row is held
 * as W_nonzero / W_negative ([BitState] §4), and the signed sum is
 * sum_{nz & !neg} x - sum_{nz & neg} x ([IntEngine] §4.2).
 */
int oracle_gemv_i8_masked(int64_t M, int64_t N, int64_t K, const int8_t *t,
                          const int32_t *d, const int8_t *x, int64_t *y)
{
    if (M < 1 || N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t r = 0; r < N; r++) {
            int64_t out = 0;
            for (int64_t g = 0; g < G; g++) {
                uint64_t nz[2], neg[2];
                oracle_group_masks(t + r * K, g, nz, neg);
                int64_t pos_sum = 0, neg_sum = 0;
                for (int j = 0; j < ORACLE_GROUP; j++) {
                    uint64_t bit = (uint64_t)1 << (j & 63);
                    int64_t xv = x[m * K + g * ORACLE_GROUP + j];
                    if ((nz[j >> 6] & bit) && !(neg[j >> 6] & bit))
                        pos_sum += xv;
                    if ((nz[j >> 6] & bit) && (neg[j >> 6] & bit))
                        neg_sum += xv;
                }
                out += (int64_t)d[r * G + g] * (pos_sum - neg_sum);
            }
            y[m * N + r] = out;
        }
    }
    return 0;
}

/*
 * The same GEMV through signed state populations ([BitState] §4). The
 * activation state is the magnitude s = |x_i| (0..128). For each state:
 *   A_s  = lanes whose activation magnitude is s
 *   M    = A_s & W_nonzero
 *   PNEG = activation_sign XOR W_negative
 *   C_s  = popcount(M) - 2 * popcount(M & PNEG)
 * and the group's signed sum is sum_s s * C_s.
 */
int oracle_gemv_i8_stateset(int64_t M, int64_t N, int64_t K, const int8_t *t,
                            const int32_t *d, const int8_t *x, int64_t *y)
{
    if (M < 1 || N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t r = 0; r < N; r++) {
            int64_t out = 0;
            for (int64_t g = 0; g < G; g++) {
                uint64_t nz[2], neg[2], asign[2] = {0, 0};
                oracle_group_masks(t + r * K, g, nz, neg);
                for (int j = 0; j < ORACLE_GROUP; j++)
                    if (x[m * K + g * ORACLE_GROUP + j] < 0)
                        asign[j >> 6] |= (uint64_t)1 << (j & 63);
                int64_t signed_sum = 0;
                for (int s = 1; s <= 128; s++) {
                    uint64_t As[2] = {0, 0};
                    for (int j = 0; j < ORACLE_GROUP; j++) {
                        int xv = x[m * K + g * ORACLE_GROUP + j];
                        if ((xv < 0 ? -xv : xv) == s)
                            As[j >> 6] |= (uint64_t)1 << (j & 63);
                    }
                    int64_t C = 0;
                    for (int h = 0; h < 2; h++) {
                        uint64_t Mh = As[h] & nz[h];
                        uint64_t pneg = asign[h] ^ neg[h];
                        C += oracle_popcount64(Mh) - 2 * oracle_popcount64(Mh & pneg);
                    }
                    signed_sum += (int64_t)s * C;
                }
                out += (int64_t)d[r * G + g] * signed_sum;
            }
            y[m * N + r] = out;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* 2. LNS8 S1|E4|L3 product states, eight phase accumulators.                */
/* ------------------------------------------------------------------------- */

/*
 * Product state of one lane ([BitState] §3, §3.1, §4 generic variant).
 * Activation byte xa = sign<<7 | code; code 0 is exact zero. Weight t in
 * {-1,0,1} with the group's scale code dcode. The scale is applied before the
 * L3/E4 split (the generic variant of §4): k = a + dcode - 74, which is the
 * product of the magnitudes 2^((a-74)/8) * 2^((dcode-74)/8) written as a code.
 * k <= 0 -> exact zero; k > 127 -> 127. Sign S1 = activation sign XOR [t < 0].
 * Returns 0 for an exact-zero product, else 1 with *k_out in 1..127 and
 * *neg_out the sign.
 */
static int oracle_lns8_product(uint8_t xa, int8_t t, uint8_t dcode, int *k_out, int *neg_out)
{
    int a = xa & 0x7f;
    int s_a = xa >> 7;
    if (t == 0 || a == 0)
        return 0;
    int k = a + (int)dcode - 74;
    if (k <= 0)
        return 0;
    if (k > 127)
        k = 127;
    *k_out = k;
    *neg_out = s_a ^ (t < 0 ? 1 : 0);
    return 1;
}

/*
 * Direct eight-phase accumulation ([BitState] §3.1): for every nonzero product
 * state k, phase = k & 7 (L3), payload = sign * (1 << (k >> 3)) (E4), and
 * A[phase] += payload. Layouts: t [N][K]; dcode [N][K/128] uint8;
 * xa [K] uint8; A [N][8] int64.
 */
int oracle_lns8_direct(int64_t N, int64_t K, const int8_t *t, const uint8_t *dcode,
                       const uint8_t *xa, int64_t *A)
{
    if (N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t r = 0; r < N; r++) {
        int64_t acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int64_t i = 0; i < K; i++) {
            int k, neg;
            if (!oracle_lns8_product(xa[i], t[r * K + i], dcode[r * G + i / ORACLE_GROUP], &k, &neg))
                continue;
            int64_t payload = (int64_t)1 << (k >> 3);
            acc[k & 7] += neg ? -payload : payload;
        }
        for (int p = 0; p < 8; p++)
            A[r * 8 + p] = acc[p];
    }
    return 0;
}

/*
 * Histogram path ([BitState] §3.1, last formula; §7 Phase A "signed POPCOUNT
 * histogram" and "histogram-to-A[0..7] equivalence"): build the signed count
 * H[phase][band] first, then A[p] = sum_b H[p][b] << b.
 */
int oracle_lns8_histogram(int64_t N, int64_t K, const int8_t *t, const uint8_t *dcode,
                          const uint8_t *xa, int64_t *A)
{
    if (N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t r = 0; r < N; r++) {
        int64_t H[8][16];
        memset(H, 0, sizeof(H));
        for (int64_t i = 0; i < K; i++) {
            int k, neg;
            if (!oracle_lns8_product(xa[i], t[r * K + i], dcode[r * G + i / ORACLE_GROUP], &k, &neg))
                continue;
            H[k & 7][k >> 3] += neg ? -1 : 1;
        }
        for (int p = 0; p < 8; p++) {
            int64_t a = 0;
            for (int b = 0; b < 16; b++)
                a += H[p][b] * ((int64_t)1 << b);
            A[r * 8 + p] = a;
        }
    }
    return 0;
}

/*
 * Tile64 x 2 phase-mask path ([BitState] §3.1, the spreadsheet procedure, read
 * from its prose since the workbook is not available): the 128 inputs of a
 * group are two 64-lane tiles; in each tile L3 builds eight phase selector
 * masks (lanes whose product phase is p), E4 supplies the power-of-two payload
 * and S1 the sign of each selected lane.
 */
int oracle_lns8_tile64(int64_t N, int64_t K, const int8_t *t, const uint8_t *dcode,
                       const uint8_t *xa, int64_t *A)
{
    if (N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t r = 0; r < N; r++) {
        int64_t acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int64_t g = 0; g < G; g++) {
            for (int tile = 0; tile < 2; tile++) {
                uint64_t sel[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                int e4[64], s1[64];
                for (int j = 0; j < 64; j++) {
                    int64_t i = g * ORACLE_GROUP + tile * 64 + j;
                    int k, neg;
                    e4[j] = 0;
                    s1[j] = 0;
                    if (!oracle_lns8_product(xa[i], t[r * K + i], dcode[r * G + g], &k, &neg))
                        continue;
                    sel[k & 7] |= (uint64_t)1 << j;
                    e4[j] = k >> 3;
                    s1[j] = neg;
                }
                for (int p = 0; p < 8; p++) {
                    for (int j = 0; j < 64; j++) {
                        if (!(sel[p] >> j & 1))
                            continue;
                        int64_t payload = (int64_t)1 << e4[j];
                        acc[p] += s1[j] ? -payload : payload;
                    }
                }
            }
        }
        for (int p = 0; p < 8; p++)
            A[r * 8 + p] = acc[p];
    }
    return 0;
}

/*
 * State-set population path ([BitState] §4 with §6): the activation state is
 * its code a (1..127; code 0 is excluded as exact zero). Per group and state,
 *   C_a = popcount(A_a & W_nonzero) - 2 * popcount(A_a & W_nonzero & PNEG),
 *   PNEG = activation_sign XOR W_negative,
 * is the signed population of state a, and all lanes of that state share one
 * product code k = a + dcode - 74 (the group shares dcode), so
 * A[k & 7] += C_a * 2^(k >> 3) after the same zero / saturation rule.
 */
int oracle_lns8_stateset(int64_t N, int64_t K, const int8_t *t, const uint8_t *dcode,
                         const uint8_t *xa, int64_t *A)
{
    if (N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t r = 0; r < N; r++) {
        int64_t acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int64_t g = 0; g < G; g++) {
            uint64_t nz[2], neg[2], asign[2] = {0, 0};
            oracle_group_masks(t + r * K, g, nz, neg);
            for (int j = 0; j < ORACLE_GROUP; j++)
                if (xa[g * ORACLE_GROUP + j] >> 7)
                    asign[j >> 6] |= (uint64_t)1 << (j & 63);
            for (int a = 1; a <= 127; a++) {
                uint64_t As[2] = {0, 0};
                for (int j = 0; j < ORACLE_GROUP; j++)
                    if ((xa[g * ORACLE_GROUP + j] & 0x7f) == a)
                        As[j >> 6] |= (uint64_t)1 << (j & 63);
                int64_t C = 0;
                for (int h = 0; h < 2; h++) {
                    uint64_t Mh = As[h] & nz[h];
                    uint64_t pneg = asign[h] ^ neg[h];
                    C += oracle_popcount64(Mh) - 2 * oracle_popcount64(Mh & pneg);
                }
                if (C == 0)
                    continue;
                int k = a + (int)dcode[r * G + g] - 74;
                if (k <= 0)
                    continue;
                if (k > 127)
                    k = 127;
                acc[k & 7] += C * ((int64_t)1 << (k >> 3));
            }
        }
        for (int p = 0; p < 8; p++)
            A[r * 8 + p] = acc[p];
    }
    return 0;
}

/*
 * Pure fractional-LNS reduction ([BitState] §5.2), as this library reads it
 * (the page fixes the primitives, not the table rounding or the tree shapes):
 *
 *   A value is (s, L): s in {-1, 0, +1} (0 = exact zero), L its log magnitude
 *   in code units with F fractional bits, held as the integer L * 2^F; the
 *   value is s * 2^((L - 74) / 8).
 *   Count fold: a signed state population C != 0 of product code k becomes
 *   (sign C, k * 2^F + LOG8[|C|]), LOG8[n] = round(8 log2(n) 2^F), n <= 128.
 *   Pairwise add, hi = the operand with the larger L (the first on a tie),
 *   diff = L_hi - L_lo:
 *     same sign:     (s_hi, L_hi + KP[diff]),  KP[i] = round(8 log2(1 + 2^(-i / (8 2^F))) 2^F)
 *     opposite sign: diff = 0 -> exact zero,
 *                    else (s_hi, L_hi + KM[diff]), KM[i] = round(8 log2(1 - 2^(-i / (8 2^F))) 2^F)
 *   with KP[i] = KM[i] = 0 from i = (8F + 40) 2^F on (both round to 0 there).
 *   Balanced tree over 2^m values: add(tree(left half), tree(right half)).
 *   Per row: each group's signed populations C_g[k] (k = a + d - 74 with the
 *   zero / saturation rule of the direct route) are folded into buckets; per
 *   phase p the sixteen band slots k = 8b + p form a tree; the groups' phase
 *   aggregates form a tree over G padded with zeros to a power of two; the
 *   eight phase aggregates form the final tree (8 -> 4 -> 2 -> 1).
 * Rounding is round half away from zero (llround). 1 <= F <= 6.
 * Output per row: sign[r], lam[r] (= L * 2^F) and S[r] = s * 2^((L - 74) / 8).
 */
typedef struct {
    int8_t s;
    int64_t lam;
} oracle_lnsv;

static int64_t oracle_lns_len(int F) { return (int64_t)(8 * F + 40) << F; }

static oracle_lnsv oracle_lns_add(oracle_lnsv u, oracle_lnsv v, const int64_t *KP, const int64_t *KM, int64_t len)
{
    if (u.s == 0)
        return v;
    if (v.s == 0)
        return u;
    const oracle_lnsv hi = u.lam >= v.lam ? u : v;
    const oracle_lnsv lo = u.lam >= v.lam ? v : u;
    const int64_t diff = hi.lam - lo.lam;
    oracle_lnsv r = hi;
    if (hi.s == lo.s) {
        r.lam = hi.lam + (diff < len ? KP[diff] : 0);
    } else if (diff == 0) {
        r.s = 0;
        r.lam = 0;
    } else {
        r.lam = hi.lam + (diff < len ? KM[diff] : 0);
    }
    return r;
}

static oracle_lnsv oracle_lns_tree(const oracle_lnsv *v, int64_t n, const int64_t *KP, const int64_t *KM,
                                   int64_t len)
{
    if (n == 1)
        return v[0];
    return oracle_lns_add(oracle_lns_tree(v, n / 2, KP, KM, len), oracle_lns_tree(v + n / 2, n / 2, KP, KM, len),
                          KP, KM, len);
}

/* The three tables of the pure-LNS reduction for F fractional bits (definitions above). */
int oracle_lns_tables(int F, int64_t *LOG8 /*[129]*/, int64_t *KP /*[len]*/, int64_t *KM /*[len]*/)
{
    if (F < 1 || F > 6)
        return -1;
    const double scale = ldexp(1.0, F);
    const int64_t len = oracle_lns_len(F);
    LOG8[0] = 0;
    for (int n = 1; n <= 128; n++)
        LOG8[n] = llround(8.0 * log2((double)n) * scale);
    for (int64_t i = 0; i < len; i++) {
        const double q = exp2(-(double)i / (8.0 * scale));
        KP[i] = llround(8.0 * log2(1.0 + q) * scale);
        KM[i] = i == 0 ? 0 : llround(8.0 * log2(1.0 - q) * scale);
    }
    return 0;
}

int64_t oracle_lns_table_len(int F) { return (F < 1 || F > 6) ? -1 : oracle_lns_len(F); }

int oracle_lns8_purelns(int64_t N, int64_t K, const int8_t *t, const uint8_t *dcode, const uint8_t *xa, int F,
                        int64_t *sign, int64_t *lam, double *S)
{
    if (N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0 || F < 1 || F > 6)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    int64_t Gp = 1;
    while (Gp < G)
        Gp *= 2;
    const int64_t len = oracle_lns_len(F);
    int64_t LOG8[129];
    int64_t *KP = malloc(sizeof(int64_t) * (size_t)len);
    int64_t *KM = malloc(sizeof(int64_t) * (size_t)len);
    oracle_lnsv *gagg = malloc(sizeof(oracle_lnsv) * (size_t)(8 * Gp));   /* [phase][group] */
    if (!KP || !KM || !gagg) {
        free(KP);
        free(KM);
        free(gagg);
        return -1;
    }
    oracle_lns_tables(F, LOG8, KP, KM);
    for (int64_t r = 0; r < N; r++) {
        for (int64_t g = 0; g < Gp; g++) {
            int64_t C[128];
            memset(C, 0, sizeof(C));
            if (g < G) {
                for (int64_t i = g * ORACLE_GROUP; i < (g + 1) * ORACLE_GROUP; i++) {
                    const int tv = t[r * K + i];
                    const int a = xa[i] & 0x7f;
                    if (tv == 0 || a == 0)
                        continue;
                    int k = a + (int)dcode[r * G + g] - 74;
                    if (k <= 0)
                        continue;
                    if (k > 127)
                        k = 127;
                    const int neg = (tv < 0) ^ (xa[i] >> 7);
                    C[k] += neg ? -1 : 1;
                }
            }
            for (int p = 0; p < 8; p++) {
                oracle_lnsv slots[16];
                for (int b = 0; b < 16; b++) {
                    const int64_t c = C[8 * b + p];
                    slots[b].s = (int8_t)(c > 0 ? 1 : (c < 0 ? -1 : 0));
                    slots[b].lam = c == 0 ? 0 : (int64_t)(8 * b + p) * ((int64_t)1 << F) + LOG8[c < 0 ? -c : c];
                }
                gagg[p * Gp + g] = oracle_lns_tree(slots, 16, KP, KM, len);
            }
        }
        oracle_lnsv ph[8];
        for (int p = 0; p < 8; p++)
            ph[p] = oracle_lns_tree(gagg + p * Gp, Gp, KP, KM, len);
        const oracle_lnsv R = oracle_lns_tree(ph, 8, KP, KM, len);
        sign[r] = R.s;
        lam[r] = R.s == 0 ? 0 : R.lam;
        S[r] = R.s == 0 ? 0.0 : (double)R.s * exp2(((double)R.lam / ldexp(1.0, F) - 74.0) / 8.0);
    }
    free(KP);
    free(KM);
    free(gagg);
    return 0;
}

/* F[p] = 2^((p - 2) / 8) ([BitState] §3), as fp64 from libm's exp2. */
void oracle_lns8_F(double F[8])
{
    for (int p = 0; p < 8; p++)
        F[p] = exp2((double)(p - 2) / 8.0);
}

/*
 * Dyadic materialisation ([BitState] §3.1): S = 2^-9 * sum_p A[p] * F[p],
 * summed in the fixed order p = 0..7 in fp64, each product and sum rounded
 * once (this file is built without FP contraction), then scaled by 2^-9.
 * F is the caller's table of 8 doubles.
 */
int oracle_lns8_materialise(int64_t N, const int64_t *A, const double *F, double *S)
{
    if (N < 0)
        return -1;
    for (int64_t r = 0; r < N; r++) {
        double acc = 0.0;
        for (int p = 0; p < 8; p++) {
            double term = (double)A[r * 8 + p] * F[p];
            acc = acc + term;
        }
        S[r] = acc * 0x1p-9;
    }
    return 0;
}

/*
 * The same materialisation in long double with F from exp2l, rounded to double
 * at the end: a higher-precision reference for S. S_abs receives
 * 2^-9 * sum_p |A[p]| * F[p], the scale against which rounding error is measured.
 */
int oracle_lns8_materialise_hi(int64_t N, const int64_t *A, double *S_hi, double *S_abs)
{
    if (N < 0)
        return -1;
    long double F[8];
    for (int p = 0; p < 8; p++)
        F[p] = exp2l((long double)(p - 2) / 8.0L);
    for (int64_t r = 0; r < N; r++) {
        long double acc = 0.0L, mag = 0.0L;
        for (int p = 0; p < 8; p++) {
            long double v = (long double)A[r * 8 + p] * F[p];
            acc += v;
            mag += v < 0 ? -v : v;
        }
        S_hi[r] = (double)(acc / 512.0L);
        S_abs[r] = (double)(mag / 512.0L);
    }
    return 0;
}

/*
 * Direct FP64 decode ([BitState] §7 Phase A "exact LNS8 decode reference"):
 * every nonzero product state contributes sign * 2^((k - 74) / 8), summed in
 * lane order. Also returns the sum of magnitudes for an error bound.
 */
int oracle_lns8_decode_fp64(int64_t N, int64_t K, const int8_t *t, const uint8_t *dcode,
                            const uint8_t *xa, double *S, double *S_abs)
{
    if (N < 1 || K < ORACLE_GROUP || K % ORACLE_GROUP != 0)
        return -1;
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t r = 0; r < N; r++) {
        double acc = 0.0, mag = 0.0;
        for (int64_t i = 0; i < K; i++) {
            int k, neg;
            if (!oracle_lns8_product(xa[i], t[r * K + i], dcode[r * G + i / ORACLE_GROUP], &k, &neg))
                continue;
            double v = exp2((double)(k - 74) / 8.0);
            acc += neg ? -v : v;
            mag += v;
        }
        S[r] = acc;
        S_abs[r] = mag;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* 3. Vocab-scale lm_head over 8 base-3 planes.                              */
/* ------------------------------------------------------------------------- */

static const int64_t oracle_pow3[8] = {2187, 729, 243, 81, 27, 9, 3, 1}; /* 3^(7-p) */

/*
 * Exact logits ([SKaiNET] BITNET_PLANES: 8 ternary planes, plane p weighted
 * 3^-p; here scaled by 3^7 so every weight is an integer):
 *   W[r][i] = sum_p planes[p][r][i] * 3^(7-p),   logit[r] = s[r] * sum_i W[r][i] * x[i].
 * Layouts: planes [8][N][K] int8; s [N] int32; x [K] int8; logits [N] int64.
 */
int oracle_lmhead_logits(int64_t N, int64_t K, const int8_t *planes, const int32_t *s,
                         const int8_t *x, int64_t *logits)
{
    if (N < 1 || K < 1)
        return -1;
    for (int64_t r = 0; r < N; r++) {
        int64_t dot = 0;
        for (int64_t i = 0; i < K; i++) {
            int64_t w = 0;
            for (int p = 0; p < 8; p++)
                w += (int64_t)planes[(int64_t)p * N * K + r * K + i] * oracle_pow3[p];
            dot += w * (int64_t)x[i];
        }
        logits[r] = (int64_t)s[r] * dot;
    }
    return 0;
}

/* Ordering for the top-k: score descending, then row index ascending. */
static const int64_t *oracle_sort_scores;

static int oracle_cmp_desc(const void *pa, const void *pb)
{
    int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
    int64_t sa = oracle_sort_scores[a], sb = oracle_sort_scores[b];
    if (sa != sb)
        return sa > sb ? -1 : 1;
    return a < b ? -1 : (a > b ? 1 : 0);
}

/* Rows sorted by (score desc, index asc); the first k are the top-k. */
static int64_t *oracle_sorted_rows(int64_t n, const int64_t *scores)
{
    int64_t *idx = (int64_t *)malloc((size_t)n * sizeof(int64_t));
    if (!idx)
        return NULL;
    for (int64_t r = 0; r < n; r++)
        idx[r] = r;
    oracle_sort_scores = scores;
    qsort(idx, (size_t)n, sizeof(int64_t), oracle_cmp_desc);
    return idx;
}

/*
 * Argmax with the lowest-index tie-break ([IntEngine] §3.3 "Argmax / sampling:
 * lowest-index tie-break", §3.2).
 */
int64_t oracle_argmax(int64_t N, const int64_t *scores)
{
    if (N < 1)
        return -1;
    int64_t best = 0;
    for (int64_t r = 1; r < N; r++)
        if (scores[r] > scores[best])
            best = r;
    return best;
}

/* Top-k of a score vector under (score desc, index asc): the full sort, first k. */
int oracle_topk(int64_t N, const int64_t *scores, int64_t k, int32_t *ids, int64_t *top)
{
    if (N < 1 || k < 1 || k > N)
        return -1;
    int64_t *idx = oracle_sorted_rows(N, scores);
    if (!idx)
        return -1;
    for (int64_t j = 0; j < k; j++) {
        ids[j] = (int32_t)idx[j];
        top[j] = scores[idx[j]];
    }
    free(idx);
    return 0;
}

/*
 * Two-stage top-k ([SKaiNET] closing comments, BitNetTwoStageDecode):
 *   stage 1: a scan of planes 0..3 over the whole vocabulary,
 *            stage1[r] = sum_i (sum_{p<4} planes[p][r][i] * 3^(7-p)) * x[i];
 *   bound:   the truncation of row r is at most rowScale(r) * (sum_{p=4..7} 3^-p)
 *            * sum|x|, i.e. B[r] = s[r] * 40 * sum_i |x_i| in integer units;
 *            lo[r] = s[r]*stage1[r] - B[r], hi[r] = s[r]*stage1[r] + B[r];
 *   select:  tau = the k-th best lower bound; every row whose upper bound
 *            reaches it (hi[r] >= tau) is rescored exactly with planes 4..7;
 *   result:  the top-k of the rescored rows, equal to the full-matmul top-k.
 * The candidate cap of the page (maxCandidates) is not applied: this is the
 * exact procedure. lo, hi may be NULL; n_cand receives the candidate count.
 */
int oracle_lmhead_two_stage(int64_t N, int64_t K, const int8_t *planes, const int32_t *s,
                            const int8_t *x, int64_t k, int32_t *ids, int64_t *top,
                            int64_t *lo_out, int64_t *hi_out, int64_t *n_cand)
{
    if (N < 1 || K < 1 || k < 1 || k > N)
        return -1;
    int64_t sum_abs_x = 0;
    for (int64_t i = 0; i < K; i++)
        sum_abs_x += x[i] < 0 ? -(int64_t)x[i] : (int64_t)x[i];

    int64_t *stage1 = (int64_t *)malloc((size_t)N * sizeof(int64_t));
    int64_t *lo = (int64_t *)malloc((size_t)N * sizeof(int64_t));
    int64_t *hi = (int64_t *)malloc((size_t)N * sizeof(int64_t));
    int64_t *exact = (int64_t *)malloc((size_t)N * sizeof(int64_t));
    if (!stage1 || !lo || !hi || !exact) {
        free(stage1); free(lo); free(hi); free(exact);
        return -1;
    }
    for (int64_t r = 0; r < N; r++) {
        int64_t dot = 0;
        for (int64_t i = 0; i < K; i++) {
            int64_t w = 0;
            for (int p = 0; p < 4; p++)
                w += (int64_t)planes[(int64_t)p * N * K + r * K + i] * oracle_pow3[p];
            dot += w * (int64_t)x[i];
        }
        stage1[r] = dot;
        int64_t B = (int64_t)s[r] * 40 * sum_abs_x;
        lo[r] = (int64_t)s[r] * dot - B;
        hi[r] = (int64_t)s[r] * dot + B;
    }
    /* tau = k-th largest lower bound. */
    int64_t *order = oracle_sorted_rows(N, lo);
    if (!order) {
        free(stage1); free(lo); free(hi); free(exact);
        return -1;
    }
    int64_t tau = lo[order[k - 1]];
    free(order);

    /* Rescore every candidate exactly; non-candidates get the lowest score. */
    int64_t C = 0;
    for (int64_t r = 0; r < N; r++) {
        if (hi[r] < tau) {
            exact[r] = INT64_MIN;
            continue;
        }
        C++;
        int64_t rest = 0;
        for (int64_t i = 0; i < K; i++) {
            int64_t w = 0;
            for (int p = 4; p < 8; p++)
                w += (int64_t)planes[(int64_t)p * N * K + r * K + i] * oracle_pow3[p];
            rest += w * (int64_t)x[i];
        }
        exact[r] = (int64_t)s[r] * (stage1[r] + rest);
    }
    int64_t *idx = oracle_sorted_rows(N, exact);
    if (!idx) {
        free(stage1); free(lo); free(hi); free(exact);
        return -1;
    }
    for (int64_t j = 0; j < k; j++) {
        ids[j] = (int32_t)idx[j];
        top[j] = exact[idx[j]];
    }
    if (lo_out)
        memcpy(lo_out, lo, (size_t)N * sizeof(int64_t));
    if (hi_out)
        memcpy(hi_out, hi, (size_t)N * sizeof(int64_t));
    if (n_cand)
        *n_cand = C;
    free(idx);
    free(stage1); free(lo); free(hi); free(exact);
    return 0;
}

/*
 * Balanced-ternary digits of an integer weight ([SKaiNET] BITNET_PLANES: plane
 * p is the base-3 digit of weight 3^(7-p) in {-1,0,1}). w must lie in
 * [-3280, 3280] = +-(3^8 - 1)/2. Digits are produced least significant first
 * by taking the remainder in {-1,0,1}.
 */
int oracle_planes_of_weight(int32_t w, int8_t digits[8])
{
    if (w < -3280 || w > 3280)
        return -1;
    int32_t v = w;
    for (int p = 7; p >= 0; p--) {
        int32_t rem = ((v % 3) + 3) % 3; /* 0, 1, 2 */
        int32_t digit = rem == 2 ? -1 : rem;
        digits[p] = (int8_t)digit;
        v = (v - digit) / 3;
    }
    return v == 0 ? 0 : -1;
}
