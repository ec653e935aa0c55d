/*
 * tg.h -- C ABI of libtg.so, an exact ternary weight apply for one GB300 GPU.
 *
 * Three forms of the batch-1 decode weight apply, all computed in integers:
 *
 *   1. Ternary GEMV with int8 activations and per-group integer scales
 *      (integer_engine.md §4.2 "BitNet b1.58 ternary", §4.4 "int8 activations +
 *      int32 accumulation"; BitState brief §4 for the W_nonzero / W_negative
 *      representation):
 *          y[m][r] = sum_g d[r][g] * ( sum_{i in group g} t[r][i] * x[m][i] ).
 *      Groups are 128 weights; the per-group partial is an int32, the sum over
 *      groups an int64. The same call takes binary Q1_0 weights {-1, +1}
 *      (§4.1, one sign bit per weight), the per-group floor arshift(., frac)
 *      of §4.1/§4.2 (layout field frac, 0 by default), 1 to 64 tokens, and
 *      int64 fixed-point activations (§4.4, sums modulo 2^64; TG_FLAG_X_INT64).
 *
 *   2. LNS8 S1|E4|L3 eight-phase accumulation (BitState brief §3, §3.1 and the
 *      generic variant of §4): every nonzero product state
 *          k = a + d - 74   (k <= 0 -> exact zero, k > 127 -> 127)
 *      adds sign * (1 << (k >> 3)) into A[k & 7], and
 *          S = 2^-9 * sum_p A[p] * 2^((p - 2) / 8)        (fp64).
 *      Besides the direct per-lane route, the same result by signed state
 *      populations (§4 with §6; TG_FLAG_LNS8_STATE_SET), and an approximate
 *      pure fractional-LNS reduction (§5.2; TG_FLAG_LNS8_PURE_LNS).
 *
 *   3. Vocab-scale lm_head over 8 base-3 planes (SKaiNET-transformers issue
 *      #337, BITNET_PLANES and BitNetTwoStageDecode): the integer weight is
 *      W = sum_p t_p * 3^(7 - p), the logit s[r] * sum_i W[r][i] x[i]; the call
 *      returns the argmax (lowest index among equal maxima, integer_engine.md
 *      §3.3) and the exact top-k, either from all 8 planes or by the two-stage
 *      scan (planes 0-3) with exact bounded rescoring (planes 4-7).
 *
 * Conventions shared by every call:
 *   - Every call returns a tg_status: 0 on success, a negative code on error.
 *     Nothing aborts, throws or prints; tg_status_string() names a code.
 *   - The caller owns every buffer. Compute calls take DEVICE pointers and a
 *     cudaStream_t passed as void* (NULL = the legacy default stream); they
 *     only enqueue work on that stream and return at once. The library
 *     allocates no memory; the lm_head takes a caller-owned device workspace.
 *   - Stream order holds as usual: a call's kernels start after the work
 *     enqueued before it has finished (or, for kernels launched as
 *     programmatic dependents, wait for it before touching x, y or the
 *     workspace). Some of the library's kernels let the next kernel on the
 *     stream launch early; a caller's kernel launched with programmatic stream
 *     serialisation right after a call must wait (griddepcontrol.wait /
 *     cudaGridDependencySynchronize) before it reads that call's outputs.
 *   - Arguments are validated on the host before anything is enqueued; on an
 *     argument error no output buffer is touched.
 *   - The library keeps no state between calls, apart from one device error
 *     word that a kernel sets if a bounded wait of its own runs out
 *     (tg_device_error()), the fixed device scratch of
 *     tg_lmhead_argmax_topk_noalloc, and the constant host tables of the
 *     pure-LNS route (computed on first use for each precision).
 *   - Packing (tg_pack_weights) runs synchronously on the host, from host
 *     arrays into a host buffer; the caller copies that buffer to the device.
 */
#ifndef TG_H
#define TG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
    TG_OK = 0,
    TG_ERR_ARG = -1,       /* null pointer, misaligned pointer, unknown kind, or a
                              layout that does not match the call */
    TG_ERR_SHAPE = -2,     /* N < 1, K < 128 or K % 128 != 0, M or k out of range */
    TG_ERR_VALUE = -3,     /* a trit outside {-1,0,1}, or an lm_head row scale <= 0 */
    TG_ERR_BOUND = -4,     /* a worst-case sum could leave its integer type
                              (the fail-loud bound of integer_engine.md §3.4) */
    TG_ERR_WORKSPACE = -5, /* workspace pointer missing, misaligned or too small */
    TG_ERR_CUDA = -6,      /* a CUDA launch or query failed */
    TG_ERR_DEVICE = -7     /* a kernel gave up a bounded wait (tg_device_error) */
};

/* Weight kinds (argument `kind`). */
enum {
    TG_TERNARY_I8 = 1,   /* ternary weights, int32 scale per 128-weight group   */
    TG_TERNARY_LNS8 = 2, /* ternary weights, uint8 LNS8 scale code per group    */
    TG_PLANES8 = 3,      /* 8 ternary base-3 planes, int32 scale per row        */
    TG_BINARY_Q1 = 4     /* binary Q1_0 weights {-1,+1}, int32 scale per group  */
};

#define TG_GROUP 128     /* weights per group (BitState brief §2: 128-weight groups) */
#define TG_MAX_M 64      /* largest token count of tg_gemv_i8 */
#define TG_MAX_K 1024    /* largest k of tg_lmhead_argmax_topk */

/*
 * Description of one packed weight blob, filled by tg_pack_weights (or by
 * tg_layout_init, which computes the same sizes without packing). Offsets are
 * byte offsets from the start of the blob; every region starts on a 256-byte
 * boundary. The blob's device copy must be 256-byte aligned.
 *
 * TG_TERNARY_I8 (rows tiled by 32, tiles = ceil(N/32)):
 *   masks  [tiles][G][2][32][16 B]: for tile T, group g, half h (group lanes
 *          64h..64h+63) and row r = 32T + l, 16 bytes = four little-endian
 *          uint32 words; word u holds group lanes 64h + 16u + (0..15), lane
 *          64h + 16u + 4j + b in bits 8b+2j (W_nonzero) and 8b+2j+1
 *          (W_negative). W_negative is set only where W_nonzero is.
 *   scales [tiles][G][32]: int32 scale of row 32T + l.
 *   Rows N..32*tiles-1 are padding: zero masks, zero scales.
 * TG_BINARY_Q1 (integer_engine.md §4.1 Q1_0; rows tiled by 32, tiles = ceil(N/32)):
 *   masks  [tiles][G][32][16 B]: for tile T, group g and row r = 32T + l,
 *          16 bytes = four little-endian uint32 words; word u holds group
 *          lanes 32u + (0..31), lane 32u + 4j + b in bit 8b + j, set for a +1
 *          weight and clear for -1.
 *   scales [tiles][G][32]: int32 scale of row 32T + l (as TG_TERNARY_I8).
 *   Rows N..32*tiles-1 are padding: zero bits, zero scales.
 * TG_TERNARY_LNS8 (rows in blocks of 16, tiles = ceil(N/16)): the same mask
 * pair, ordered for 16x8x16 tensor-core steps:
 *   masks  [tiles][G][32][16 B]: entry l = 4q + j (q = 0..7, j = 0..3) holds,
 *          for each 16-lane chunk c = 0..7 of group g, the trits of rows q and
 *          q+8 of the block at group lanes 16c + {2j, 2j+1, 2j+8, 2j+9}: four
 *          pairs r = 0..3 = (row q; 2j, 2j+1), (row q+8; 2j, 2j+1),
 *          (row q; 2j+8, 2j+9), (row q+8; 2j+8, 2j+9). Pair r of chunk c sits in
 *          word c/2 with r' = 4(c%2) + r: the first trit's W_nonzero /
 *          W_negative bits at 7-r' and 15-r', the second's at 23-r' and 31-r'.
 *   scales [tiles][G][16]: uint8 LNS8 code of row 16*tile + i.
 *   Rows N..16*tiles-1 are padding: zero masks, zero codes.
 * TG_PLANES8: rows of 2K bytes, row r at byte 2rK of the blob (mask_off = 0):
 *   masks  the row's first K bytes (hi at mask_off + 2rK), int8, planes 0-3 as
 *          one balanced base-3 number per weight, hi = 27 t0 + 9 t1 + 3 t2 + t3
 *          in [-40, 40];
 *   aux    its next K bytes (lo at aux_off + 2rK, aux_off = K), int8, planes
 *          4-7 the same way, lo = 27 t4 + 9 t5 + 3 t6 + t7, so W = 81 hi + lo
 *          (one row's two digit groups are adjacent: the full scan then reads
 *          one contiguous stream, measured 13% faster than two regions);
 *          mask_bytes = aux_bytes = N * K;
 *   scales [N] int32 row scale s[r] >= 1;
 *   aux2   [N] uint8, m[r] = max_i |lo[r][i]| (<= 40), the row's own bound on
 *          the planes 4-7 residual (0 for an exactly-ternary row).
 */
typedef struct tg_layout {
    int32_t kind;
    int32_t version;        /* 1 */
    int64_t N, K;           /* rows, columns (K % 128 == 0) */
    int64_t G;              /* groups per row, K / 128 */
    int64_t tiles;          /* ceil(N/32) (I8), ceil(N/16) (LNS8), else 0 */
    int64_t mask_off, mask_bytes;
    int64_t scale_off, scale_bytes;
    int64_t aux_off, aux_bytes;
    int64_t aux2_off, aux2_bytes;
    int64_t total_bytes;
    int64_t max_abs_scale;  /* max |scale| seen when packing (0 from tg_layout_init) */
    int64_t flags;          /* TG_FLAG_* bits, 0 after packing; the caller may set them */
    int64_t frac;           /* per-group floor shift (TG_TERNARY_I8, TG_BINARY_Q1): 0..62;
                               internal fractional bits of the pure-LNS route (TG_TERNARY_LNS8
                               with TG_FLAG_LNS8_PURE_LNS): 1..6; otherwise 0. 0 after packing */
    int64_t wait_limit;     /* SM clock cycles each bounded device-side wait may last before
                               the kernel gives up and reports TG_ERR_DEVICE (the tensor-memory
                               batched GEMM is the kernel with such waits); 0 = the default,
                               2^32 cycles (about two seconds). A caller that wants a stuck
                               kernel to fail sooner sets it; tests set it very low to exercise
                               the give-up path. 0 after packing */
    int64_t reserved[1];
} tg_layout;

/*
 * Layout flag: the packed weights are constant -- no device work on the stream
 * of an apply call writes them. A tg_gemv_i8 call on such weights with up to 16
 * tokens (or int64 activations) is launched as a programmatic dependent of the
 * previous kernel on the stream: it may start streaming its weights while that
 * kernel is still running, and it waits for that kernel to finish (and its
 * writes to be visible) before it reads x or writes y. Without the flag every
 * call starts after the previous work on the stream has finished.
 */
#define TG_FLAG_CONST_WEIGHTS 1

/*
 * Layout flag (TG_TERNARY_LNS8): tg_gemv_lns8_phase takes the signed
 * state-population route of the BitState brief (§4, W_nonzero / W_negative
 * with C_s = popcount(M) - 2 * popcount(M & PNEG), and §6, the activation state
 * sets built once and reused across rows) instead of the direct per-lane
 * route. A and S are identical; only the work and its cost differ.
 */
#define TG_FLAG_LNS8_STATE_SET 2

/*
 * Layout flag (TG_TERNARY_I8, TG_BINARY_Q1): the activations of tg_gemv_i8 are
 * int64 fixed-point values (integer_engine.md §4.4) -- x points to int64
 * [M][K], 16-byte aligned, passed through the int8_t pointer. Every sum and
 * product of the apply is then taken modulo 2^64 (two's-complement wrapping,
 * §5: the base-256 limb decomposition is exact modulo 2^64): the result is
 * exact whenever no step leaves the int64 range, and there is no TG_ERR_BOUND
 * check. Computed by signed base-256 digit planes of x, as many as the largest
 * activation needs; eight planes of one token must fit the kernel's staging
 * area, so K is at most 23,680 for one token and 17,792 for more
 * (TG_ERR_SHAPE beyond).
 */
#define TG_FLAG_X_INT64 4

/*
 * Layout flag (TG_TERNARY_LNS8): tg_gemv_lns8_phase takes the pure
 * fractional-LNS reduction of the BitState brief §5.2 -- no linear
 * accumulator; signed state populations are folded into log-domain buckets
 * and summed by pairwise kappa+/kappa- adds from tables with layout->frac
 * (1..6) internal fractional bits, in balanced trees over the bands, the
 * groups and the eight phases. Approximate by design. Outputs: A[r][0] = sign
 * (-1, 0, +1), A[r][1] = log magnitude in code units times 2^frac,
 * A[r][2..7] = 0; S[r] (if not NULL) = sign * 2^((A[r][1] / 2^frac - 74) / 8).
 * Not combinable with TG_FLAG_LNS8_STATE_SET.
 */
#define TG_FLAG_LNS8_PURE_LNS 8

/* Static string naming a status code. Never NULL. */
const char *tg_status_string(int status);

/*
 * Fill *out with the sizes and offsets of the packed blob of `kind` for an
 * N x K weight, without packing anything (max_abs_scale = 0).
 * Errors: TG_ERR_ARG (null out, unknown kind), TG_ERR_SHAPE.
 */
int tg_layout_init(int kind, int64_t N, int64_t K, tg_layout *out);

/* Size in bytes of the packed blob of `kind` for an N x K weight; 0 if invalid. */
size_t tg_packed_bytes(int kind, int64_t N, int64_t K);

/*
 * Pack host weights into the device layout above (host -> host, synchronous).
 *   trits   TG_TERNARY_*: int8 [N][K] in {-1,0,1}; TG_BINARY_Q1: int8 [N][K] in {-1,+1};
 *           TG_PLANES8:   int8 [8][N][K] in {-1,0,1}, plane p weighs 3^(7-p)
 *           (SKaiNET #337: plane p has weight 3^-p; scaled by 3^7 to integers).
 *   scales  TG_TERNARY_I8, TG_BINARY_Q1: int32 [N][K/128]; TG_TERNARY_LNS8: uint8 [N][K/128]
 *           LNS8 codes; TG_PLANES8: int32 [N], each >= 1.
 *   out     host buffer of out_bytes >= tg_packed_bytes(kind, N, K); any
 *           alignment. layout receives the description (may not be NULL).
 * Errors: TG_ERR_ARG, TG_ERR_SHAPE, TG_ERR_VALUE (bad trit / row scale <= 0),
 * TG_ERR_WORKSPACE (out_bytes too small). On error *out is unspecified.
 */
int tg_pack_weights(int kind, int64_t N, int64_t K, const int8_t *trits, const void *scales,
                    void *out, size_t out_bytes, tg_layout *layout);

/*
 * Ternary (or binary Q1_0) GEMV / small-batch GEMM with int8 activations
 * (integer_engine.md §4.1, §4.2 with §4.4; BitState brief §4 masks):
 *   y[m][r] = sum_g arshift( d[r][g] * sum_{i in group g} t[r][i] * x[m][i], frac )   (int64)
 *   arshift(v, frac) is floor(v / 2^frac) (each group's scaled sum floored on
 *   its own, then summed); frac = layout->frac, 0 by default (no floor). For
 *   TG_BINARY_Q1 every t is -1 or +1 and the group's signed sum is formed as
 *   2 * (sum of x over the +1 weights) - (sum of x over the group).
 *   layout  a TG_TERNARY_I8 or TG_BINARY_Q1 layout from tg_pack_weights
 *           (max_abs_scale set), frac in 0..62.
 *   w       device copy of the packed blob, 256-byte aligned.
 *   x       device int8 [M][K], 16-byte aligned; any value in [-128, 127].
 *   M       1..TG_MAX_M tokens (1 = batch-1 decode).
 *   y       device int64 [M][N], 8-byte aligned; fully overwritten.
 * The result does not depend on launch geometry or order: every sum is an
 * integer sum with no possible overflow (checked: G * 128 * 128 * max|d| < 2^62).
 * Errors: TG_ERR_ARG, TG_ERR_SHAPE, TG_ERR_BOUND, TG_ERR_CUDA.
 */
int tg_gemv_i8(const tg_layout *layout, const void *w, const int8_t *x, int64_t M,
               int64_t *y, void *stream);

/*
 * LNS8 eight-phase GEMV (BitState brief §3, §3.1; generic variant of §4):
 *   xa      device uint8 [K] activation bytes sign<<7 | code (code 0 = zero,
 *           whatever the sign), 16-byte aligned.
 *   For every lane with t != 0 and code a != 0 the product code is
 *   k = a + d[r][g] - 74 with d the group's scale code; k <= 0 is exact zero,
 *   k > 127 saturates to 127; the sign is the activation sign XOR [t < 0].
 *   F       device fp64 [8], 8-byte aligned, or NULL: the phase constants of
 *           the materialisation. NULL uses the built-in F[p] = 2^((p-2)/8)
 *           (BitState brief §3.1: phase p of band b is worth 2^(b + (p-2)/8 - 9)),
 *           the correctly rounded fp64 values from the host's exp2. A caller
 *           that keeps its own table (another rounding, a rescaled basis)
 *           passes it here. Read by the kernel; the caller keeps it valid until
 *           the call's work on the stream is done. Must be NULL with
 *           TG_FLAG_LNS8_PURE_LNS (that route's S is a log-domain value).
 *   A       device int64 [N][8]: A[r][k & 7] += sign * (1 << (k >> 3)).
 *   S       device fp64 [N] or NULL: S[r] = 2^-9 * sum_{p=0..7} A[r][p] * F[p],
 *           summed in the order p = 0..7, each product and sum rounded once
 *           (no fused multiply-add).
 * Errors: TG_ERR_ARG, TG_ERR_SHAPE, TG_ERR_BOUND (K >= 65536), TG_ERR_CUDA.
 */
int tg_gemv_lns8_phase(const tg_layout *layout, const void *w, const uint8_t *xa, const double *F,
                       int64_t *A, double *S, void *stream);

/* Device workspace bytes tg_lmhead_argmax_topk needs for this layout and k. */
size_t tg_lmhead_workspace_bytes(const tg_layout *layout, int32_t k);

/*
 * lm_head over 8 base-3 planes with argmax and exact top-k (SKaiNET #337):
 *   x       device int8 [K], 16-byte aligned.
 *   k       1..min(N, TG_MAX_K).
 *   logits  device int64 [N] or NULL.
 *           Non-NULL: all 8 planes are read, logits[r] = s[r] * sum_i W[r][i] x[i]
 *           is written for every row, and the top-k is taken over them.
 *           NULL: the two-stage path. Stage 1 scans planes 0-3 for every row;
 *           the planes 4-7 residual of row r is bounded by s[r] * m[r] * sum|x|
 *           (m[r] <= 40, the page's bound rowScale * (sum_{p=4..7} 3^-p) * sum|h|
 *           in integer units); every row whose upper bound reaches a lower bound
 *           on the k-th best lower bound is rescored exactly with planes 4-7.
 *           The result equals the full 8-plane top-k.
 *   argmax  device int32 [1]: the lowest row index among the maximal logits.
 *   ids     device int32 [k], scores device int64 [k]: the top-k in the order
 *           (score descending, row index ascending).
 *   ncand   device int32 [1] or NULL: rows rescored (two-stage) or rows
 *           considered by the final selection (full path).
 *   ws      device workspace, 256-byte aligned, ws_bytes >=
 *           tg_lmhead_workspace_bytes(layout, k). Contents on entry do not matter.
 * Errors: TG_ERR_ARG, TG_ERR_SHAPE, TG_ERR_BOUND, TG_ERR_WORKSPACE, TG_ERR_CUDA.
 */
int tg_lmhead_argmax_topk(const tg_layout *layout, const void *w, const int8_t *x, int32_t k,
                          int64_t *logits, int32_t *argmax, int32_t *ids, int64_t *scores,
                          int32_t *ncand, void *ws, size_t ws_bytes, void *stream);

/* Size of the library's own lm_head scratch used by tg_lmhead_argmax_topk_noalloc. */
#define TG_NOALLOC_SCRATCH_BYTES (4 * 1024 * 1024)

/*
 * tg_lmhead_argmax_topk without a caller workspace. The pages have no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory themselves: a plugin whose host framework hands out device memory only
 * through its own allocator, a serving process whose device memory is already
 * reserved by a cache pool, or a latency-critical loop that may not call
 * cudaMalloc because it can block on the device.
 *
 * Same arguments, results and errors as tg_lmhead_argmax_topk, minus ws and
 * ws_bytes: the workspace is a fixed array of TG_NOALLOC_SCRATCH_BYTES in the
 * library's own device memory, which every GPU that loads the library keeps
 * until the process exits. The call itself allocates nothing.
 *   - Limit: problems whose tg_lmhead_workspace_bytes(layout, k) exceeds
 *     TG_NOALLOC_SCRATCH_BYTES (N above 259,008 rows) are rejected with
 *     TG_ERR_WORKSPACE before anything is enqueued. The other arguments are
 *     checked first, in the same order as tg_lmhead_argmax_topk, so an invalid
 *     call gets the same TG_ERR_ARG / TG_ERR_SHAPE whatever its size.
 *   - The first call on each device looks up the array's device address with
 *     that device current and caches it for the life of the process; make that
 *     first call before any stream capture. A failed lookup returns
 *     TG_ERR_CUDA. The cached address does not survive cudaDeviceReset: after
 *     resetting a device, do not use this call on it again in the same process.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents (nothing needs to be cleared: each call resets what it counts).
 *     Calls whose work overlaps on the GPU race on it; the caller must order
 *     them (one stream, or explicit events).
 */
int tg_lmhead_argmax_topk_noalloc(const tg_layout *layout, const void *w, const int8_t *x,
                                  int32_t k, int64_t *logits, int32_t *argmax, int32_t *ids,
                                  int64_t *scores, int32_t *ncand, void *stream);

/*
 * Read and clear the device error word: *code receives 0, or TG_ERR_DEVICE if
 * a kernel gave up a bounded wait since the last read. Synchronises `stream`.
 * Errors: TG_ERR_ARG (null code), TG_ERR_CUDA.
 */
int tg_device_error(void *stream, int32_t *code);

#ifdef __cplusplus
}
#endif

#endif /* TG_H */
