// tg_internal.h -- definitions shared by the translation units of libtg.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "tg.h"

namespace tgi {

constexpr int kTileRows = 32;   // rows per mask tile: one row per lane of a warp
constexpr int kLnsBlockRows = 16;  // rows per LNS8 block: the M of one 16x8x16 tensor-core step

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Per translation unit: read-and-clear of that unit's device error word.
// Each returns 0 or TG_ERR_DEVICE, or TG_ERR_CUDA if the query failed.
int gemv_take_device_error(void *stream);
int gemv_mma_take_device_error(void *stream);
int lns8_take_device_error(void *stream);
int lmhead_take_device_error(void *stream);

// Small-batch ternary GEMM on the tensor cores (2 <= M <= 64); arguments as
// checked by tg_gemv_i8; wait_cycles bounds each device-side wait (0 = the
// default). Returns a tg_status.
int gemv_i8_mma(const uint4 *masks, const int32_t *scales, const int8_t *x, int64_t *y, int N, int G,
                int tiles, int M, int64_t max_abs_scale, bool q1, int frac, int64_t wait_cycles, cudaStream_t s);

// Ternary / Q1_0 GEMV for a few tokens on the CUDA cores; x is int8 [M][K], or
// int64 [M][K] when x64 (sums modulo 2^64); pdl: launch as a programmatic
// dependent (constant weights). Arguments as checked by tg_gemv_i8. Returns a
// tg_status.
int gemv_i8_mt(const uint4 *masks, const int32_t *scales, const void *x, int64_t *y, int N, int G, int tiles,
               int M, bool q1, bool x64, int frac, bool pdl, cudaStream_t s);

// Ternary / Q1_0 GEMV for a few tokens through warp-level fp16 MMAs; the token
// activations' fragments must fit in shared memory (gemv_i8_hmma_fits(G)).
bool gemv_i8_hmma_fits(int G);
int gemv_i8_hmma(const uint4 *masks, const int32_t *scales, const int8_t *x, int64_t *y, int N, int G, int tiles,
                 int M, bool q1, int frac, bool pdl, cudaStream_t s);

// The argument checks of tg_lmhead_argmax_topk that precede its workspace check
// (pointers, alignment, kind, shape), in the same order; TG_OK or the status.
int lmhead_check_args(const tg_layout *L, const void *w, const int8_t *x, int32_t k, const int64_t *logits,
                      const int32_t *argmax, const int32_t *ids, const int64_t *scores, const int32_t *ncand);

// LNS8 eight-phase GEMV by the state-population route (TG_FLAG_LNS8_STATE_SET);
// arguments as checked by tg_gemv_lns8_phase. Returns a tg_status.
int lns8_stateset(const uint4 *masks, const uint8_t *codes, const uint8_t *xa, int64_t *A, double *S,
                  const double F[8], const double *F_dev, int N, int G, int tiles, cudaStream_t s);

// LNS8 by the pure fractional-LNS reduction (TG_FLAG_LNS8_PURE_LNS), F
// internal fractional bits (1..6); arguments as checked by tg_gemv_lns8_phase.
int lns8_purelns(const uint4 *masks, const uint8_t *codes, const uint8_t *xa, int64_t *A, double *S, int N, int G,
                 int F, cudaStream_t s);

}  // namespace tgi
