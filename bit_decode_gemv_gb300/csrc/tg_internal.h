// tg_internal.h -- definitions shared by the translation units of libtg.
#pragma once

#include <cstddef>
#include <cstdint>

#include "tg.h"

namespace tgi {

constexpr int kTileRows = 32;   // rows per mask tile: one row per lane of a warp
constexpr int kLnsBlockRows = 16;  // rows per LNS8 block: the M of one 16x8x16 tensor-core step

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Per translation unit: read-and-clear of that unit's device error word.
// Each returns 0 or TG_ERR_DEVICE, or TG_ERR_CUDA if the query failed.
int gemv_take_device_error(void *stream);
int lns8_take_device_error(void *stream);
int lmhead_take_device_error(void *stream);

}  // namespace tgi
