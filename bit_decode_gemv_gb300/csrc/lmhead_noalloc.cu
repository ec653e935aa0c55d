// lmhead_noalloc.cu -- the lm_head call for callers that cannot allocate device
// memory.
//
// tg_lmhead_argmax_topk needs a device workspace (per-row stage-1 sums,
// per-warp bounds, the candidate list). Some callers cannot provide one: a
// plugin inside a host framework that hands out device memory only through its
// own allocator, a serving process whose device memory is already fully
// reserved by a cache pool, or a latency-critical decode loop that is not
// allowed to call cudaMalloc because it can block on the device. For them the
// library keeps one fixed scratch array in device memory of its own and runs
// the same lm_head kernels on it. Every GPU that loads this code holds the
// array until the process exits.
//
// The array is shared by every call in the process on a given device and keeps
// the last call's contents. Each lm_head call clears the counters and
// histograms it relies on at its start and writes everything else it reads
// before reading it, so nothing has to be cleared between calls. Two calls
// whose work overlaps on the GPU (different streams, or different host threads
// without ordering) use the same memory and race: the caller must order them.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "tg.h"
#include "tg_internal.h"

namespace {

// The fixed scratch. Host code must not use this name as an address: on the
// host it is only a stand-in symbol; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char tg_noalloc_scratch[TG_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached; NULL on failure. The cache
// lives as long as the process: after cudaDeviceReset the array's address on
// that device is no longer valid, so the call must not be used on a device
// that was reset (tg.h says so).
void *scratch_for_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, tg_noalloc_scratch) != cudaSuccess || !ptr)
            return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int tg_lmhead_argmax_topk_noalloc(const tg_layout *L, const void *w, const int8_t *x,
                                             int32_t k, int64_t *logits, int32_t *argmax,
                                             int32_t *ids, int64_t *scores, int32_t *ncand,
                                             void *stream)
{
    // the same checks, in the same order, as the workspace-taking call; only then
    // whether the problem's workspace fits the fixed array
    const int bad = tgi::lmhead_check_args(L, w, x, k, logits, argmax, ids, scores, ncand);
    if (bad != TG_OK)
        return bad;
    if (tg_lmhead_workspace_bytes(L, k) > (size_t)TG_NOALLOC_SCRATCH_BYTES)
        return TG_ERR_WORKSPACE;
    void *ws = scratch_for_current_device();
    if (!ws)
        return TG_ERR_CUDA;
    return tg_lmhead_argmax_topk(L, w, x, k, logits, argmax, ids, scores, ncand, ws,
                                 (size_t)TG_NOALLOC_SCRATCH_BYTES, stream);
}
