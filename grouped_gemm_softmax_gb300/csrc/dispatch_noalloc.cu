// dispatch_noalloc.cu -- moe_dispatch_noalloc: the dispatch step for callers
// that cannot hand the library a device workspace. The dispatch kernels need a
// little scratch (per-chunk, per-expert row bases); here it lives in a fixed
// array in this library's own device memory instead of in caller memory, so
// the call allocates nothing and needs no workspace argument.
#include <mutex>

#include "../../include/moe.h"
#include "kernels.cuh"

namespace {

// (chunk, expert) cells of scratch: 16 KiB, plus 256 B of status words.
constexpr long kNoAllocCells = 4096;
constexpr int kNoAllocStatusWords = 64;

// One copy per GPU that loads this library, kept until the process exits.
// Host code must not use this name as an address (it is a host-side stand-in):
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocCells + kNoAllocStatusWords];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int32_t *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
cudaError_t scratch_on_current_device(int32_t **out)
{
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_addr[dev] = static_cast<int32_t *>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status_t moe_dispatch_noalloc(const moe_shape_t *shape, const moe_bf16_t *x,
                                             const int32_t *topk_idx, int32_t *expert_counts,
                                             int32_t *expert_offsets, int32_t *row_of_slot,
                                             int32_t *slot_of_row, moe_bf16_t *x_perm,
                                             moe_stream_t stream)
{
    // shape validation (same rules and codes as every other entry point)
    size_t off = 0, bytes = 0;
    moe_status_t st = moe_workspace_region(shape, MOE_WS_STATUS, &off, &bytes);
    if (st != MOE_OK) return st;
    if (!expert_counts || !expert_offsets) return MOE_ERR_INVALID_ARG;
    if (shape->T > 0 && (!x || !topk_idx || !row_of_slot || !slot_of_row || !x_perm))
        return MOE_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm)) ||
        (reinterpret_cast<uintptr_t>(expert_counts) & 3u) ||
        (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) ||
        (reinterpret_cast<uintptr_t>(topk_idx) & 3u) || (reinterpret_cast<uintptr_t>(row_of_slot) & 3u) ||
        (reinterpret_cast<uintptr_t>(slot_of_row) & 3u))
        return MOE_ERR_INVALID_ARG;

    // the same chunking as moe_dispatch; it must fit the fixed scratch
    const int chunk_tokens = moe::dispatch_chunk_tokens(shape->T, shape->E);
    const long nchunks = shape->T == 0 ? 0 : (shape->T + chunk_tokens - 1) / chunk_tokens;
    if (nchunks * shape->E > kNoAllocCells) return MOE_ERR_UNSUPPORTED;

    int32_t *scratch = nullptr;
    if (scratch_on_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned *status = reinterpret_cast<unsigned *>(scratch + kNoAllocCells);
    // The status words keep an earlier call's record: clear them. The cells
    // need no clearing (every cell a call reads was written by that call).
    if (shape->T > 0 && cudaMemsetAsync(status, 0, 4 * sizeof(unsigned), s) != cudaSuccess)
        return MOE_ERR_CUDA;

    moe::DispatchArgs a{};
    a.x = x;
    a.topk_idx = topk_idx;
    a.counts = expert_counts;
    a.offsets = expert_offsets;
    a.row_of_slot = row_of_slot;
    a.slot_of_row = slot_of_row;
    a.x_perm = x_perm;
    a.chunk_base = scratch;
    a.status = status;
    a.zero_words = nullptr;
    a.zero_count = 0;
    a.T = shape->T;
    a.d = shape->d;
    a.E = shape->E;
    a.k = shape->top_k;
    a.chunk_tokens = chunk_tokens;
    return moe::launch_dispatch(a, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
