// kernels.cuh -- host-side launch interface between the C ABI (moe_api.cu) and
// the kernels (route.cu, dispatch.cu, grouped_gemm.cu, combine.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

namespace moe {

// Programmatic dependent launch: every kernel of the layer is launched with
// programmatic stream serialization, calls pdl_wait() before it reads anything
// an earlier kernel on the stream wrote (it returns once those grids have
// completed and their writes are visible) and pdl_trigger() to let the next
// kernel's blocks be scheduled early. Both are no-ops without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kMaxSegments = 64;

struct RouteArgs {
    const uint16_t *x;       // [T,d] bf16
    const uint16_t *wr;      // [E,d] bf16
    const float *bias;       // [E] or null
    int32_t *topk_idx;       // [T,k]
    float *topk_gate;        // [T,k]
    int T, d, E, k;
};
cudaError_t launch_route(const RouteArgs &a, cudaStream_t s);

// Filter-then-verify routing (route_tc.cu): the same results as launch_route
// from four launches that sum exactly only the candidate experts. Needs
// route_fast_scratch_bytes(T, E) bytes of 256-byte aligned device scratch and
// the layer's status words (a bounded wait that runs out is recorded there).
size_t route_fast_scratch_bytes(long T, int E);
bool route_fast_supported(long T, int d, int E, int k);
cudaError_t launch_route_fast(const RouteArgs &a, unsigned *status, void *scratch, size_t scratch_bytes,
                              cudaStream_t s);

struct DispatchArgs {
    const uint16_t *x;       // [T,d]
    const int32_t *topk_idx; // [T,k]
    int32_t *counts;         // [E]
    int32_t *offsets;        // [E+1]
    int32_t *row_of_slot;    // [R]
    int32_t *slot_of_row;    // [R]
    uint16_t *x_perm;        // [R,d]
    int32_t *chunk_base;     // [nchunks,E] scratch
    unsigned *status;        // device status words (an expert id outside [0,E) is reported here)
    unsigned *zero_words;    // optional: words to clear for the grouped GEMM (may be null)
    long zero_count;
    int T, d, E, k;
    int chunk_tokens;
};
int dispatch_chunk_tokens(int T, int E);
cudaError_t launch_dispatch(const DispatchArgs &a, cudaStream_t s);

struct FfnArgs {
    const uint16_t *x_perm;  // [R,d]
    const int32_t *offsets;  // [E+1]
    const uint16_t *w1, *w3; // [E,F,d]
    const uint16_t *w2;      // [E,d,F]
    uint16_t *h;             // [R,F]
    uint16_t *y;             // [R,d]
    unsigned *l1_done;       // [2 * max_rows]: Linear-1 counters, then Linear-2 counters
    unsigned *l2_flags;      // [max_rows * P2]
    unsigned *status;        // 4 words
    long max_rows;
    int R, d, F, E;
    int schedule, lead, num_ctas, l2_block_n, group_rows, cta_group;
    int orientation;  // 0 = choose, 1 = tokens on the MMA's M side, 2 = on its N side
    int h_ring_rows;  // h ring slots in scheduler rows (0 = h holds every row)
    int row_order;    // 0 = default, 1 = expert order, 2 = mixed (single-row experts spread out)
    // fused combine (consumer warps in the GEMM kernel); gate == nullptr = off
    const float *gate;            // [T,k]
    const int32_t *row_of_slot;   // [R]
    const int32_t *slot_of_row;   // [R]
    uint16_t *seg[kMaxSegments];  // S segments of [T/S, d]
    int T, k, S;
    int wait_limit_us, unmet_dependency;
    unsigned long long *trace;  // optional per-CTA counters (16 per CTA)
    unsigned long long *tile_trace;  // optional per-tile timeline (8 words per tile)
    int tile_trace_cap;              // tiles recorded per CTA
    bool counters_zeroed;    // l1_done already cleared by an earlier kernel on the stream
    unsigned epoch;
};
int ffn_l2_block_n(int d, int requested);
long ffn_max_rows(long R, int E);
cudaError_t launch_ffn(const FfnArgs &a, cudaStream_t s);

struct CombineArgs {
    const uint16_t *y;        // [R,d]
    const float *gate;        // [T,k]
    const int32_t *row_of_slot;
    uint16_t *seg[kMaxSegments];
    int T, d, k, S;
    // the gates and the row map were complete before the kernel launched just
    // ahead of the combine passed its own wait (the layer's grouped GEMM), so
    // the combine may read them before its wait
    bool early_maps;
};
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s);

// driver entry point for tensor-map encoding, resolved once through the runtime
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();
int device_sm_count();

// Per-device one-time setup of a launch (kernel attributes, occupancy): the
// first caller on a device runs init and every later caller on that device
// gets its result. Thread safe; devices past kOnceDevices run init on every
// call. Each distinct `Tag` type (one per kernel instantiation) has its own
// state.
constexpr int kOnceDevices = 64;
template <typename Tag, typename Init>
cudaError_t once_per_device(Init &&init)
{
    static std::once_flag flags[kOnceDevices];
    static cudaError_t results[kOnceDevices];
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kOnceDevices) return init(dev);
    std::call_once(flags[dev], [&] { results[dev] = init(dev); });
    return results[dev];
}

}  // namespace moe
