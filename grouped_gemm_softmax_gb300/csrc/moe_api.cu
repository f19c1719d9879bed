// moe_api.cu -- the extern "C" entry points declared in include/moe.h:
// argument validation, workspace layout, tensor-map set-up and the launch
// sequence of one MoE-layer forward on a caller stream.
#include <atomic>
#include <mutex>

#include "../../include/moe.h"
#include "kernels.cuh"

namespace moe {

EncodeTiledFn encode_tiled_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int device_sm_count()
{
    static std::atomic<int> cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace moe

namespace {

using moe::kMaxExperts;
using moe::kMaxSegments;
using moe::kMaxTopK;

struct Layout {
    size_t off[MOE_WS_NUM_REGIONS];
    size_t bytes[MOE_WS_NUM_REGIONS];
    size_t total;
    long max_rows;
    int chunk_tokens;
};

constexpr size_t kAlign = 1024;
// moe_route_filtered's scratch: the status word, then route_tc.cu's scratch
constexpr size_t kRouteStatusBytes = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_shape(const moe_shape_t *s)
{
    if (s == nullptr) return MOE_ERR_INVALID_ARG;
    if (s->T < 0 || s->d < 8 || s->ffn < 8 || s->E < 1 || s->top_k < 1 || s->num_segments < 1)
        return MOE_ERR_INVALID_ARG;
    if (s->d % 8 != 0 || s->ffn % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (s->top_k > s->E) return MOE_ERR_INVALID_ARG;
    if (s->T % s->num_segments != 0) return MOE_ERR_INVALID_ARG;
    if (s->E > kMaxExperts || s->top_k > kMaxTopK || s->num_segments > kMaxSegments)
        return MOE_ERR_UNSUPPORTED;
    const long long R = static_cast<long long>(s->T) * s->top_k;
    const long long w = s->d > s->ffn ? s->d : s->ffn;
    if (R >= (1ll << 31) || R * w >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

Layout make_layout(const moe_shape_t *s, const moe_tuning_t *t = nullptr)
{
    Layout L{};
    const size_t T = s->T, d = s->d, E = s->E, k = s->top_k, F = s->ffn;
    const size_t R = T * k;
    L.chunk_tokens = moe::dispatch_chunk_tokens(s->T, s->E);
    const size_t chunks = T == 0 ? 1 : (T + L.chunk_tokens - 1) / L.chunk_tokens;
    L.max_rows = moe::ffn_max_rows(static_cast<long>(R), s->E);
    const size_t p2max = (d + 63) / 64;  // widest flag grid: Linear-2 tiles of 64 columns
    L.bytes[MOE_WS_STATUS] = 16;
    L.bytes[MOE_WS_TOPK_IDX] = R * 4;
    L.bytes[MOE_WS_TOPK_GATE] = R * 4;
    L.bytes[MOE_WS_COUNTS] = E * 4;
    L.bytes[MOE_WS_OFFSETS] = (E + 1) * 4;
    L.bytes[MOE_WS_ROW_OF_SLOT] = R * 4;
    L.bytes[MOE_WS_SLOT_OF_ROW] = R * 4;
    L.bytes[MOE_WS_X_PERM] = R * d * 2;
    const size_t ring = t ? static_cast<size_t>(t->h_ring_rows) : 0;
    L.bytes[MOE_WS_H] = ring ? ring * 256 * F * 2 : R * F * 2;
    L.bytes[MOE_WS_Y_PERM] = R * d * 2;
    L.bytes[MOE_WS_CHUNK_BASE] = chunks * E * 4;
    // Linear-1 then Linear-2 counts, then the grouped GEMM's tile ticket
    L.bytes[MOE_WS_L1_DONE] = (2 * static_cast<size_t>(L.max_rows) + 4) * 4;
    L.bytes[MOE_WS_L2_FLAGS] = static_cast<size_t>(L.max_rows) * p2max * 4;
    // h last: the other regions keep their offsets whatever h's size
    size_t off = 0;
    for (int i = 0; i < MOE_WS_NUM_REGIONS; ++i) {
        if (i == MOE_WS_H) continue;
        L.off[i] = off;
        off = align_up(off + L.bytes[i]);
    }
    L.off[MOE_WS_H] = off;
    L.total = align_up(off + L.bytes[MOE_WS_H]);
    return L;
}

template <typename T>
T *region(void *ws, const Layout &L, int r)
{
    return reinterpret_cast<T *>(static_cast<char *>(ws) + L.off[r]);
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

std::atomic<uint32_t> g_epoch{0};
uint32_t next_epoch()
{
    uint32_t e = ++g_epoch;
    if (e == 0) e = ++g_epoch;
    return e;
}

// detail words of the last device failure read by this thread
thread_local uint32_t g_detail[3] = {0, 0, 0};

moe_status_t check_tuning(const moe_tuning_t *t)
{
    if (t == nullptr) return MOE_OK;
    if (t->schedule != MOE_SCHEDULE_INTERLEAVED && t->schedule != MOE_SCHEDULE_EXPERT_WAVE)
        return MOE_ERR_INVALID_ARG;
    if (t->lead_rows < 0 || t->num_ctas < 0) return MOE_ERR_INVALID_ARG;
    if (t->l2_block_n != 0 && (t->l2_block_n < 64 || t->l2_block_n > 256 || t->l2_block_n % 64))
        return MOE_ERR_INVALID_ARG;
    if (t->group_rows < 0 || t->cta_group < 0 || t->cta_group > 2) return MOE_ERR_INVALID_ARG;
    if (t->wait_limit_us < 0 || t->unmet_dependency < 0 || t->unmet_dependency > 1)
        return MOE_ERR_INVALID_ARG;
    if (t->tile_trace && (t->tile_trace_cap <= 0 || (reinterpret_cast<uintptr_t>(t->tile_trace) & 7u)))
        return MOE_ERR_INVALID_ARG;
    if (t->orientation < 0 || t->orientation > 2) return MOE_ERR_INVALID_ARG;
    if (t->trace && (reinterpret_cast<uintptr_t>(t->trace) & 7u)) return MOE_ERR_INVALID_ARG;
    if (t->h_ring_rows < 0 || (t->h_ring_rows > 0 && t->schedule != MOE_SCHEDULE_INTERLEAVED))
        return MOE_ERR_INVALID_ARG;
    if (t->fused_combine < 0 || t->fused_combine > 1) return MOE_ERR_INVALID_ARG;
    if (t->row_order < 0 || t->row_order > 2) return MOE_ERR_INVALID_ARG;
    if (t->router < 0 || t->router > 2) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status_t enqueue_ffn(const moe_shape_t *s, const moe_tuning_t *tune, const Layout &L,
                         const moe_bf16_t *x_perm, const int32_t *offsets, const moe_bf16_t *W1,
                         const moe_bf16_t *W3, const moe_bf16_t *W2, moe_bf16_t *y_perm, void *ws,
                         bool counters_zeroed, cudaStream_t stream,
                         const moe::CombineArgs *fused = nullptr)
{
    moe::FfnArgs a{};
    if (fused != nullptr) {
        a.gate = fused->gate;
        a.row_of_slot = fused->row_of_slot;
        a.slot_of_row = region<int32_t>(ws, L, MOE_WS_SLOT_OF_ROW);
        for (int i = 0; i < kMaxSegments; ++i) a.seg[i] = fused->seg[i];
        a.T = fused->T;
        a.k = fused->k;
        a.S = fused->S;
    }
    a.x_perm = x_perm;
    a.offsets = offsets;
    a.w1 = W1;
    a.w3 = W3;
    a.w2 = W2;
    a.h = region<uint16_t>(ws, L, MOE_WS_H);
    a.y = y_perm;
    a.l1_done = region<unsigned>(ws, L, MOE_WS_L1_DONE);
    a.l2_flags = region<unsigned>(ws, L, MOE_WS_L2_FLAGS);
    a.status = region<unsigned>(ws, L, MOE_WS_STATUS);
    a.max_rows = L.max_rows;
    a.R = s->T * s->top_k;
    a.d = s->d;
    a.F = s->ffn;
    a.E = s->E;
    a.schedule = tune ? tune->schedule : MOE_SCHEDULE_INTERLEAVED;
    a.lead = tune ? tune->lead_rows : 0;
    a.num_ctas = tune ? tune->num_ctas : 0;
    a.l2_block_n = tune ? tune->l2_block_n : 0;
    a.group_rows = tune ? tune->group_rows : 0;
    a.cta_group = tune ? tune->cta_group : 0;
    a.orientation = tune ? tune->orientation : 0;
    a.h_ring_rows = tune ? tune->h_ring_rows : 0;
    a.row_order = tune ? tune->row_order : 0;
    a.wait_limit_us = tune ? tune->wait_limit_us : 0;
    a.unmet_dependency = tune ? tune->unmet_dependency : 0;
    a.trace = tune ? static_cast<unsigned long long *>(tune->trace) : nullptr;
    a.tile_trace = tune ? static_cast<unsigned long long *>(tune->tile_trace) : nullptr;
    a.tile_trace_cap = tune ? tune->tile_trace_cap : 0;
    a.counters_zeroed = counters_zeroed;
    a.epoch = next_epoch();
    if (moe::encode_tiled_fn() == nullptr) return MOE_ERR_CUDA;
    const cudaError_t err = moe::launch_ffn(a, stream);
    // a ring too small for the raster group is a configuration the caller chose
    if (err == cudaErrorInvalidConfiguration && a.h_ring_rows > 0) return MOE_ERR_INVALID_ARG;
    return cuda_status(err);
}

}  // namespace

extern "C" {

const char *moe_status_string(moe_status_t st)
{
    switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

size_t moe_workspace_bytes(const moe_shape_t *shape)
{
    if (check_shape(shape) != MOE_OK) return 0;
    return make_layout(shape).total;
}

size_t moe_workspace_bytes_tuned(const moe_shape_t *shape, const moe_tuning_t *tuning)
{
    if (check_shape(shape) != MOE_OK || check_tuning(tuning) != MOE_OK) return 0;
    return make_layout(shape, tuning).total;
}

moe_status_t moe_workspace_region_tuned(const moe_shape_t *shape, const moe_tuning_t *tuning,
                                        int r, size_t *offset, size_t *bytes)
{
    moe_status_t st = check_shape(shape);
    if (st != MOE_OK) return st;
    if ((st = check_tuning(tuning)) != MOE_OK) return st;
    if (r < 0 || r >= MOE_WS_NUM_REGIONS || offset == nullptr || bytes == nullptr)
        return MOE_ERR_INVALID_ARG;
    const Layout L = make_layout(shape, tuning);
    *offset = L.off[r];
    *bytes = L.bytes[r];
    return MOE_OK;
}

moe_status_t moe_workspace_region(const moe_shape_t *shape, int r, size_t *offset, size_t *bytes)
{
    const moe_status_t st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (r < 0 || r >= MOE_WS_NUM_REGIONS || offset == nullptr || bytes == nullptr)
        return MOE_ERR_INVALID_ARG;
    const Layout L = make_layout(shape);
    *offset = L.off[r];
    *bytes = L.bytes[r];
    return MOE_OK;
}

moe_status_t moe_route(const moe_shape_t *shape, const moe_bf16_t *x, const moe_bf16_t *w_router,
                       const float *expert_bias, int32_t *topk_idx, float *topk_gate,
                       moe_stream_t stream)
{
    moe_status_t st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (shape->T == 0) return MOE_OK;
    if (!x || !w_router || !topk_idx || !topk_gate) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_router) || !aligned16(topk_idx) || !aligned16(topk_gate) ||
        (expert_bias && (reinterpret_cast<uintptr_t>(expert_bias) & 3u)))
        return MOE_ERR_INVALID_ARG;
    moe::RouteArgs a{x, w_router, expert_bias, topk_idx, topk_gate, shape->T, shape->d, shape->E,
                     shape->top_k};
    return cuda_status(moe::launch_route(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_route_scratch_bytes(const moe_shape_t *shape)
{
    if (check_shape(shape) != MOE_OK) return 0;
    return kRouteStatusBytes + moe::route_fast_scratch_bytes(shape->T, shape->E);
}

moe_status_t moe_route_filtered(const moe_shape_t *shape, const moe_bf16_t *x, const moe_bf16_t *w_router,
                                const float *expert_bias, int32_t *topk_idx, float *topk_gate, void *scratch,
                                size_t scratch_bytes, moe_stream_t stream)
{
    moe_status_t st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (shape->T == 0) return MOE_OK;
    if (!x || !w_router || !topk_idx || !topk_gate || !scratch) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_router) || !aligned16(topk_idx) || !aligned16(topk_gate) ||
        (reinterpret_cast<uintptr_t>(scratch) & 255u) ||
        (expert_bias && (reinterpret_cast<uintptr_t>(expert_bias) & 3u)))
        return MOE_ERR_INVALID_ARG;
    if (!moe::route_fast_supported(shape->T, shape->d, shape->E, shape->top_k)) return MOE_ERR_UNSUPPORTED;
    if (scratch_bytes < moe_route_scratch_bytes(shape)) return MOE_ERR_WORKSPACE;
    if (moe::encode_tiled_fn() == nullptr) return MOE_ERR_CUDA;
    moe::RouteArgs a{x, w_router, expert_bias, topk_idx, topk_gate, shape->T, shape->d, shape->E,
                     shape->top_k};
    char *base = static_cast<char *>(scratch);
    return cuda_status(moe::launch_route_fast(a, reinterpret_cast<unsigned *>(base), base + kRouteStatusBytes,
                                              scratch_bytes - kRouteStatusBytes,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_dispatch(const moe_shape_t *shape, const moe_bf16_t *x, const int32_t *topk_idx,
                          int32_t *expert_counts, int32_t *expert_offsets, int32_t *row_of_slot,
                          int32_t *slot_of_row, moe_bf16_t *x_perm, void *ws, size_t ws_bytes,
                          moe_stream_t stream)
{
    moe_status_t st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (!expert_counts || !expert_offsets || !ws) return MOE_ERR_INVALID_ARG;
    const Layout L = make_layout(shape);
    if (ws_bytes < L.off[MOE_WS_H]) return MOE_ERR_WORKSPACE;  // every region it uses lies before h
    if (shape->T > 0 && (!x || !topk_idx || !row_of_slot || !slot_of_row || !x_perm))
        return MOE_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm)) || !aligned16(ws) ||
        (reinterpret_cast<uintptr_t>(expert_counts) & 3u) ||
        (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) ||
        (reinterpret_cast<uintptr_t>(topk_idx) & 3u) || (reinterpret_cast<uintptr_t>(row_of_slot) & 3u) ||
        (reinterpret_cast<uintptr_t>(slot_of_row) & 3u))
        return MOE_ERR_INVALID_ARG;
    moe::DispatchArgs a{};
    a.x = x;
    a.topk_idx = topk_idx;
    a.counts = expert_counts;
    a.offsets = expert_offsets;
    a.row_of_slot = row_of_slot;
    a.slot_of_row = slot_of_row;
    a.x_perm = x_perm;
    a.chunk_base = region<int32_t>(ws, L, MOE_WS_CHUNK_BASE);
    a.status = region<unsigned>(ws, L, MOE_WS_STATUS);
    a.zero_words = nullptr;
    a.zero_count = 0;
    a.T = shape->T;
    a.d = shape->d;
    a.E = shape->E;
    a.k = shape->top_k;
    a.chunk_tokens = L.chunk_tokens;
    return cuda_status(moe::launch_dispatch(a, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expert_ffn_tuned(const moe_shape_t *shape, const moe_tuning_t *tuning,
                                  const moe_bf16_t *x_perm, const int32_t *expert_offsets,
                                  const moe_bf16_t *W1, const moe_bf16_t *W3, const moe_bf16_t *W2,
                                  moe_bf16_t *y_perm, void *ws, size_t ws_bytes,
                                  moe_stream_t stream)
{
    moe_status_t st = check_shape(shape);
    if (st != MOE_OK) return st;
    if ((st = check_tuning(tuning)) != MOE_OK) return st;
    if (!ws) return MOE_ERR_INVALID_ARG;
    const Layout L = make_layout(shape, tuning);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (shape->T == 0) return MOE_OK;
    if (!x_perm || !expert_offsets || !W1 || !W3 || !W2 || !y_perm) return MOE_ERR_INVALID_ARG;
    if (tuning && tuning->fused_combine) return MOE_ERR_INVALID_ARG;  // needs the layer's routing
    if (!aligned16(x_perm) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) ||
        !aligned16(y_perm) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(expert_offsets) & 3u))
        return MOE_ERR_INVALID_ARG;
    return enqueue_ffn(shape, tuning, L, x_perm, expert_offsets, W1, W3, W2, y_perm, ws, false,
                       reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_expert_ffn(const moe_shape_t *shape, const moe_bf16_t *x_perm,
                            const int32_t *expert_offsets, const moe_bf16_t *W1,
                            const moe_bf16_t *W3, const moe_bf16_t *W2, moe_bf16_t *y_perm,
                            void *ws, size_t ws_bytes, moe_stream_t stream)
{
    return moe_expert_ffn_tuned(shape, nullptr, x_perm, expert_offsets, W1, W3, W2, y_perm, ws,
                                ws_bytes, stream);
}

moe_status_t moe_combine(const moe_shape_t *shape, const moe_bf16_t *y_perm,
                         const float *topk_gate, const int32_t *row_of_slot,
                         moe_bf16_t *const *out_segments, moe_stream_t stream)
{
    moe_status_t st = check_shape(shape);
    if (st != MOE_OK) return st;
    if (shape->T == 0) return MOE_OK;
    if (!y_perm || !topk_gate || !row_of_slot || !out_segments) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y_perm) || (reinterpret_cast<uintptr_t>(topk_gate) & 3u) ||
        (reinterpret_cast<uintptr_t>(row_of_slot) & 3u))
        return MOE_ERR_INVALID_ARG;
    moe::CombineArgs a{};
    for (int i = 0; i < shape->num_segments; ++i) {
        if (!out_segments[i] || !aligned16(out_segments[i])) return MOE_ERR_INVALID_ARG;
        a.seg[i] = out_segments[i];
    }
    a.y = y_perm;
    a.gate = topk_gate;
    a.row_of_slot = row_of_slot;
    a.T = shape->T;
    a.d = shape->d;
    a.k = shape->top_k;
    a.S = shape->num_segments;
    return cuda_status(moe::launch_combine(a, reinterpret_cast<cudaStream_t>(stream)));
}

// Whether the layer routes by filter then verify: the tuning's choice, else
// for more than 128 experts (where the direct kernels are slowest per token);
// only where route_tc.cu supports the shape and the X_PERM region holds its
// scratch.
bool filter_verify_route(const moe_shape_t *s, const moe_tuning_t *t, const Layout &L)
{
    const int mode = t ? t->router : MOE_ROUTER_DEFAULT;
    if (mode == MOE_ROUTER_DIRECT) return false;
    if (mode == MOE_ROUTER_DEFAULT && s->E <= 128) return false;
    return moe::route_fast_supported(s->T, s->d, s->E, s->top_k) &&
           moe::route_fast_scratch_bytes(s->T, s->E) <= L.bytes[MOE_WS_X_PERM];
}

moe_status_t moe_layer_forward_ex(const moe_shape_t *shape, const moe_tuning_t *tuning,
                                  const moe_bf16_t *x, const moe_bf16_t *w_router,
                                  const float *expert_bias, const moe_bf16_t *W1,
                                  const moe_bf16_t *W3, const moe_bf16_t *W2,
                                  moe_bf16_t *const *out_segments, void *ws, size_t ws_bytes,
                                  moe_stream_t stream, void *const *stage_events)
{
    moe_status_t st = check_shape(shape);
    if (st != MOE_OK) return st;
    if ((st = check_tuning(tuning)) != MOE_OK) return st;
    if (!ws) return MOE_ERR_INVALID_ARG;
    const Layout L = make_layout(shape, tuning);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (shape->T == 0) return MOE_OK;
    if (!x || !w_router || !W1 || !W3 || !W2 || !out_segments) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_router) || !aligned16(W1) || !aligned16(W3) ||
        !aligned16(W2) || !aligned16(ws) ||
        (expert_bias && (reinterpret_cast<uintptr_t>(expert_bias) & 3u)))
        return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < shape->num_segments; ++i)
        if (!out_segments[i] || !aligned16(out_segments[i])) return MOE_ERR_INVALID_ARG;
    if (moe::encode_tiled_fn() == nullptr) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    auto mark = [&](int i) -> bool {
        if (stage_events == nullptr) return true;
        return cudaEventRecord(reinterpret_cast<cudaEvent_t>(stage_events[i]), s) == cudaSuccess;
    };
    if (stage_events)
        for (int i = 0; i < 5; ++i)
            if (!stage_events[i]) return MOE_ERR_INVALID_ARG;

    int32_t *idx = region<int32_t>(ws, L, MOE_WS_TOPK_IDX);
    float *gate = region<float>(ws, L, MOE_WS_TOPK_GATE);
    moe::RouteArgs ra{x, w_router, expert_bias, idx, gate, shape->T, shape->d, shape->E,
                      shape->top_k};
    if (!mark(0)) return MOE_ERR_CUDA;
    cudaError_t err = filter_verify_route(shape, tuning, L)
                          ? moe::launch_route_fast(ra, region<unsigned>(ws, L, MOE_WS_STATUS),
                                                   region<void>(ws, L, MOE_WS_X_PERM),
                                                   L.bytes[MOE_WS_X_PERM], s)
                          : moe::launch_route(ra, s);
    if (err != cudaSuccess || !mark(1)) return MOE_ERR_CUDA;

    moe::DispatchArgs da{};
    da.x = x;
    da.topk_idx = idx;
    da.counts = region<int32_t>(ws, L, MOE_WS_COUNTS);
    da.offsets = region<int32_t>(ws, L, MOE_WS_OFFSETS);
    da.row_of_slot = region<int32_t>(ws, L, MOE_WS_ROW_OF_SLOT);
    da.slot_of_row = region<int32_t>(ws, L, MOE_WS_SLOT_OF_ROW);
    da.x_perm = region<uint16_t>(ws, L, MOE_WS_X_PERM);
    da.chunk_base = region<int32_t>(ws, L, MOE_WS_CHUNK_BASE);
    da.status = region<unsigned>(ws, L, MOE_WS_STATUS);
    da.zero_words = region<unsigned>(ws, L, MOE_WS_L1_DONE);
    da.zero_count = 2 * L.max_rows + 1;  // Linear-1 and Linear-2 row counters, tile ticket
    da.T = shape->T;
    da.d = shape->d;
    da.E = shape->E;
    da.k = shape->top_k;
    da.chunk_tokens = L.chunk_tokens;
    err = moe::launch_dispatch(da, s);
    if (err != cudaSuccess || !mark(2)) return MOE_ERR_CUDA;

    moe::CombineArgs ca{};
    for (int i = 0; i < shape->num_segments; ++i) ca.seg[i] = out_segments[i];
    ca.y = region<uint16_t>(ws, L, MOE_WS_Y_PERM);
    ca.gate = gate;
    ca.row_of_slot = da.row_of_slot;
    ca.T = shape->T;
    ca.d = shape->d;
    ca.k = shape->top_k;
    ca.S = shape->num_segments;
    ca.early_maps = true;  // the combine follows the grouped GEMM
    const bool fused = tuning && tuning->fused_combine;
    st = enqueue_ffn(shape, tuning, L, da.x_perm, da.offsets, W1, W3, W2,
                     region<uint16_t>(ws, L, MOE_WS_Y_PERM), ws, true, s, fused ? &ca : nullptr);
    if (st != MOE_OK) return st;
    if (!mark(3)) return MOE_ERR_CUDA;
    if (!fused) {
        err = moe::launch_combine(ca, s);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (!mark(4)) return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_layer_kernel_launches(const moe_shape_t *shape, const moe_tuning_t *tuning)
{
    if (check_shape(shape) != MOE_OK || check_tuning(tuning) != MOE_OK) return 0;
    const bool fused = tuning && tuning->fused_combine;
    const int route = filter_verify_route(shape, tuning, make_layout(shape, tuning)) ? 4 : 1;
    // route; count, scan, rank, copy; grouped GEMM; combine
    return route + 4 + 1 + (fused ? 0 : 1);
}

moe_status_t moe_layer_forward_tuned(const moe_shape_t *shape, const moe_tuning_t *tuning,
                                     const moe_bf16_t *x, const moe_bf16_t *w_router,
                                     const float *expert_bias, const moe_bf16_t *W1,
                                     const moe_bf16_t *W3, const moe_bf16_t *W2,
                                     moe_bf16_t *const *out_segments, void *ws, size_t ws_bytes,
                                     moe_stream_t stream)
{
    return moe_layer_forward_ex(shape, tuning, x, w_router, expert_bias, W1, W3, W2, out_segments,
                                ws, ws_bytes, stream, nullptr);
}

moe_status_t moe_layer_forward(const moe_shape_t *shape, const moe_bf16_t *x,
                               const moe_bf16_t *w_router, const float *expert_bias,
                               const moe_bf16_t *W1, const moe_bf16_t *W3, const moe_bf16_t *W2,
                               moe_bf16_t *const *out_segments, void *ws, size_t ws_bytes,
                               moe_stream_t stream)
{
    return moe_layer_forward_tuned(shape, nullptr, x, w_router, expert_bias, W1, W3, W2,
                                   out_segments, ws, ws_bytes, stream);
}

moe_status_t moe_last_device_status(void *ws, moe_stream_t stream)
{
    if (!ws) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t host[4] = {0, 0, 0, 0};
    if (cudaMemcpyAsync(host, ws, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (host[0] == 0) return MOE_OK;
    g_detail[0] = host[1];
    g_detail[1] = host[2];
    g_detail[2] = host[3];
    if (cudaMemsetAsync(ws, 0, sizeof(host), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    switch (host[0]) {
    case MOE_ERR_TIMEOUT: return MOE_ERR_TIMEOUT;
    case MOE_ERR_INVALID_ARG: return MOE_ERR_INVALID_ARG;
    default: return MOE_ERR_CUDA;
    }
}

void moe_last_device_detail(uint32_t *where, uint32_t *block, uint32_t *detail)
{
    if (where) *where = g_detail[0];
    if (block) *block = g_detail[1];
    if (detail) *detail = g_detail[2];
}

}  // extern "C"
