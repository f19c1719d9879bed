/*
 * moe.h -- C ABI of libmoe_gb300: the forward pass of one Mixture-of-Experts
 * layer on one GB300 GPU (sm_103a), as hand-written CUDA kernels.
 *
 * The forward pass follows the five steps of Cui et al., "Fine-grained
 * Computation-Communication Overlap via Tile-level Signaling and Scheduling
 * for MoE", section 2.1: routing (top-k experts and gate weights), dispatch of
 * each token copy to its expert, expert computation, return, and the
 * gate-weighted sum. Each expert is the two-layer SwiGLU network of Xian et
 * al., "X-Stage: An Overlooked Pipeline Stage for Communication-Computation
 * Overlap in DiT Inference", section 2.2 (MegaMoE Execution): Linear-1 to the
 * intermediate width, SwiGLU, Linear-2 back to the hidden width.
 *
 * Conventions shared by every entry point:
 *   - Notation: T tokens, d hidden width, E experts, k = top_k, F = ffn
 *     (SwiGLU intermediate width), R = T*k routed rows, S = num_segments.
 *   - All matrices are dense row-major. bf16 is IEEE bfloat16 passed as its
 *     16-bit pattern (moe_bf16_t); fp32 is IEEE binary32.
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise, must
 *     be 16-byte aligned, and is owned by the caller. The library never
 *     allocates device memory and never synchronises, except
 *     moe_last_device_status. Work is enqueued on the caller's stream
 *     (NULL = the legacy default stream) and returns immediately.
 *   - Shape rules: T >= 0; d, F >= 8 and multiples of 8; 1 <= k <= 8, k <= E;
 *     1 <= E <= 256; 1 <= S <= 64 and T % S == 0; T*k*max(d,F) < 2^40.
 *     Violations return MOE_ERR_INVALID_ARG (bad value or pointer) or
 *     MOE_ERR_UNSUPPORTED (legal but outside the supported range). T == 0 is
 *     a valid empty call that enqueues nothing.
 *   - Synchronous failures are return values. A device-side failure (a bounded
 *     wait that ran out) is written to the status word at the start of the
 *     workspace and read back by moe_last_device_status.
 *   - Inputs must be finite. Calls that share a workspace must not overlap on
 *     the GPU.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16_t;             /* raw bfloat16 bits */
typedef struct CUstream_st *moe_stream_t; /* same type as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_UNSUPPORTED = 2,
    MOE_ERR_WORKSPACE = 3,
    MOE_ERR_CUDA = 4,
    MOE_ERR_TIMEOUT = 5
} moe_status_t;

typedef struct {
    int T;            /* tokens */
    int d;            /* hidden width */
    int E;            /* experts */
    int top_k;        /* experts per token */
    int ffn;          /* SwiGLU intermediate width F */
    int num_segments; /* S owner-aligned output segments, T % S == 0 */
} moe_shape_t;

/* Tile schedule of the grouped GEMM. Both orders compute bit-identical outputs;
 * they differ only in the order tiles run (Xian et al., section 4.2). */
typedef enum {
    MOE_SCHEDULE_INTERLEAVED = 0, /* Linear-2 tiles merged into the Linear-1 stream (Algorithm 1) */
    MOE_SCHEDULE_EXPERT_WAVE = 1  /* per wave of experts: all Linear-1 tiles, then its Linear-2 tiles */
} moe_schedule_t;

/* Operand orientation of the grouped GEMM. Tokens on the M side: each MMA tile
   is 128 (single CTA) or 256 (CTA pair) token rows by a block of weight rows,
   and every expert's last tile is padded to that height. Tokens on the N side:
   each tile is 128 (single CTA) or 256 (CTA pair) weight rows by up to 256
   tokens, the width rounded up to 16 tokens, so an expert pads at most 15
   tokens. The
   default puts tokens on the N side unless d is not a multiple of 256 and the
   experts average 1024 rows or more. Results agree within the rounding of the
   fp32 accumulation order. */
typedef enum {
    MOE_ORIENT_DEFAULT = 0,
    MOE_ORIENT_TOKENS_M = 1,
    MOE_ORIENT_TOKENS_N = 2
} moe_orientation_t;

/* How moe_layer_forward routes (step 1). Both give the same bits as moe_route:
 * DIRECT sums every logit exactly (moe_route's kernels); FILTER_VERIFY computes
 * every logit approximately on the tensor cores, bounds the error of both
 * sums by |x_t| |w_e| (Cauchy-Schwarz), keeps the experts that can still be in
 * the top k and sums exactly only those (tokens with too many candidates fall
 * back to all experts). FILTER_VERIFY runs in four launches and uses the
 * X_PERM region as scratch before the dispatch writes it. */
typedef enum {
    MOE_ROUTER_DEFAULT = 0,       /* FILTER_VERIFY when E > 128, else DIRECT */
    MOE_ROUTER_DIRECT = 1,
    MOE_ROUTER_FILTER_VERIFY = 2
} moe_router_t;

typedef struct {
    int schedule;   /* moe_schedule_t */
    int lead_rows;  /* D: minimum lead of Linear-1 over Linear-2 in scheduler rows; 0 = default;
                       raised to the raster group if smaller (needed for deadlock freedom) */
    int num_ctas;   /* persistent grid size in CTAs (rounded down to whole CTA groups); 0 = as
                       many as are co-resident (one per SM) */
    int l2_block_n; /* Linear-2 tile width (64, 128, 192 or 256) with tokens on the M side;
                       0 = default (ignored with tokens on the N side: 256) */
    int group_rows; /* raster group: an expert's tiles run N-tile-major over groups of this many
                       128-row M-tiles, so each weight tile is reused while hot in L2; 0 = default
                       (16 when T*k/E < 1024, i.e. experts average under 4 rows of 256 tokens,
                       else 32) */
    int cta_group;  /* CTAs per MMA tile: 2 = CTA pairs with 256-row tiles, 1 = single CTAs
                       with 128-row (tokens on M) or 128-weight-row (tokens on N) tiles;
                       0 = default (pairs, except tokens on the M side with T*k/E < 1024) */
    int wait_limit_us;    /* limit of every bounded wait in the grouped GEMM; 0 = 2 s */
    int unmet_dependency; /* failure-detection test only: 1 makes each Linear-2 tile wait for one
                             more finished Linear-1 tile than exists, so the wait runs out and the
                             call reports MOE_ERR_TIMEOUT; must be 0 otherwise */
    void *trace;    /* optional device buffer of num_ctas x 16 uint64 per-CTA counters (wait
                       cycles per role, tile counts, start/end times); NULL = off */
    void *tile_trace;   /* optional per-tile timeline: num_ctas x tile_trace_cap x 8 uint64
                           (SM clock stamps: tile id, producer start and dependency wait,
                           MMA start / last issue / stage-wait cycles, epilogue start / end);
                           NULL = off */
    int tile_trace_cap; /* tiles recorded per CTA (later tiles are not recorded) */
    int orientation;    /* moe_orientation_t: which MMA operand holds the tokens; 0 = default */
    int h_ring_rows;    /* 0 = h holds all R rows; Q > 0 = h is a ring of Q scheduler rows
                           (Xian et al., Algorithm 1, "destination ring slot"): row p lives in
                           slot p mod Q and a Linear-1 tile of row p >= Q waits (bounded)
                           until every Linear-2 tile of row p - Q has finished. Q must be at
                           least 3 * raster group scheduler rows (48 for CTA pairs with the
                           default group of 32 M-tiles, 24 with 16) and the lead is lowered
                           to Q - 2 * group if above it, which keeps the waits deadlock-free;
                           interleaved schedule only (else MOE_ERR_INVALID_ARG). The
                           workspace must then come from moe_workspace_bytes_tuned with the
                           same tuning. */
    int fused_combine;  /* moe_layer_forward_tuned / _ex only (else MOE_ERR_INVALID_ARG): 1 =
                           combine inside the grouped GEMM (Cui et al. section 3.3: consumers
                           poll the per-row Linear-2 completion and write each token to its
                           owner segment as soon as its last expert row is finished); the
                           output bits equal the separate combine's. 0 = separate kernel. */
    int row_order;      /* order of the scheduler rows: 1 = expert order, 2 = mixed (experts with
                           a single row spread evenly among the other experts' rows, so
                           weight-streaming and compute-bound tiles run side by side; taken with
                           the interleaved schedule when both kinds exist and the rows number at
                           most 1024, never with fused_combine), 0 = default (mixed when
                           single-row experts are at least a quarter of the rows, else expert
                           order). Results are bit-identical either way. */
    int router;         /* moe_router_t: how the layer routes; results are bit-identical either
                           way. 0 = default (filter-then-verify for E > 128, else direct) */
} moe_tuning_t;

/* Human-readable name of a status code. Never NULL. */
const char *moe_status_string(moe_status_t status);

/* Bytes of device workspace that moe_layer_forward needs for this shape (a
 * superset of what moe_dispatch and moe_expert_ffn need). 0 for an invalid shape. */
size_t moe_workspace_bytes(const moe_shape_t *shape);

/* The same for a tuning (NULL = defaults): with h_ring_rows = Q > 0 the h
 * region is Q x 256 x F bf16 instead of R x F. The h region is the last in the
 * workspace, so every other region has the same offset in both layouts. */
size_t moe_workspace_bytes_tuned(const moe_shape_t *shape, const moe_tuning_t *tuning);

/* Byte offset and size of one named region inside the workspace (for
 * inspection: routing results, the permuted rows, h, y_perm, flags).
 * region: see MOE_WS_* below. */
enum {
    MOE_WS_STATUS = 0,      /* 4 x u32 device status: code, where, block, detail */
    MOE_WS_TOPK_IDX = 1,    /* [T,k] int32 */
    MOE_WS_TOPK_GATE = 2,   /* [T,k] fp32 */
    MOE_WS_COUNTS = 3,      /* [E] int32 */
    MOE_WS_OFFSETS = 4,     /* [E+1] int32 */
    MOE_WS_ROW_OF_SLOT = 5, /* [R] int32 */
    MOE_WS_SLOT_OF_ROW = 6, /* [R] int32 */
    MOE_WS_X_PERM = 7,      /* [R,d] bf16 */
    MOE_WS_H = 8,           /* [R,F] bf16: SwiGLU activations (a ring of Q x 256 rows with
                               h_ring_rows = Q); placed last in the workspace */
    MOE_WS_Y_PERM = 9,      /* [R,d] bf16 */
    MOE_WS_CHUNK_BASE = 10, /* dispatch scratch: [chunks,E] int32 */
    MOE_WS_L1_DONE = 11,    /* per scheduler row: finished Linear-1 tiles, u32; then per row the
                               finished Linear-2 tiles (used by the h ring); then the grouped
                               GEMM's tile ticket counter */
    MOE_WS_L2_FLAGS = 12,   /* per Linear-2 tile: ready flag = epoch of the call that wrote it, u32
                               (a call captured in a CUDA Graph keeps its capture-time epoch on
                               every replay) */
    MOE_WS_NUM_REGIONS = 13
};
moe_status_t moe_workspace_region(const moe_shape_t *shape, int region, size_t *offset,
                                  size_t *bytes);
/* The same for the layout of moe_workspace_bytes_tuned(shape, tuning). */
moe_status_t moe_workspace_region_tuned(const moe_shape_t *shape, const moe_tuning_t *tuning,
                                        int region, size_t *offset, size_t *bytes);

/* Step 1, routing (Cui et al. section 2.1 step 1; Xian et al. section 2.2).
 *   z[t,e] = sum_i x[t,i] * w_router[e,i] (+ expert_bias[e]), accumulated in
 *   fp32 in ascending i; topk_idx[t,:] = the k largest z, descending, ties to
 *   the lower expert index; topk_gate[t,:] = softmax of those k logits.
 * x [T,d] bf16, w_router [E,d] bf16, expert_bias [E] fp32 or NULL,
 * topk_idx [T,k] int32 (out), topk_gate [T,k] fp32 (out). */
moe_status_t moe_route(const moe_shape_t *shape, const moe_bf16_t *x, const moe_bf16_t *w_router,
                       const float *expert_bias, int32_t *topk_idx, float *topk_gate,
                       moe_stream_t stream);

/* Bytes of device scratch moe_route_filtered needs for this shape; 0 for an
 * invalid shape. */
size_t moe_route_scratch_bytes(const moe_shape_t *shape);

/* moe_route by filter then verify (moe_router_t MOE_ROUTER_FILTER_VERIFY):
 * the same topk_idx and topk_gate bits as moe_route, in four launches that
 * sum exactly only the experts that can still be in the top k.
 * scratch: device buffer of at least moe_route_scratch_bytes, 256-byte
 * aligned, owned by the caller; its first 16 bytes are a status word like the
 * workspace's (zero before the call: allocate it zeroed, and
 * moe_last_device_status(scratch, stream) reads and clears it). Calls that
 * share a scratch buffer must not overlap on the GPU. d must be below 2^20
 * (else MOE_ERR_UNSUPPORTED). */
moe_status_t moe_route_filtered(const moe_shape_t *shape, const moe_bf16_t *x, const moe_bf16_t *w_router,
                                const float *expert_bias, int32_t *topk_idx, float *topk_gate, void *scratch,
                                size_t scratch_bytes, moe_stream_t stream);

/* Step 2, dispatch (Cui et al. section 2.1 step 2): a stable counting sort of
 * the R token copies by expert, in (token, choice) order.
 *   expert_counts[e] = #{(t,j): topk_idx[t,j] == e}; expert_offsets = exclusive
 *   scan (E+1 entries, last = R); row_of_slot[t*k+j] = destination row;
 *   slot_of_row = its inverse; x_perm[r] = x[slot_of_row[r] / k].
 * x [T,d] bf16, topk_idx [T,k] int32, outputs as named; ws: a workspace of
 * moe_workspace_bytes or moe_workspace_bytes_tuned (uses the CHUNK_BASE and
 * STATUS regions, which lie before h; ws_bytes must reach the start of h).
 * An expert id outside [0,E) is skipped (its row_of_slot entry becomes -1, it
 * is not counted) and recorded as MOE_ERR_INVALID_ARG in the device status. */
moe_status_t moe_dispatch(const moe_shape_t *shape, const moe_bf16_t *x, const int32_t *topk_idx,
                          int32_t *expert_counts, int32_t *expert_offsets, int32_t *row_of_slot,
                          int32_t *slot_of_row, moe_bf16_t *x_perm, void *ws, size_t ws_bytes,
                          moe_stream_t stream);

/* moe_dispatch without a workspace. The pages have no counterpart to this
 * call; it exists for callers that cannot allocate device memory for the
 * library: a host application that owns every device buffer and passes only
 * the tensors it already holds, or a latency-critical loop that must not call
 * cudaMalloc (which can synchronise the device) and has no spare memory budget.
 * Same arguments, results and rules as moe_dispatch, minus ws/ws_bytes.
 *   - Its scratch is a fixed array inside this library's device memory: 4096
 *     (chunk, expert) cells (16 KiB) plus 256 B of status words, present on
 *     every GPU that loads the library until the process exits. Shapes whose
 *     dispatch needs more cells than that (roughly T*E > 2^20 token-expert
 *     pairs) return MOE_ERR_UNSUPPORTED without enqueuing anything.
 *   - The first call on each device looks up that array's device address
 *     (with the device current) and caches it; make that first call before
 *     any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind: calls that overlap on the GPU (other streams, other threads)
 *     race; serialise them.
 *   - An expert id outside [0,E) is skipped (row_of_slot = -1, not counted)
 *     but, with no workspace, not reported through a device status word. */
moe_status_t moe_dispatch_noalloc(const moe_shape_t *shape, const moe_bf16_t *x,
                                  const int32_t *topk_idx, int32_t *expert_counts,
                                  int32_t *expert_offsets, int32_t *row_of_slot,
                                  int32_t *slot_of_row, moe_bf16_t *x_perm, moe_stream_t stream);

/* Step 3, expert computation (Xian et al. section 2.2) as one persistent
 * grouped GEMM over all experts (tcgen05 MMA, bf16 in, fp32 accumulation in
 * tensor memory):
 *   for rows r in [off[e], off[e+1]):
 *     h[r]      = bf16( silu(x_perm[r] W1[e]^T) * (x_perm[r] W3[e]^T) )
 *     y_perm[r] = bf16( h[r] W2[e]^T )
 * Linear-2 tiles are interleaved with Linear-1 tiles (Xian et al., Algorithm 1)
 * and each publishes a ready flag after its store (Cui et al. section 3.3.1).
 * x_perm [R,d] bf16; expert_offsets [E+1] int32 (non-decreasing, off[0]=0,
 * off[E]=R; other offsets are recorded as MOE_ERR_INVALID_ARG in the device
 * status and nothing is computed); W1, W3 [E,F,d] bf16; W2 [E,d,F] bf16;
 * y_perm [R,d] bf16 (out); h lives in the workspace (region MOE_WS_H).
 * The grouped GEMM is a persistent grid of one CTA (or CTA pair) per SM. Its
 * CTAs take tiles in one global order from a counter in the workspace, and a
 * tile only ever waits for tiles earlier in that order, which running CTAs
 * hold; so it completes whatever share of the GPU it gets, also beside other
 * grouped GEMMs (other streams, other threads, other workspaces). */
moe_status_t moe_expert_ffn(const moe_shape_t *shape, const moe_bf16_t *x_perm,
                            const int32_t *expert_offsets, const moe_bf16_t *W1,
                            const moe_bf16_t *W3, const moe_bf16_t *W2, moe_bf16_t *y_perm,
                            void *ws, size_t ws_bytes, moe_stream_t stream);

/* moe_expert_ffn with an explicit tile schedule (tuning may be NULL = defaults);
 * ws_bytes is checked against moe_workspace_bytes_tuned(shape, tuning). */
moe_status_t moe_expert_ffn_tuned(const moe_shape_t *shape, const moe_tuning_t *tuning,
                                  const moe_bf16_t *x_perm, const int32_t *expert_offsets,
                                  const moe_bf16_t *W1, const moe_bf16_t *W3, const moe_bf16_t *W2,
                                  moe_bf16_t *y_perm, void *ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* Steps 4-5, combine and weighted sum (Cui et al. section 2.1 steps 4-5):
 *   out[t] = bf16( sum_j topk_gate[t,j] * y_perm[row_of_slot[t*k+j]] ), an fp32
 *   sum in j order; token t is row (t mod T/S) of segment t / (T/S).
 * y_perm [R,d] bf16, topk_gate [T,k] fp32, row_of_slot [R] int32;
 * out_segments: HOST array of S device pointers, each [T/S, d] bf16 (out). */
moe_status_t moe_combine(const moe_shape_t *shape, const moe_bf16_t *y_perm,
                         const float *topk_gate, const int32_t *row_of_slot,
                         moe_bf16_t *const *out_segments, moe_stream_t stream);

/* The whole layer: route -> dispatch -> grouped SwiGLU GEMM -> combine, seven
 * kernel launches on one stream (route; count, scan, rank and copy for the
 * dispatch; the grouped GEMM; combine), ten when the route filters then
 * verifies (moe_router_t: weight norms, candidates, exact candidates, full
 * rows), no host synchronisation. Intermediates (routing, permutation, x_perm,
 * h, y_perm) stay in the workspace regions. */
moe_status_t moe_layer_forward(const moe_shape_t *shape, const moe_bf16_t *x,
                               const moe_bf16_t *w_router, const float *expert_bias,
                               const moe_bf16_t *W1, const moe_bf16_t *W3, const moe_bf16_t *W2,
                               moe_bf16_t *const *out_segments, void *ws, size_t ws_bytes,
                               moe_stream_t stream);

/* Kernel launches one moe_layer_forward_tuned call makes for this shape and
 * tuning (NULL = defaults): route (1, or 4 when it filters then verifies), the
 * dispatch's count, scan, rank and row copy, the grouped GEMM, and the combine
 * unless fused_combine. 0 for an
 * invalid shape or tuning; the layer makes no launch at all when T == 0. */
int moe_layer_kernel_launches(const moe_shape_t *shape, const moe_tuning_t *tuning);

/* moe_layer_forward with an explicit tile schedule (tuning may be NULL); the
 * workspace is sized by moe_workspace_bytes_tuned(shape, tuning). */
moe_status_t moe_layer_forward_tuned(const moe_shape_t *shape, const moe_tuning_t *tuning,
                                     const moe_bf16_t *x, const moe_bf16_t *w_router,
                                     const float *expert_bias, const moe_bf16_t *W1,
                                     const moe_bf16_t *W3, const moe_bf16_t *W2,
                                     moe_bf16_t *const *out_segments, void *ws, size_t ws_bytes,
                                     moe_stream_t stream);

/* moe_layer_forward_tuned that also records caller-created CUDA events
 * (cudaEvent_t, passed as void*) on `stream` at the stage boundaries:
 * stage_events[0] before routing, [1] after routing, [2] after dispatch,
 * [3] after the grouped GEMM, [4] after combine. stage_events may be NULL;
 * otherwise all five entries must be valid events of the stream's device. */
moe_status_t moe_layer_forward_ex(const moe_shape_t *shape, const moe_tuning_t *tuning,
                                  const moe_bf16_t *x, const moe_bf16_t *w_router,
                                  const float *expert_bias, const moe_bf16_t *W1,
                                  const moe_bf16_t *W3, const moe_bf16_t *W2,
                                  moe_bf16_t *const *out_segments, void *ws, size_t ws_bytes,
                                  moe_stream_t stream, void *const *stage_events);

/* Synchronises `stream`, returns the device status recorded in `ws`
 * (MOE_OK, or MOE_ERR_TIMEOUT when a bounded wait ran out) and clears it.
 * A failed CUDA call returns MOE_ERR_CUDA. */
moe_status_t moe_last_device_status(void *ws, moe_stream_t stream);

/* Detail words of the last device failure that moe_last_device_status read on
 * the calling thread (valid after it returned non-OK there): where (kernel/role
 * code: 1-5 grouped-GEMM pipeline waits, 6 dispatch, 7 GEMM offsets, 8 fused
 * combine, 9-10 GEMM drains, 11 tile queue, 12 filter-then-verify router),
 * block index, detail. */
void moe_last_device_detail(uint32_t *where, uint32_t *block, uint32_t *detail);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
