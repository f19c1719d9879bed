// dispatch.cu -- step 2 of the MoE forward, dispatch (Cui et al., "Fine-grained
// Computation-Communication Overlap ...", section 2.1 step 2): every token copy
// (t, j) goes to a row of its expert's contiguous block, stable in (t, j)
// order, and its hidden vector is copied there.
//
// Four kernels, all deterministic (no atomics whose order decides a result):
//   1. count   one block per chunk of C tokens: per-expert counts of its slots
//   2. scan    one block: per expert, exclusive scan over chunks, then over
//              experts -> expert_counts, expert_offsets, and each chunk's
//              first row per expert; also clears the grouped GEMM's counters
//   3. rank    one block per chunk: each warp takes a contiguous slice of the
//              chunk's slots; per-warp counts and a prefix over warps give each
//              warp its bases; it then ranks equal experts 32 slots at a time
//              with __match_any_sync and writes row_of_slot / slot_of_row
//   4. copy    one warp per token: x[t] read once with 16-byte loads (the
//              first 2048 features before the wait on rank) and written to
//              its k destination rows
#include "kernels.cuh"
#include "sm100.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kScanMaxCells = 8192;  // chunks * E held in shared memory by the scan
constexpr int kRankBatch = 2048;      // slots staged in shared memory per pass

__global__ void __launch_bounds__(kThreads) count_kernel(const int32_t *__restrict__ idx, int T, int k,
                                                         int E, int C, int32_t *chunk_base,
                                                         unsigned *status)
{
    __shared__ int cnt[kMaxExperts];
    pdl_wait();
    pdl_trigger();
    for (int e = threadIdx.x; e < E; e += kThreads) cnt[e] = 0;
    __syncthreads();
    const long s0 = static_cast<long>(blockIdx.x) * C * k;
    const long s1 = min(static_cast<long>(T), static_cast<long>(blockIdx.x + 1) * C) * k;
    for (long s = s0 + threadIdx.x; s < s1; s += kThreads) {
        const int e = idx[s];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else report_failure(status, kStatusBadExpert, kWhereDispatch, static_cast<unsigned>(s));
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads)
        chunk_base[static_cast<long>(blockIdx.x) * E + e] = cnt[e];
}

__global__ void __launch_bounds__(kThreads) scan_kernel(int32_t *chunk_base, int nchunks, int E,
                                                        int32_t *counts, int32_t *offsets,
                                                        unsigned *zero_words, long zero_count)
{
    __shared__ int cells[kScanMaxCells];
    __shared__ int tot[kMaxExperts];
    __shared__ int warp_sums[kThreads / 32];
    pdl_wait();
    pdl_trigger();
    const int n = nchunks * E;
    for (int i = threadIdx.x; i < n; i += kThreads) cells[i] = chunk_base[i];
    __syncthreads();
    // per expert: exclusive scan over chunks (in chunk order)
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int run = 0;
        for (int c = 0; c < nchunks; ++c) {
            const int v = cells[c * E + e];
            cells[c * E + e] = run;
            run += v;
        }
        tot[e] = run;
    }
    __syncthreads();
    // exclusive scan over experts (E <= 256 = kThreads)
    const int e = threadIdx.x;
    const int v = e < E ? tot[e] : 0;
    const int lane = e & 31, w = e >> 5;
    int incl = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < w; ++i) before += warp_sums[i];
    const int excl = before + incl - v;
    if (e < E) {
        counts[e] = v;
        offsets[e] = excl;
        if (e == E - 1) offsets[E] = excl + v;
        tot[e] = excl;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kThreads) chunk_base[i] = cells[i] + tot[i % E];
    for (long i = threadIdx.x; i < zero_count; i += kThreads) zero_words[i] = 0u;
}

// Each warp of the block owns a contiguous slice of the staged slots. Pass 1:
// per-warp, per-expert counts. Then each expert's base for warp w is the
// chunk's base plus the counts of warps 0..w-1 (slot order is preserved).
// Pass 2: each warp ranks its slice 32 slots at a time (__match_any_sync),
// in order, from its own bases.
__global__ void __launch_bounds__(kThreads) rank_kernel(const int32_t *__restrict__ idx, int T, int k,
                                                        int E, int C,
                                                        const int32_t *__restrict__ chunk_base,
                                                        int32_t *row_of_slot, int32_t *slot_of_row)
{
    constexpr int NW = kThreads / 32;
    __shared__ int cur[kMaxExperts];            // running base per expert across batches
    __shared__ int wcnt[NW][kMaxExperts];       // per-warp counts, then per-warp bases
    __shared__ int sidx[kRankBatch];
    pdl_wait();
    pdl_trigger();
    for (int e = threadIdx.x; e < E; e += kThreads)
        cur[e] = chunk_base[static_cast<long>(blockIdx.x) * E + e];
    const long s0 = static_cast<long>(blockIdx.x) * C * k;
    const long s1 = min(static_cast<long>(T), static_cast<long>(blockIdx.x + 1) * C) * k;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt = (1u << lane) - 1u;
    for (long b0 = s0; b0 < s1; b0 += kRankBatch) {
        const int nb = static_cast<int>(min(static_cast<long>(kRankBatch), s1 - b0));
        __syncthreads();
        for (int i = threadIdx.x; i < nb; i += kThreads) sidx[i] = idx[b0 + i];
        for (int i = threadIdx.x; i < NW * E; i += kThreads) wcnt[i / E][i % E] = 0;
        __syncthreads();
        // this warp's slice of the batch, in 32-slot steps
        const int per = (nb + NW - 1) / NW;
        const int lo = min(nb, warp * per), hi = min(nb, lo + per);
        for (int i0 = lo; i0 < hi; i0 += 32) {
            const int i = i0 + lane;
            const int e0 = i < hi ? sidx[i] : -1;
            const int e = (e0 >= 0 && e0 < E) ? e0 : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && __popc(peers & lt) == 0) wcnt[warp][e] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        // exclusive prefix over warps, per expert; advance the running base
        for (int e = threadIdx.x; e < E; e += kThreads) {
            int run = cur[e];
            for (int w = 0; w < NW; ++w) {
                const int c = wcnt[w][e];
                wcnt[w][e] = run;
                run += c;
            }
            cur[e] = run;
        }
        __syncthreads();
        for (int i0 = lo; i0 < hi; i0 += 32) {
            const int i = i0 + lane;
            const int e0 = i < hi ? sidx[i] : -1;
            const bool in_range = e0 >= 0 && e0 < E;
            const int e = in_range ? e0 : -1;
            if (i < hi && !in_range) row_of_slot[b0 + i] = -1;
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(peers & lt);
            const int base = e >= 0 ? wcnt[warp][e] : 0;
            __syncwarp();
            if (e >= 0) {
                const int row = base + rank;
                const long sl = b0 + i;
                row_of_slot[sl] = row;
                slot_of_row[row] = static_cast<int32_t>(sl);
                if (rank == 0) wcnt[warp][e] = base + __popc(peers);
            }
            __syncwarp();
        }
    }
}

// One warp per token. The first 2048 features of the token's row are loaded
// before the wait on the rank kernel: x was complete before the first
// dispatch kernel passed its own wait, and each kernel of the chain launches
// only after every block of its predecessor passed that predecessor's wait,
// so the x loads overlap the bookkeeping kernels; only the row map needs the
// wait.
__global__ void __launch_bounds__(kThreads) copy_kernel(const uint16_t *__restrict__ x,
                                                        const int32_t *__restrict__ row_of_slot,
                                                        int T, int d, int k, uint16_t *x_perm)
{
    constexpr int U = 8;  // 16-byte vectors per lane loaded ahead
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long t = static_cast<long>(blockIdx.x) * (kThreads / 32) + warp;
    const bool live = t < T;
    const int nvec = d / 8;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (live ? t : 0) * d);
    uint4 ahead[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int v = u * 32 + lane;
        if (live && v < nvec) ahead[u] = src[v];
    }
    pdl_wait();
    if (!live) return;
    int rows[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) rows[j] = j < k ? row_of_slot[t * k + j] : -1;
    auto put = [&](int v, const uint4 &val) {
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
            if (j < k && rows[j] >= 0) reinterpret_cast<uint4 *>(x_perm + static_cast<long>(rows[j]) * d)[v] = val;
    };
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int v = u * 32 + lane;
        if (v < nvec) put(v, ahead[u]);
    }
    for (int v = U * 32 + lane; v < nvec; v += 32) put(v, src[v]);
}

}  // namespace

int dispatch_chunk_tokens(int T, int E)
{
    // at most kScanMaxCells (chunk, expert) cells for the single-block scan
    const long max_chunks = kScanMaxCells / E;
    long c = (static_cast<long>(T) + max_chunks - 1) / max_chunks;
    c = (c + 31) / 32 * 32;
    return static_cast<int>(c < 256 ? 256 : c);
}

cudaError_t launch_dispatch(const DispatchArgs &a, cudaStream_t s)
{
    if (a.T == 0) {
        // no tokens: counts and offsets are all zero
        cudaError_t err = cudaMemsetAsync(a.counts, 0, sizeof(int32_t) * a.E, s);
        if (err == cudaSuccess) err = cudaMemsetAsync(a.offsets, 0, sizeof(int32_t) * (a.E + 1), s);
        return err;
    }
    const int C = a.chunk_tokens;
    const int nchunks = (a.T + C - 1) / C;
    cudaError_t err = launch_pdl(count_kernel, dim3(nchunks), dim3(kThreads), 0, s, a.topk_idx, a.T, a.k,
                                 a.E, C, a.chunk_base, a.status);
    if (err == cudaSuccess)
        err = launch_pdl(scan_kernel, dim3(1), dim3(kThreads), 0, s, a.chunk_base, nchunks, a.E, a.counts,
                         a.offsets, a.zero_words, a.zero_words ? a.zero_count : 0L);
    if (err == cudaSuccess)
        err = launch_pdl(rank_kernel, dim3(nchunks), dim3(kThreads), 0, s, a.topk_idx, a.T, a.k, a.E, C,
                         static_cast<const int32_t *>(a.chunk_base), a.row_of_slot, a.slot_of_row);
    const unsigned copy_blocks = static_cast<unsigned>((a.T + kThreads / 32 - 1) / (kThreads / 32));
    if (err == cudaSuccess)
        err = launch_pdl(copy_kernel, dim3(copy_blocks), dim3(kThreads), 0, s, a.x,
                         static_cast<const int32_t *>(a.row_of_slot), a.T, a.d, a.k, a.x_perm);
    return err;
}

}  // namespace moe
