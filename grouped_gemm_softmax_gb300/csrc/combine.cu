// combine.cu -- steps 4-5 of the MoE forward, combine and weighted sum (Cui et
// al., "Fine-grained Computation-Communication Overlap ...", section 2.1: the
// expert outputs return to their token and the layer output is their
// gate-weighted sum; Xian et al., "X-Stage ...", section 2.2).
//
//   out[t] = bf16( sum_j gate[t,j] * y_perm[row_of_slot[t*k+j]] )   (fp32, j order)
//
// Token t belongs to simulated source rank s = t / (T/S) and is written to row
// t mod (T/S) of that rank's segment, the owner-aligned layout a multi-GPU
// combine would send as one contiguous block per rank.
//
// One warp per token; each lane owns 16-byte column vectors (8 bf16), loads the
// k expert rows with 128-bit loads and accumulates in fp32 in j order.
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

struct Segments {
    uint16_t *p[kMaxSegments];
};

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4 &v, float g)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        acc[2 * h] = fmaf(g, __uint_as_float(w[h] << 16), acc[2 * h]);
        acc[2 * h + 1] = fmaf(g, __uint_as_float(w[h] & 0xFFFF0000u), acc[2 * h + 1]);
    }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// KMAX bounds k; each lane keeps U = 16 / KMAX column vectors of every expert
// row in flight (up to 16 loads of 16 bytes), so few warps still have enough
// memory-level parallelism to cover HBM latency.
template <int KMAX>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const uint16_t *__restrict__ y, const float *__restrict__ gate,
               const int32_t *__restrict__ row_of_slot, int T, int d, int k, int rows_per_seg,
               const Segments seg, int early_maps)
{
    constexpr int U = 16 / KMAX;
    // Inside the layer the row map and the gates come from kernels that
    // finished before the grouped GEMM passed its own wait, so they are read
    // before this kernel's wait; only y_perm needs it. Called on its own, the
    // combine may follow the kernels that write them, and waits first.
    if (!early_maps) pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long t = static_cast<long>(blockIdx.x) * (kThreads / 32) + warp;
    const uint4 *src[KMAX];
    float g[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        // a slot whose expert id was out of range has no row (-1): no term;
        // neither has a row index past the T*k rows of y_perm
        const int r = (t < T && j < k) ? row_of_slot[t * k + j] : -1;
        src[j] = (r >= 0 && r < static_cast<long>(T) * k)
                     ? reinterpret_cast<const uint4 *>(y + static_cast<long>(r) * d)
                     : nullptr;
        g[j] = (t < T && j < k) ? gate[t * k + j] : 0.0f;
    }
    if (early_maps) pdl_wait();
    if (t >= T) return;
    uint4 *dst = reinterpret_cast<uint4 *>(seg.p[t / rows_per_seg] + (t % rows_per_seg) * static_cast<long>(d));
    const int nvec = d / 8;
    for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
        uint4 val[U][KMAX];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (src[j] != nullptr && v0 + 32 * u < nvec) val[u][j] = src[j][v0 + 32 * u];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (v0 + 32 * u >= nvec) break;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (src[j] != nullptr) acc_bf16x8(acc, val[u][j], g[j]);
            uint4 o;
            o.x = pack2(acc[0], acc[1]);
            o.y = pack2(acc[2], acc[3]);
            o.z = pack2(acc[4], acc[5]);
            o.w = pack2(acc[6], acc[7]);
            dst[v0 + 32 * u] = o;
        }
    }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s)
{
    if (a.T == 0) return cudaSuccess;
    Segments seg;
    for (int i = 0; i < kMaxSegments; ++i) seg.p[i] = i < a.S ? a.seg[i] : nullptr;
    const unsigned blocks = static_cast<unsigned>((a.T + kThreads / 32 - 1) / (kThreads / 32));
    if (a.k <= 2)
        return launch_pdl(combine_kernel<2>, dim3(blocks), dim3(kThreads), 0, s, a.y, a.gate, a.row_of_slot,
                          a.T, a.d, a.k, a.T / a.S, seg, a.early_maps ? 1 : 0);
    if (a.k <= 4)
        return launch_pdl(combine_kernel<4>, dim3(blocks), dim3(kThreads), 0, s, a.y, a.gate, a.row_of_slot,
                          a.T, a.d, a.k, a.T / a.S, seg, a.early_maps ? 1 : 0);
    return launch_pdl(combine_kernel<8>, dim3(blocks), dim3(kThreads), 0, s, a.y, a.gate, a.row_of_slot,
                          a.T, a.d, a.k, a.T / a.S, seg, a.early_maps ? 1 : 0);
}

}  // namespace moe
