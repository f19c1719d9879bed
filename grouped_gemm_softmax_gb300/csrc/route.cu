// route.cu -- step 1 of the MoE forward, routing (Cui et al., "Fine-grained
// Computation-Communication Overlap ...", section 2.1 step 1: the router picks
// the top-k experts from a probability distribution and yields the gate
// weights; Xian et al., "X-Stage ...", section 2.2).
//
//   z[t,e]        = sum_i x[t,i] * Wr[e,i]  (+ bias[e])
//   topk_idx[t,:] = the k largest z[t,:], descending, ties to the lower index
//   topk_gate[t,:]= softmax over those k logits
//
// Logits are computed on CUDA cores in fp32 (tensor cores are kept for the
// expert GEMMs). Each logit is accumulated by ONE thread in ascending i, one
// fused multiply-add per feature: every bf16 x bf16 product is exact in fp32,
// so the result is the fp32 sequential sum, rounded once per addition,
// independent of the tiling. The selection is therefore reproducible bit for
// bit by any implementation of that sum.
//
// Kernels, by expert count (each thread owns TM tokens x TN experts of a
// block tile; the tiles of x and the weights pass through shared memory a
// chunk of features at a time):
//   E > 128, 33..64   route_kernel_bf16: bf16 tiles in a cp.async ring, the
//                     mixed-precision FMA (bf16 operands, fp32 accumulator)
//   <= 16             route_kernel_resident: weights resident per block,
//                     per-warp rings over 32-token (9..16 experts) or 8-token
//                     (<= 8) tasks, selection in lane (when the weights fit;
//                     else route_kernel or route_kernel_async)
//   65..128, 17..32   route_kernel: fp32 tiles, register prefetch
// Except in route_kernel_resident, one warp per token then runs k rounds of a
// shuffle arg-max over the block's logits and writes idx and gates.
#include <cuda_bf16.h>
#include <float.h>

#include "kernels.cuh"

namespace moe {
namespace {

constexpr size_t kMaxSmemPerBlock = 232448;  // opt-in shared memory per block (227 KB)

struct RouteParams {
    const uint16_t *x;
    const uint16_t *wr;
    const float *bias;
    int32_t *idx;
    float *gate;
    int T, d, E, k;
};

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16)
{
    return __uint_as_float(bits16 << 16);
}

// One warp per token of the block: k rounds of a shuffle arg-max (descending
// logit, ties to the lower expert index) over the block's logits, then the
// softmax of the k selected logits in fp32.
template <int BE, int NW>
__device__ __forceinline__ void select_topk(const RouteParams &p, const float *lg, long t0, int BT,
                                            int warp, int lane)
{
    for (int r = warp; r < BT; r += NW) {
        const long t = t0 + r;
        if (t >= p.T) break;
        const float *row = lg + r * (BE + 1);
        constexpr int PER = (BE + 31) / 32;
        float v[PER];
        uint32_t avail = 0;  // bit i: expert lane + 32*i not yet selected
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = lane + 32 * i;
            if (e < p.E) avail |= 1u << i;
            v[i] = e < p.E ? row[e] : 0.0f;
        }
        int sel_e = 0;
        float sel_v = 0.0f;
        for (int j = 0; j < p.k; ++j) {
            float bv = -FLT_MAX;
            int be = INT_MAX;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int e = lane + 32 * i;
                if (((avail >> i) & 1u) && (be == INT_MAX || v[i] > bv || (v[i] == bv && e < be))) {
                    bv = v[i];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane) avail &= ~(1u << (be >> 5));
            if (lane == j) {
                sel_e = be;
                sel_v = bv;
            }
        }
        // softmax over the k selected logits (lane j holds choice j)
        const float zmax = __shfl_sync(0xffffffffu, sel_v, 0);
        const float ex = lane < p.k ? expf(sel_v - zmax) : 0.0f;
        float den = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (lane < p.k) {
            p.idx[t * p.k + lane] = sel_e;
            p.gate[t * p.k + lane] = ex / den;
        }
    }
}

// Thread layout: lane = 8 token lanes x 4 expert lanes; warps = WE along
// experts x WT along tokens. Thread (a, b) of warp (we, wt) owns tokens
// tb + a + 8i (i < TM) and experts eb + b + 4j (j < TN), so for any fixed i
// (or j) the warp touches consecutive rows of the shared tiles, which are
// padded to 36 floats a row: every 16-byte access is bank-conflict free.
template <int TM, int TN, int WE, int WT, int kBK>
__global__ void __launch_bounds__(32 * WE * WT) route_kernel(const RouteParams p)
{
    constexpr int NT = 32 * WE * WT;
    constexpr int BT = WT * 8 * TM;  // tokens per block
    constexpr int BE = WE * 4 * TN;  // experts per block (>= E)
    constexpr int NW = NT / 32;
    constexpr int LD = kBK + 4;      // padded row (floats)
    constexpr int XV = BT * (kBK / 8);
    constexpr int WV = BE * (kBK / 8);
    constexpr int XPT = (XV + NT - 1) / NT;
    constexpr int WPT = (WV + NT - 1) / NT;
    extern __shared__ float rsm[];
    float *xs = rsm;            // [BT][LD]
    float *ws = rsm + BT * LD;  // [BE][LD]
    float *lg = rsm;            // [BT][BE + 1] (reused after the K loop)
    pdl_wait();
    pdl_trigger();

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int a = lane & 7, b = lane >> 3;
    const int eb = (warp % WE) * 4 * TN, tb = (warp / WE) * 8 * TM;
    const long t0 = static_cast<long>(blockIdx.x) * BT;

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

    // register prefetch of the next chunk (global -> registers -> shared)
    uint4 px[XPT], pw[WPT];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int u = 0; u < XPT; ++u) {
            const int v = tid + u * NT;
            px[u] = make_uint4(0, 0, 0, 0);
            if (v < XV) {
                const int r = v / (kBK / 8), c8 = (v % (kBK / 8)) * 8;
                const long t = t0 + r;
                if (t < p.T && k0 + c8 < p.d)
                    px[u] = __ldg(reinterpret_cast<const uint4 *>(p.x + t * p.d + k0 + c8));
            }
        }
#pragma unroll
        for (int u = 0; u < WPT; ++u) {
            const int v = tid + u * NT;
            pw[u] = make_uint4(0, 0, 0, 0);
            if (v < WV) {
                const int r = v / (kBK / 8), c8 = (v % (kBK / 8)) * 8;
                if (r < p.E && k0 + c8 < p.d)
                    pw[u] = __ldg(reinterpret_cast<const uint4 *>(p.wr + static_cast<long>(r) * p.d +
                                                                  k0 + c8));
            }
        }
    };
    auto widen = [](const uint4 &q, float4 &lo, float4 &hi) {
        lo = make_float4(bf16_bits_to_f32(q.x & 0xFFFFu), bf16_bits_to_f32(q.x >> 16),
                         bf16_bits_to_f32(q.y & 0xFFFFu), bf16_bits_to_f32(q.y >> 16));
        hi = make_float4(bf16_bits_to_f32(q.z & 0xFFFFu), bf16_bits_to_f32(q.z >> 16),
                         bf16_bits_to_f32(q.w & 0xFFFFu), bf16_bits_to_f32(q.w >> 16));
    };
    auto stage = [&]() {
#pragma unroll
        for (int u = 0; u < XPT; ++u) {
            const int v = tid + u * NT;
            if (v < XV) {
                const int r = v / (kBK / 8), c8 = (v % (kBK / 8)) * 8;
                float4 lo, hi;
                widen(px[u], lo, hi);
                *reinterpret_cast<float4 *>(xs + r * LD + c8) = lo;
                *reinterpret_cast<float4 *>(xs + r * LD + c8 + 4) = hi;
            }
        }
#pragma unroll
        for (int u = 0; u < WPT; ++u) {
            const int v = tid + u * NT;
            if (v < WV) {
                const int r = v / (kBK / 8), c8 = (v % (kBK / 8)) * 8;
                float4 lo, hi;
                widen(pw[u], lo, hi);
                *reinterpret_cast<float4 *>(ws + r * LD + c8) = lo;
                *reinterpret_cast<float4 *>(ws + r * LD + c8 + 4) = hi;
            }
        }
    };

    fetch(0);
    for (int k0 = 0; k0 < p.d; k0 += kBK) {
        stage();
        __syncthreads();
        if (k0 + kBK < p.d) fetch(k0 + kBK);
#pragma unroll 2
        for (int kk = 0; kk < kBK; kk += 4) {
            float4 xv[TM], wv[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i)
                xv[i] = *reinterpret_cast<const float4 *>(xs + (tb + a + 8 * i) * LD + kk);
#pragma unroll
            for (int j = 0; j < TN; ++j)
                wv[j] = *reinterpret_cast<const float4 *>(ws + (eb + b + 4 * j) * LD + kk);
            // ascending feature order for every (token, expert) accumulator
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    acc[i][j] = fmaf(xv[i].x, wv[j].x, acc[i][j]);
                    acc[i][j] = fmaf(xv[i].y, wv[j].y, acc[i][j]);
                    acc[i][j] = fmaf(xv[i].z, wv[j].z, acc[i][j]);
                    acc[i][j] = fmaf(xv[i].w, wv[j].w, acc[i][j]);
                }
        }
        __syncthreads();
    }

    // logits (+ bias, one fp32 addition) into shared memory
#pragma unroll
    for (int i = 0; i < TM; ++i) {
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int e = eb + b + 4 * j;
            float z = acc[i][j];
            if (p.bias != nullptr && e < p.E) z = z + p.bias[e];
            lg[(tb + a + 8 * i) * (BE + 1) + e] = z;
        }
    }
    __syncthreads();

    select_topk<BE, NW>(p, lg, t0, BT, warp, lane);
}

// Small expert counts: the FMA work per token is light, so the kernel is bound
// by how many bytes of x each SM has in flight. This variant streams raw bf16
// chunks of KB features into a STAGES-deep shared-memory ring with cp.async
// (16-byte copies, zero-filled past the end) and widens to fp32 at use. Same
// thread layout and the same ascending-feature accumulation as route_kernel.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src, bool valid)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int TM, int TN, int WE, int WT, int KB, int STAGES>
__global__ void __launch_bounds__(32 * WE * WT) route_kernel_async(const RouteParams p)
{
    constexpr int NT = 32 * WE * WT;
    constexpr int BT = WT * 8 * TM;
    constexpr int BE = WE * 4 * TN;
    constexpr int NW = NT / 32;
    constexpr int LD = KB + 8;  // padded row (bf16): rows 4 banks apart
    constexpr int STAGE = (BT + BE) * LD;  // bf16 per stage
    constexpr int CPR = KB / 8;            // 16-byte copies per row
    extern __shared__ __align__(16) uint16_t rsm16[];
    float *lg = reinterpret_cast<float *>(rsm16);  // [BT][BE + 1] after the K loop
    pdl_wait();
    pdl_trigger();

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int a = lane & 7, b = lane >> 3;
    const int eb = (warp % WE) * 4 * TN, tb = (warp / WE) * 8 * TM;
    const long t0 = static_cast<long>(blockIdx.x) * BT;
    const int nchunks = (p.d + KB - 1) / KB;

    auto issue = [&](int chunk) {
        uint16_t *st = rsm16 + (chunk % STAGES) * STAGE;
        const int k0 = chunk * KB;
        for (int v = tid; v < (BT + BE) * CPR; v += NT) {
            const int r = v / CPR, c8 = (v % CPR) * 8;
            const bool is_x = r < BT;
            const long row = is_x ? t0 + r : static_cast<long>(r - BT);
            const bool ok = k0 + c8 < p.d && (is_x ? row < p.T : row < p.E);
            const uint16_t *src = is_x ? p.x + (ok ? row * p.d + k0 + c8 : 0)
                                       : p.wr + (ok ? row * p.d + k0 + c8 : 0);
            cp_async_16(st + r * LD + c8, src, ok);
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

#pragma unroll
    for (int c = 0; c < STAGES - 1; ++c) {
        if (c < nchunks) issue(c);
        cp_async_commit();
    }
    for (int c = 0; c < nchunks; ++c) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        if (c + STAGES - 1 < nchunks) issue(c + STAGES - 1);
        cp_async_commit();
        const uint16_t *xs = rsm16 + (c % STAGES) * STAGE;
        const uint16_t *ws = xs + BT * LD;
#pragma unroll 4
        for (int kk = 0; kk < KB; kk += 4) {
            float xv[TM][4], wv[TN][4];
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const uint2 q = *reinterpret_cast<const uint2 *>(xs + (tb + a + 8 * i) * LD + kk);
                xv[i][0] = bf16_bits_to_f32(q.x & 0xFFFFu);
                xv[i][1] = bf16_bits_to_f32(q.x >> 16);
                xv[i][2] = bf16_bits_to_f32(q.y & 0xFFFFu);
                xv[i][3] = bf16_bits_to_f32(q.y >> 16);
            }
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const uint2 q = *reinterpret_cast<const uint2 *>(ws + (eb + b + 4 * j) * LD + kk);
                wv[j][0] = bf16_bits_to_f32(q.x & 0xFFFFu);
                wv[j][1] = bf16_bits_to_f32(q.x >> 16);
                wv[j][2] = bf16_bits_to_f32(q.y & 0xFFFFu);
                wv[j][3] = bf16_bits_to_f32(q.y >> 16);
            }
#pragma unroll
            for (int f = 0; f < 4; ++f)  // ascending feature order
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(xv[i][f], wv[j][f], acc[i][j]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();

#pragma unroll
    for (int i = 0; i < TM; ++i) {
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int e = eb + b + 4 * j;
            float z = acc[i][j];
            if (p.bias != nullptr && e < p.E) z = z + p.bias[e];
            lg[(tb + a + 8 * i) * (BE + 1) + e] = z;
        }
    }
    __syncthreads();
    select_topk<BE, NW>(p, lg, t0, BT, warp, lane);
}

template <int TM, int TN, int WE, int WT, int kBK>
cudaError_t launch_variant(const RouteParams &p, cudaStream_t s)
{
    constexpr int NT = 32 * WE * WT;
    constexpr int BT = WT * 8 * TM;
    constexpr int BE = WE * 4 * TN;
    constexpr size_t stage = sizeof(float) * (kBK + 4) * (BT + BE);
    constexpr size_t logits = sizeof(float) * BT * (BE + 1);
    constexpr size_t smem = stage > logits ? stage : logits;
    struct Tag {};
    const cudaError_t e = once_per_device<Tag>([](int) {
        return cudaFuncSetAttribute(route_kernel<TM, TN, WE, WT, kBK>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    });
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>((p.T + BT - 1) / BT);
    return launch_pdl(route_kernel<TM, TN, WE, WT, kBK>, dim3(grid), dim3(NT), smem, s, p);
}

template <int TM, int TN, int WE, int WT, int KB, int STAGES>
cudaError_t launch_variant_async(const RouteParams &p, cudaStream_t s)
{
    constexpr int NT = 32 * WE * WT;
    constexpr int BT = WT * 8 * TM;
    constexpr int BE = WE * 4 * TN;
    constexpr size_t stage = sizeof(uint16_t) * STAGES * (BT + BE) * (KB + 8);
    constexpr size_t logits = sizeof(float) * BT * (BE + 1);
    constexpr size_t smem = stage > logits ? stage : logits;
    struct Tag {};
    const cudaError_t e = once_per_device<Tag>([](int) {
        return cudaFuncSetAttribute(route_kernel_async<TM, TN, WE, WT, KB, STAGES>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    });
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>((p.T + BT - 1) / BT);
    return launch_pdl(route_kernel_async<TM, TN, WE, WT, KB, STAGES>, dim3(grid), dim3(NT), smem, s, p);
}

// Mixed-precision FMA: d = a * b + c with a and b bf16 and c, d fp32. The
// product of two bf16 values is exact in fp32 and the sum is rounded once
// (round to nearest even), so the result equals fmaf on the widened operands
// bit for bit, subnormals included; it saves the widening instructions and
// lets x and the router weights stay bf16 in shared memory (PTX ISA, "fma",
// mixed-precision form with .f32 destination and .bf16 sources).
__device__ __forceinline__ float fma_bf16(uint16_t a, uint16_t b, float c)
{
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(c) : "h"(a), "h"(b));
    return c;
}

// Half g (0..7, ascending feature) of eight packed bf16 values.
__device__ __forceinline__ uint16_t bf16_half(const uint4 &q, int g)
{
    const uint32_t w = g < 2 ? q.x : g < 4 ? q.y : g < 6 ? q.z : q.w;
    return static_cast<uint16_t>((g & 1) ? (w >> 16) : (w & 0xFFFFu));
}

// Large expert counts (E > 128) and the 33..64 range: the router is bound by
// the fp32 FMA issue rate and, with fp32 tiles, by shared-memory bandwidth.
// Same thread layout and accumulation order as route_kernel, but x and the
// weights stay raw bf16 (16-byte cp.async, zero-filled past the end) in an
// S-deep ring of kBK-feature chunks and feed fma_bf16: half the shared-memory
// bytes per value and no widening pass. TM <= 6 fits three blocks per SM.
template <int TM, int TN, int WE, int WT, int kBK, int S>
__global__ void __launch_bounds__(32 * WE * WT, TM <= 6 ? 3 : 2) route_kernel_bf16(const RouteParams p)
{
    constexpr int NT = 32 * WE * WT;
    constexpr int BT = WT * 8 * TM;  // tokens per block
    constexpr int BE = WE * 4 * TN;  // experts per block (>= E)
    constexpr int NW = NT / 32;
    constexpr int RLD = kBK + 8;     // padded bf16 row: 16-byte aligned, rows 4 banks apart
    constexpr int CPR = kBK / 8;     // 16-byte pieces per row
    constexpr int ROWS = BT + BE;
    extern __shared__ __align__(16) float rsm[];
    uint16_t *raw = reinterpret_cast<uint16_t *>(rsm);  // [S][ROWS][RLD]
    float *lg = rsm;                                     // [BT][BE + 1] after the K loop
    pdl_wait();
    pdl_trigger();

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int a = lane & 7, b = lane >> 3;
    const int eb = (warp % WE) * 4 * TN, tb = (warp / WE) * 8 * TM;
    const long t0 = static_cast<long>(blockIdx.x) * BT;
    const int nchunks = (p.d + kBK - 1) / kBK;

    auto issue = [&](int chunk) {
        const int k0 = chunk * kBK;
        uint16_t *st = raw + (chunk % S) * ROWS * RLD;
        for (int v = tid; v < ROWS * CPR; v += NT) {
            const int r = v / CPR, c8 = (v % CPR) * 8;
            const bool is_x = r < BT;
            const long row = is_x ? t0 + r : static_cast<long>(r - BT);
            const bool ok = k0 + c8 < p.d && (is_x ? row < p.T : row < p.E);
            const uint16_t *src = is_x ? p.x + (ok ? row * p.d + k0 + c8 : 0)
                                       : p.wr + (ok ? row * p.d + k0 + c8 : 0);
            cp_async_16(st + r * RLD + c8, src, ok);
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

#pragma unroll
    for (int c = 0; c < S - 1; ++c) {
        if (c < nchunks) issue(c);
        cp_async_commit();
    }
    for (int c = 0; c < nchunks; ++c) {
        cp_async_wait<S - 2>();
        __syncthreads();  // chunk c landed for every thread; chunk c - 1's slot is free
        if (c + S - 1 < nchunks) issue(c + S - 1);
        cp_async_commit();
        const uint16_t *st = raw + (c % S) * ROWS * RLD;
        const uint16_t *xs = st + (tb + a) * RLD;
        const uint16_t *ws = st + (BT + eb + b) * RLD;
#pragma unroll 1
        for (int kk = 0; kk < kBK; kk += 8) {
            uint4 xq[TM], wq[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) xq[i] = *reinterpret_cast<const uint4 *>(xs + 8 * i * RLD + kk);
#pragma unroll
            for (int j = 0; j < TN; ++j) wq[j] = *reinterpret_cast<const uint4 *>(ws + 4 * j * RLD + kk);
#pragma unroll
            for (int g = 0; g < 8; ++g)  // ascending feature order for every accumulator
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const uint16_t xh = bf16_half(xq[i], g);
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fma_bf16(xh, bf16_half(wq[j], g), acc[i][j]);
                }
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // every thread is done with the ring before the logits overwrite it

#pragma unroll
    for (int i = 0; i < TM; ++i) {
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int e = eb + b + 4 * j;
            float z = acc[i][j];
            if (p.bias != nullptr && e < p.E) z = z + p.bias[e];
            lg[(tb + a + 8 * i) * (BE + 1) + e] = z;
        }
    }
    __syncthreads();
    select_topk<BE, NW>(p, lg, t0, BT, warp, lane);
}

template <int TM, int TN, int WE, int WT, int kBK, int S>
struct Bf16Variant {
    static constexpr int NT = 32 * WE * WT;
    static constexpr int BT = WT * 8 * TM;
    static constexpr int BE = WE * 4 * TN;
    static constexpr size_t tiles = sizeof(uint16_t) * S * (BT + BE) * (kBK + 8);
    static constexpr size_t logits = sizeof(float) * BT * (BE + 1);
    static constexpr size_t smem = tiles > logits ? tiles : logits;

    // once per device: the shared-memory attribute, and how many blocks fit
    // on an SM (registers and shared memory); 0 when the setup failed
    static int blocks_per_sm()
    {
        struct Tag {};
        static int occ[kOnceDevices];
        const cudaError_t e = once_per_device<Tag>([](int dev) {
            cudaError_t err = cudaFuncSetAttribute(route_kernel_bf16<TM, TN, WE, WT, kBK, S>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
            if (err != cudaSuccess) return err;
            int n = 0;
            err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, route_kernel_bf16<TM, TN, WE, WT, kBK, S>, NT,
                                                                smem);
            if (err == cudaSuccess && dev >= 0 && dev < kOnceDevices) occ[dev] = n;
            return err;
        });
        if (e != cudaSuccess) return 0;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kOnceDevices) return 1;
        return occ[dev];
    }

    static cudaError_t launch(const RouteParams &p, cudaStream_t s)
    {
        if (blocks_per_sm() <= 0) {
            const cudaError_t e = cudaGetLastError();
            return e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
        }
        const unsigned grid = static_cast<unsigned>((p.T + BT - 1) / BT);
        return launch_pdl(route_kernel_bf16<TM, TN, WE, WT, kBK, S>, dim3(grid), dim3(NT), smem, s, p);
    }
};

// Top-k and softmax of one token whose BE logits sit in the calling lane,
// giving exactly what select_topk gives for them: the arg-max with ties to
// the lower index is unique for finite logits whatever the scan order, and
// the exponential sum pairs the same terms as select_topk's butterfly (xor
// distances 16, 8, 4, 2, 1 over lanes j < k holding choice j: the steps at
// distance 16 and 8 add exact zeros or pair j with j + 8, then j + 4, j + 2,
// j + 1), so every rounding matches.
template <int BE>
__device__ __forceinline__ void select_topk_lane(const RouteParams &p, const float *z, long t)
{
    static_assert(BE == 8 || BE == 16, "the pairing below covers up to 16 logits");
    uint32_t avail = p.E >= 32 ? 0xFFFFFFFFu : (1u << p.E) - 1u;
    float ev[16];
    float zmax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) ev[j] = 0.0f;
#pragma unroll
    for (int j = 0; j < BE; ++j) {
        if (j < p.k) {
            float bv = -FLT_MAX;
            int be = -1;
#pragma unroll
            for (int e = 0; e < BE; ++e)
                if (((avail >> e) & 1u) && (be < 0 || z[e] > bv)) {
                    bv = z[e];
                    be = e;
                }
            avail &= ~(1u << be);
            if (j == 0) zmax = bv;
            ev[j] = expf(bv - zmax);
            p.idx[t * p.k + j] = be;
        }
    }
    float s8[8], s4[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s8[i] = ev[i] + ev[i + 8];
#pragma unroll
    for (int i = 0; i < 4; ++i) s4[i] = s8[i] + s8[i + 4];
    const float den = (s4[0] + s4[2]) + (s4[1] + s4[3]);
#pragma unroll
    for (int j = 0; j < BE; ++j)
        if (j < p.k) p.gate[t * p.k + j] = ev[j] / den;
}

// E <= 16 with a short feature dimension (the weights fit in shared memory):
// the block keeps all router weights resident (bf16, rows padded by 16
// bytes) for its whole life, and each warp runs its own cp.async ring over
// BT-token tasks b + G * (w + NWARP * i) of a grid of G blocks (BT = 8 TM),
// so no block barrier sits in the main loop and every SM's warps share out
// the tasks. Lane (a, b) = (lane & 7, lane >> 3) owns tokens a + 8i (i < TM)
// and experts b + 4j (j < BE / 4): each value read from shared memory feeds
// several FMAs. The BE logits of a token meet in a per-warp buffer, then the
// token's lane selects.
template <int BE, int TM, int NWARP, int KB, int STAGES>
__global__ void __launch_bounds__(32 * NWARP, 1) route_kernel_resident(const RouteParams p)
{
    constexpr int TN = BE / 4;    // experts per lane
    constexpr int BT = 8 * TM;    // tokens per task
    constexpr int NT = 32 * NWARP;
    constexpr int XLD = KB + 8;   // padded bf16 row of x
    constexpr int CPR = KB / 8;
    constexpr int RING = STAGES * BT * XLD;
    extern __shared__ __align__(16) float rsm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int la = lane & 7, lb = lane >> 3;
    const int nchunks = (p.d + KB - 1) / KB;
    const int WLD = nchunks * KB + 8;                                // padded bf16 weight row, zero past d
    uint16_t *wsb = reinterpret_cast<uint16_t *>(rsm);               // [BE][WLD]
    float *lg = rsm + BE * WLD / 2 + warp * BT * (BE + 1);           // [BT][BE + 1] per warp
    uint16_t *ring = reinterpret_cast<uint16_t *>(rsm + BE * WLD / 2 + NWARP * BT * (BE + 1)) + warp * RING;
    pdl_wait();
    pdl_trigger();

    const long ntasks = (p.T + BT - 1) / BT;
    const long G = gridDim.x;
    const long stride = G * NWARP;
    const long first = blockIdx.x + G * warp;
    const long my_tasks = first < ntasks ? (ntasks - 1 - first) / stride + 1 : 0;
    const long nq = my_tasks * nchunks;  // this warp's chunks, task after task
    auto issue = [&](long q) {
        const long t0 = (first + (q / nchunks) * stride) * BT;
        const int k0 = static_cast<int>(q % nchunks) * KB;
        uint16_t *st = ring + static_cast<int>(q % STAGES) * BT * XLD;
#pragma unroll
        for (int v = lane; v < BT * CPR; v += 32) {
            const int r = v / CPR, c8 = (v % CPR) * 8;
            const long row = t0 + r;
            const bool ok = k0 + c8 < p.d && row < p.T;
            cp_async_16(st + r * XLD + c8, p.x + (ok ? row * p.d + k0 + c8 : 0), ok);
        }
    };
#pragma unroll
    for (int q = 0; q < STAGES - 1; ++q) {
        if (q < nq) issue(q);
        cp_async_commit();
    }
    // the weights, eight 16-byte loads in flight per thread before any store
    {
        const int rowv = WLD / 8, nv = BE * rowv;
        for (int v0 = 0; v0 < nv; v0 += 8 * NT) {
            uint4 w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int v = v0 + u * NT + tid;
                const int e = v / rowv, c = (v % rowv) * 8;
                w[u] = make_uint4(0u, 0u, 0u, 0u);
                if (v < nv && e < p.E && c < p.d)
                    w[u] = *reinterpret_cast<const uint4 *>(p.wr + static_cast<long>(e) * p.d + c);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int v = v0 + u * NT + tid;
                if (v < nv) {
                    const int e = v / rowv, c = (v % rowv) * 8;
                    *reinterpret_cast<uint4 *>(wsb + e * WLD + c) = w[u];
                }
            }
        }
    }
    __syncthreads();

    float acc[TM][TN];
    for (long q = 0; q < nq; ++q) {
        const int c = static_cast<int>(q % nchunks);
        if (c == 0) {
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;
        }
        cp_async_wait<STAGES - 2>();
        __syncwarp();  // chunk q landed for every lane; chunk q - 1's slot is free
        if (q + STAGES - 1 < nq) issue(q + STAGES - 1);
        cp_async_commit();
        const uint16_t *xs = ring + static_cast<int>(q % STAGES) * BT * XLD + la * XLD;
        const uint16_t *wc = wsb + lb * WLD + c * KB;
#pragma unroll 2
        for (int kk = 0; kk < KB; kk += 8) {
            uint4 xq[TM], wq[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) xq[i] = *reinterpret_cast<const uint4 *>(xs + 8 * i * XLD + kk);
#pragma unroll
            for (int j = 0; j < TN; ++j) wq[j] = *reinterpret_cast<const uint4 *>(wc + 4 * j * WLD + kk);
#pragma unroll
            for (int g = 0; g < 8; ++g)  // ascending feature order
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const uint16_t xh = bf16_half(xq[i], g);
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fma_bf16(xh, bf16_half(wq[j], g), acc[i][j]);
                }
        }
        if (c == nchunks - 1) {
            const long t0 = (first + (q / nchunks) * stride) * BT;
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) lg[(la + 8 * i) * (BE + 1) + lb + 4 * j] = acc[i][j];
            __syncwarp();
            const long t = t0 + lane;
            if (lane < BT && t < p.T) {
                float z[BE];
#pragma unroll
                for (int e = 0; e < BE; ++e) {
                    z[e] = lg[lane * (BE + 1) + e];
                    if (p.bias != nullptr && e < p.E) z[e] = z[e] + p.bias[e];
                }
                select_topk_lane<BE>(p, z, t);
            }
            __syncwarp();  // the buffer is rewritten by the next task
        }
    }
    cp_async_wait<0>();
}

// Shared memory of route_kernel_resident for d features; 0 when it does not
// fit in one block.
template <int BE, int TM, int NWARP, int KB, int STAGES>
size_t resident_smem(int d)
{
    const size_t nchunks = (static_cast<size_t>(d) + KB - 1) / KB;
    const size_t bytes = sizeof(uint16_t) * BE * (nchunks * KB + 8) + sizeof(float) * NWARP * 8 * TM * (BE + 1) +
                         sizeof(uint16_t) * NWARP * STAGES * 8 * TM * (KB + 8);
    return bytes <= kMaxSmemPerBlock ? bytes : 0;
}

template <int BE, int TM, int NWARP, int KB, int STAGES>
cudaError_t launch_resident(const RouteParams &p, size_t smem, cudaStream_t s)
{
    struct Tag {};
    const cudaError_t e = once_per_device<Tag>([](int) {
        return cudaFuncSetAttribute(route_kernel_resident<BE, TM, NWARP, KB, STAGES>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMaxSmemPerBlock));
    });
    if (e != cudaSuccess) return e;
    const long ntasks = (p.T + 8L * TM - 1) / (8L * TM);
    const long sms = device_sm_count() > 0 ? device_sm_count() : 1;
    const unsigned grid = static_cast<unsigned>(ntasks < sms ? ntasks : sms);
    return launch_pdl(route_kernel_resident<BE, TM, NWARP, KB, STAGES>, dim3(grid), dim3(32 * NWARP), smem, s,
                      p);
}

}  // namespace

cudaError_t launch_route(const RouteArgs &a, cudaStream_t s)
{
    if (a.T == 0) return cudaSuccess;
    RouteParams p{a.x, a.wr, a.bias, a.topk_idx, a.topk_gate, a.T, a.d, a.E, a.k};
    // a block covers every expert (BE = 4*WE*TN >= E) and BT = 8*WT*TM tokens
    // <TM, TN, WE, WT, chunk>: measured best per expert count on GB300
    if (a.E > 128) {
        // BE 256 as 4 warps x 4 expert lanes x 16 experts per thread (128
        // threads), TM tokens per thread. The token tile (8 * TM tokens) is
        // the one whose last wave of blocks is fullest, counting the blocks
        // that fit on an SM for each tile (TM <= 6 keeps to ~170 registers,
        // so three blocks fit; TM 7-8 take up to 255, two blocks), slightly
        // favouring larger tiles (more reuse of each staged feature chunk).
        const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
        const int occ[5] = {Bf16Variant<4, 16, 4, 1, 32, 3>::blocks_per_sm(),
                            Bf16Variant<5, 16, 4, 1, 32, 3>::blocks_per_sm(),
                            Bf16Variant<6, 16, 4, 1, 32, 3>::blocks_per_sm(),
                            Bf16Variant<7, 16, 4, 1, 32, 3>::blocks_per_sm(),
                            Bf16Variant<8, 16, 4, 1, 32, 3>::blocks_per_sm()};
        int best_tm = 8;
        double best = -1.0;
        for (int tm = 8; tm >= 4; --tm) {
            const long slots = static_cast<long>(occ[tm - 4] > 0 ? occ[tm - 4] : 1) * sms;
            const long blocks = (a.T + 8L * tm - 1) / (8L * tm);
            const long waves = (blocks + slots - 1) / slots;
            const double score = static_cast<double>(blocks) / (waves * slots) * (1.0 - 0.02 * (8 - tm));
            if (score > best) {
                best = score;
                best_tm = tm;
            }
        }
        switch (best_tm) {
        case 7: return Bf16Variant<7, 16, 4, 1, 32, 3>::launch(p, s);
        case 6: return Bf16Variant<6, 16, 4, 1, 32, 3>::launch(p, s);
        case 5: return Bf16Variant<5, 16, 4, 1, 32, 3>::launch(p, s);
        case 4: return Bf16Variant<4, 16, 4, 1, 32, 3>::launch(p, s);
        default: return Bf16Variant<8, 16, 4, 1, 32, 3>::launch(p, s);
        }
    }
    if (a.E > 64) return launch_variant<2, 8, 4, 2, 64>(p, s);                  // BT 32, BE 128
    if (a.E > 32) return Bf16Variant<2, 2, 8, 1, 64, 4>::launch(p, s);        // BT 16, BE 64
    if (a.E > 16) return launch_variant<2, 2, 4, 2, 128>(p, s);                 // BT 32, BE 32
    if (a.E > 8) {
        // resident weights while they fit next to eight warps' rings
        if (const size_t smem = resident_smem<16, 4, 8, 64, 4>(a.d))
            return launch_resident<16, 4, 8, 64, 4>(p, smem, s);
        return launch_variant<2, 4, 1, 8, 128>(p, s);                           // BT 128, BE 16
    }
    // E <= 8: resident weights, 8-token tasks (enough tasks for every SM even
    // at a few thousand tokens) while they fit next to sixteen warps' rings
    if (const size_t smem = resident_smem<8, 1, 16, 64, 8>(a.d)) return launch_resident<8, 1, 16, 64, 8>(p, smem, s);
    return launch_variant_async<1, 1, 2, 4, 128, 4>(p, s);                      // BT 32, BE 8
}

}  // namespace moe
