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
// expert GEMMs). Each logit is accumulated by ONE thread in ascending i with
// fmaf: every bf16 x bf16 product is exact in fp32, so the result is the fp32
// sequential sum, rounded once per addition, independent of the tiling. The
// selection is therefore reproducible bit for bit by any implementation of
// that sum.
//
// Block tile: BT tokens x BE >= E experts, staged through shared memory a
// chunk of features at a time as fp32 rows (the next chunk is prefetched into registers
// while the current one is used), each thread owning TM tokens x TN experts.
// Then one warp per token runs k rounds of a shuffle arg-max over the block's
// logits and writes idx and gates.
#include <cuda_bf16.h>
#include <float.h>

#include "kernels.cuh"

namespace moe {
namespace {


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

// Large expert counts (E > 128), where the router is bound by the fp32 FMA
// rate. Same thread layout and accumulation as route_kernel, but the staging
// holds no registers: each chunk of kBK features is copied raw (bf16, 16-byte
// cp.async, zero-filled past the end) into a shared-memory buffer while the
// previous chunk is in use, then all threads widen it into the fp32 tiles in
// one pass. The registers this frees let three blocks share an SM for the
// smaller token tiles, and the FMAs of a 4-feature step run feature by
// feature over the whole TM x TN tile, so consecutive FMAs never depend on
// each other.
template <int TM, int TN, int WE, int WT, int kBK>
__global__ void __launch_bounds__(32 * WE * WT, TM <= 6 ? 3 : 2) route_kernel_cvt(const RouteParams p)
{
    constexpr int NT = 32 * WE * WT;
    constexpr int BT = WT * 8 * TM;  // tokens per block
    constexpr int BE = WE * 4 * TN;  // experts per block (>= E)
    constexpr int NW = NT / 32;
    constexpr int LD = kBK + 4;      // padded fp32 row (floats)
    constexpr int RLD = kBK + 8;     // padded raw row (bf16): 16-byte aligned rows
    constexpr int CPR = kBK / 8;     // 16-byte pieces per row
    constexpr int ROWS = BT + BE;
    extern __shared__ __align__(16) float rsm[];
    float *xs = rsm;                                                // [BT][LD]
    float *ws = rsm + BT * LD;                                      // [BE][LD]
    uint16_t *raw = reinterpret_cast<uint16_t *>(rsm + ROWS * LD);  // [ROWS][RLD]
    float *lg = rsm;                                                // [BT][BE + 1] after the K loop
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
        for (int v = tid; v < ROWS * CPR; v += NT) {
            const int r = v / CPR, c8 = (v % CPR) * 8;
            const bool is_x = r < BT;
            const long row = is_x ? t0 + r : static_cast<long>(r - BT);
            const bool ok = k0 + c8 < p.d && (is_x ? row < p.T : row < p.E);
            const uint16_t *src = is_x ? p.x + (ok ? row * p.d + k0 + c8 : 0)
                                       : p.wr + (ok ? row * p.d + k0 + c8 : 0);
            cp_async_16(raw + r * RLD + c8, src, ok);
        }
    };
    auto widen_chunk = [&]() {
        const uint16_t *st = raw;
        for (int v = tid; v < ROWS * CPR; v += NT) {
            const int r = v / CPR, c8 = (v % CPR) * 8;
            const uint4 q = *reinterpret_cast<const uint4 *>(st + r * RLD + c8);
            float *dst = r < BT ? xs + r * LD + c8 : ws + (r - BT) * LD + c8;
            *reinterpret_cast<float4 *>(dst) =
                make_float4(bf16_bits_to_f32(q.x & 0xFFFFu), bf16_bits_to_f32(q.x >> 16),
                            bf16_bits_to_f32(q.y & 0xFFFFu), bf16_bits_to_f32(q.y >> 16));
            *reinterpret_cast<float4 *>(dst + 4) =
                make_float4(bf16_bits_to_f32(q.z & 0xFFFFu), bf16_bits_to_f32(q.z >> 16),
                            bf16_bits_to_f32(q.w & 0xFFFFu), bf16_bits_to_f32(q.w >> 16));
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

    issue(0);
    cp_async_commit();
    for (int c = 0; c < nchunks; ++c) {
        cp_async_wait<0>();  // chunk c has landed (the only copies in flight)
        __syncthreads();     // ... for every thread, and chunk c - 1's tiles are no longer read
        widen_chunk();
        __syncthreads();     // tiles of chunk c ready; the raw buffer is free again
        if (c + 1 < nchunks) issue(c + 1);  // lands while chunk c is used
        cp_async_commit();
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
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(xv[i].x, wv[j].x, acc[i][j]);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(xv[i].y, wv[j].y, acc[i][j]);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(xv[i].z, wv[j].z, acc[i][j]);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(xv[i].w, wv[j].w, acc[i][j]);
        }
    }
    __syncthreads();  // every thread is done with the tiles before the logits overwrite them

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
struct CvtVariant {
    static constexpr int NT = 32 * WE * WT;
    static constexpr int BT = WT * 8 * TM;
    static constexpr int BE = WE * 4 * TN;
    static constexpr size_t tiles =
        sizeof(float) * (kBK + 4) * (BT + BE) + sizeof(uint16_t) * (BT + BE) * (kBK + 8);
    static constexpr size_t logits = sizeof(float) * BT * (BE + 1);
    static constexpr size_t smem = tiles > logits ? tiles : logits;

    // once per device: the shared-memory attribute, and how many blocks fit
    // on an SM (registers and shared memory); 0 when the setup failed
    static int blocks_per_sm()
    {
        struct Tag {};
        static int occ[kOnceDevices];
        const cudaError_t e = once_per_device<Tag>([](int dev) {
            cudaError_t err = cudaFuncSetAttribute(route_kernel_cvt<TM, TN, WE, WT, kBK>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
            if (err != cudaSuccess) return err;
            int n = 0;
            err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, route_kernel_cvt<TM, TN, WE, WT, kBK>, NT,
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
        return launch_pdl(route_kernel_cvt<TM, TN, WE, WT, kBK>, dim3(grid), dim3(NT), smem, s, p);
    }
};

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
        // that fit on an SM for each tile (TM <= 6 needs ~170 registers, so
        // three blocks fit; TM 7-8 take up to 255, two blocks), slightly
        // favouring larger tiles (more reuse of each staged feature chunk).
        const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
        const int occ[5] = {CvtVariant<4, 16, 4, 1, 32>::blocks_per_sm(), CvtVariant<5, 16, 4, 1, 32>::blocks_per_sm(),
                            CvtVariant<6, 16, 4, 1, 32>::blocks_per_sm(), CvtVariant<7, 16, 4, 1, 32>::blocks_per_sm(),
                            CvtVariant<8, 16, 4, 1, 32>::blocks_per_sm()};
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
        case 7: return CvtVariant<7, 16, 4, 1, 32>::launch(p, s);
        case 6: return CvtVariant<6, 16, 4, 1, 32>::launch(p, s);
        case 5: return CvtVariant<5, 16, 4, 1, 32>::launch(p, s);
        case 4: return CvtVariant<4, 16, 4, 1, 32>::launch(p, s);
        default: return CvtVariant<8, 16, 4, 1, 32>::launch(p, s);
        }
    }
    if (a.E > 64) return launch_variant<2, 8, 4, 2, 64>(p, s);    // BT 32, BE 128
    if (a.E > 32) return launch_variant_async<2, 4, 4, 1, 128, 4>(p, s);  // BT 16, BE 64
    if (a.E > 16) return launch_variant<2, 2, 4, 2, 128>(p, s);           // BT 32, BE 32
    if (a.E > 8) return launch_variant<2, 4, 1, 8, 128>(p, s);            // BT 128, BE 16
    return launch_variant_async<1, 1, 2, 4, 128, 4>(p, s);                // BT 32, BE 8
}

}  // namespace moe
