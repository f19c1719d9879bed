// route_tc.cu -- the router of moe_layer_forward, filter then verify (Cui et
// al., "Fine-grained Computation-Communication Overlap ...", section 2.1
// step 1). It returns exactly what route.cu returns -- the top-k of the fp32
// logits summed in ascending feature order, ties to the lower expert, and the
// softmax of those k logits -- but sums exactly only the experts that can
// still be among the top k:
//
//   1. route_wnorm_kernel: the squared norm of every router weight row.
//   2. route_cand_kernel: the tensor cores compute every logit approximately
//      (bf16 operands, fp32 accumulation in the tensor core's own order) while
//      the epilogue warps take the squared norm of each token row from the
//      staged x tiles. For token t and expert e the approximation and the
//      exact sequential sum both lie within gamma * sum_i |x_ti w_ei| of the
//      real dot product, and sum_i |x_ti w_ei| <= |x_t| |w_e| (Cauchy-Schwarz),
//      so with B = gamma |x_t| |w_e| (plus the roundings of the bias addition)
//      the exact logit lies in [z~ - B, z~ + B]. An expert whose upper end is
//      below the k-th largest lower end has k experts strictly above it and
//      cannot be selected; the others ("candidates", about 15 of 256 on
//      random data) are listed per token in ascending expert order.
//   3. route_exact_kernel: CUDA cores sum the candidates' logits exactly, the
//      same fused multiply-add per feature in ascending order as route.cu, and
//      select among them (ties to the lower expert; the exponential sum paired
//      as route.cu's warp butterfly pairs it).
//   4. route_full_kernel: tokens with more than kMaxCand candidates (exact
//      ties, rows of zeros, huge values) get every expert's exact logit and the
//      same warp selection as route.cu.
//
// The error bound: every step of the sequential fp32 sum rounds once with
// relative error at most u = 2^-24, so the sum is within gamma_d(u) *
// sum |x w| of the real value (gamma_n(u) = n u / (1 - n u)). The tensor
// core's internal order and rounding are not published; its accumulation is
// taken as d steps each with relative error at most 2^-21 (8 u). Even if each
// K = 16 step truncated all 16 products and the accumulator to 24 bits of the
// largest of them, the error would stay under 17/16 * d * 2^-23 * sum |x w|,
// a quarter of that allowance; on the fine-grained workload's inputs the
// largest measured difference between the two sums is 0.0023 d 2^-24
// sum |x w|. The norms are inflated by 1/256 for their own rounding.
#include <float.h>
#include <limits.h>
#include <math.h>

#include <cmath>

#include "kernels.cuh"
#include "sm100.cuh"

namespace moe {
namespace {

constexpr int kCandM = 128;        // tokens per CTA of the candidate kernel (the MMA's M)
constexpr int kCandK = 64;         // features per stage: one 128-byte swizzle row of bf16
constexpr int kCandStages = 4;
constexpr int kCandSlices = 4;     // epilogue warps per 32-lane quarter of tensor memory
constexpr int kCandEpiWarps = 4 * kCandSlices;
constexpr int kCandThreads = 64 + 32 * kCandEpiWarps;  // warp 0 TMA, warp 1 MMA, then the epilogue
constexpr int kCandSliceCols = 256 / kCandSlices;
constexpr int kCandATile = kCandM * kCandK * 2;
constexpr int kCandBTile = 256 * kCandK * 2;
constexpr int kMaxCand = 64;       // candidates kept per token
constexpr uint8_t kOverflow = 255; // candidate count of a token on the full path
constexpr int kExactMaxBT = 128;   // tokens per block of the exact kernel
constexpr int kFullThreads = 256;
constexpr unsigned long long kCandWaitNs = 2000000000ull;
constexpr unsigned long long kDrainNs = 50000000ull;
constexpr size_t kSmemLimit = 232448;

struct FastParams {
    const uint16_t *x;
    const uint16_t *wr;
    const float *bias;
    int32_t *idx;
    float *gate;
    unsigned *status;
    uint8_t *cand;   // [T][kMaxCand] candidate experts, ascending
    uint8_t *cnt;    // [T] candidate count, or kOverflow
    int32_t *ovf;    // [T] tokens on the full path
    unsigned *novf;  // their count
    float *wn2;      // [E] squared norms of the router weight rows
    int T, d, E, k, npad, bt;
    float gamma;     // gamma_d(2^-24) + gamma_d(2^-21)
    float abs_eps;   // absolute slack for products and sums near the underflow threshold
};

__device__ __forceinline__ float fma_bf16x(uint16_t a, uint16_t b, float c)
{
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(c) : "h"(a), "h"(b));
    return c;
}

__device__ __forceinline__ uint16_t half_of(const uint4 &q, int g)
{
    const uint32_t w = g < 2 ? q.x : g < 4 ? q.y : g < 6 ? q.z : q.w;
    return static_cast<uint16_t>((g & 1) ? (w >> 16) : (w & 0xFFFFu));
}

// eight features in ascending order: a = fma(x_g, w_g, a) for g = 0..7
__device__ __forceinline__ float fma8(const uint4 &xq, const uint4 &wq, float a)
{
#pragma unroll
    for (int g = 0; g < 8; ++g) a = fma_bf16x(half_of(xq, g), half_of(wq, g), a);
    return a;
}

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// Softmax denominator of the k selected logits (ev[j] = exp(z_j - z_0), zero
// past k), summed in the pairing of a 32-lane xor butterfly over lanes j < k.
__device__ __forceinline__ float butterfly_den(const float (&ev)[16])
{
    float s8[8], s4[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s8[i] = ev[i] + ev[i + 8];
#pragma unroll
    for (int i = 0; i < 4; ++i) s4[i] = s8[i] + s8[i + 4];
    return (s4[0] + s4[2]) + (s4[1] + s4[3]);
}

// ------------------------------------------------------------ weight norms
// One block per expert; block 0 also clears the full-path counter.
__global__ void __launch_bounds__(128) route_wnorm_kernel(const FastParams p)
{
    pdl_wait();
    pdl_trigger();
    __shared__ float red[4];
    const int e = blockIdx.x;
    const uint16_t *row = p.wr + static_cast<long>(e) * p.d;
    float s = 0.0f;
    for (int i = threadIdx.x * 8; i < p.d; i += 128 * 8) {
        const uint4 q = *reinterpret_cast<const uint4 *>(row + i);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const float v = bf16f(half_of(q, g));
            s = fmaf(v, v, s);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        p.wn2[e] = (red[0] + red[1]) + (red[2] + red[3]);
        if (e == 0) *p.novf = 0u;
    }
}

// ------------------------------------------------------------ candidates
struct CandSmem {
    uint64_t full[kCandStages];
    uint64_t empty[kCandStages];
    uint64_t tfull;
    uint64_t drain;
    uint64_t epi;  // the epilogue warps' barrier: one arrival per warp, bounded waits
    uint32_t tmem_base;
    int abort;
    float wn[256];  // |w_e| (inflated)
    float bias[256];
    // per token row and column slice: partial squared norm, the slice's
    // kMaxTopK largest lower ends, its candidate count and sanity
    float sq[kCandSlices][kCandM];
    float top[kCandSlices][kCandM][kMaxTopK];
    int ncand[kCandSlices][kCandM];
    int insane[kCandSlices][kCandM];
};

// Barrier among the candidate kernel's epilogue warps on an mbarrier (phase
// parity `ph`): each warp reconverges, lane 0 arrives, every lane waits with
// the usual limit. Returns false (the CTA's abort flag raised) if it gave up.
__device__ __forceinline__ bool epi_barrier(CandSmem &c, uint32_t ph, volatile int *abort_flag, unsigned *status,
                                            int lane)
{
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.epi);
    const bool ok = mbar_wait(&c.epi, ph, abort_flag, status, kWhereRouteTc, 10u + ph, kCandWaitNs);
    return __all_sync(0xffffffffu, ok);
}

__global__ void __launch_bounds__(kCandThreads, 1)
route_cand_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                  const FastParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    uint8_t *sA = reinterpret_cast<uint8_t *>(base);
    uint8_t *sB = sA + kCandStages * kCandATile;
    CandSmem &c = *reinterpret_cast<CandSmem *>(sB + kCandStages * kCandBTile);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkb = (p.d + kCandK - 1) / kCandK;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kCandStages; ++s) {
            mbar_init(&c.full[s], 1);
            mbar_init(&c.empty[s], 1 + kCandEpiWarps);  // the MMAs' commit and every epilogue warp
        }
        mbar_init(&c.tfull, 1);
        mbar_init(&c.drain, 1);
        mbar_init(&c.epi, kCandEpiWarps);
        c.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    // the weight norms come from the kernel before; tensor memory is taken
    // only once every earlier kernel on the stream has finished
    pdl_wait();
    pdl_trigger();
    if (warp == 1) {
        tmem_alloc<1>(&c.tmem_base, 256);
        tmem_relinquish<1>();
    }
    for (int e = threadIdx.x; e < 256; e += kCandThreads) {
        c.wn[e] = e < p.E ? sqrtf(p.wn2[e] * (1.0f + 1.0f / 256.0f)) : 0.0f;
        c.bias[e] = (e < p.E && p.bias != nullptr) ? p.bias[e] : 0.0f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;
    volatile int *abort_flag = &c.abort;
    const int t0 = blockIdx.x * kCandM;

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t bytes = kCandATile + static_cast<uint32_t>(p.npad) * kCandK * 2;
            int issued = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kCandStages;
                const uint32_t ph = static_cast<uint32_t>(kb / kCandStages) & 1u;
                if (!mbar_wait(&c.empty[s], ph ^ 1u, abort_flag, p.status, kWhereRouteTc, 1u, kCandWaitNs))
                    break;
                mbar_arrive_expect_tx(&c.full[s], bytes);
                const uint32_t bar = smem_u32(&c.full[s]);
                tma_load_2d<1>(&tm_x, bar, sA + s * kCandATile, kb * kCandK, t0);
                tma_load_2d<1>(&tm_w, bar, sB + s * kCandBTile, kb * kCandK, 0);
                ++issued;
            }
            // every load issued has landed before the CTA can exit, also when a
            // consumer gave up waiting for it (only the last kCandStages can
            // still be in flight; their phases have completed otherwise)
            for (int i = issued > kCandStages ? issued - kCandStages : 0; i < issued; ++i)
                if (!mbar_wait_drain(&c.full[i % kCandStages], static_cast<uint32_t>(i / kCandStages) & 1u,
                                     kDrainNs))
                    report_failure(p.status, kStatusTimeout, kWhereRouteTc, 5u);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kCandM, p.npad);
            bool ok = true;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kCandStages;
                const uint32_t ph = static_cast<uint32_t>(kb / kCandStages) & 1u;
                if (!mbar_wait(&c.full[s], ph, abort_flag, p.status, kWhereRouteTc, 2u, kCandWaitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sA + s * kCandATile));
                const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sB + s * kCandBTile));
#pragma unroll
                for (int kk = 0; kk < kCandK / 16; ++kk)
                    mma_bf16_ss<1>(tmem, ad + 2u * kk, bd + 2u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
                mma_commit<1>(&c.empty[s]);
            }
            if (ok) {
                mma_commit<1>(&c.tfull);
            } else {
                // wait for the MMAs already issued before tensor memory is freed
                mma_commit<1>(&c.drain);
                if (!mbar_wait_drain(&c.drain, 0u, kDrainNs))
                    report_failure(p.status, kStatusTimeout, kWhereRouteTc, 6u);
            }
        }
        __syncwarp();
    } else {
        // Epilogue warp (quarter q, slice sl): token rows 32 q .. 32 q + 31 (one
        // per lane, the tensor-memory lanes this warp may read) and experts
        // [64 sl, 64 sl + 64). During the mainloop it adds the squares of its
        // rows' 16-byte pieces sl and sl + kCandSlices of each staged x tile
        // (in any order: the norm only bounds the error); lane i reads its
        // pieces at swizzled positions that differ across the quarter warp.
        const int q = warp & 3;
        const int sl = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        float sq = 0.0f;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % kCandStages;
            const uint32_t ph = static_cast<uint32_t>(kb / kCandStages) & 1u;
            const bool ready = mbar_wait(&c.full[s], ph, abort_flag, p.status, kWhereRouteTc, 3u, kCandWaitNs);
            if (!__all_sync(0xffffffffu, ready)) {
                ok = false;
                break;
            }
            const uint8_t *r = sA + s * kCandATile + row * (kCandK * 2);
#pragma unroll
            for (int j = 0; j < 8 / kCandSlices; ++j) {
                const int piece = sl + j * kCandSlices;
                const uint4 v = *reinterpret_cast<const uint4 *>(r + ((piece ^ (row & 7)) << 4));
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const float f = bf16f(half_of(v, g));
                    sq = fmaf(f, f, sq);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.empty[s]);
        }
        // a wait that gave up raised the CTA's abort flag before this barrier,
        // so every epilogue warp takes the same branch after it
        if (ok) mbar_wait(&c.tfull, 0u, abort_flag, p.status, kWhereRouteTc, 4u, kCandWaitNs);
        c.sq[sl][row] = sq;
        if (epi_barrier(c, 0u, abort_flag, p.status, lane) && *abort_flag == 0) {
            tc_fence_after();
            const long t = static_cast<long>(t0) + row;
            float sqa = 0.0f;
#pragma unroll
            for (int i = 0; i < kCandSlices; ++i) sqa += c.sq[i][row];
            const float xn = sqrtf(sqa * (1.0f + 1.0f / 256.0f));
            const float bscale = p.gamma * xn;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + sl * kCandSliceCols;
            const int e0 = sl * kCandSliceCols;
            // pass 1: this slice's kMaxTopK largest lower ends, descending
            // (starting with kMaxTopK - k entries of +inf, so the last entry
            // is the k-th largest inserted)
            float top[kMaxTopK];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) top[j] = j < kMaxTopK - p.k ? INFINITY : -INFINITY;
            float kth = -INFINITY;
            bool sane = true;
#pragma unroll
            for (int ch = 0; ch < kCandSliceCols / 32; ++ch) {
                if (e0 + ch * 32 < p.E) {
                    uint32_t v[32];
                    __syncwarp();
                    tmem_load_32cols(taddr + ch * 32, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int e = e0 + ch * 32 + j;
                        if (e < p.E) {
                            const float z = __uint_as_float(v[j]) + c.bias[e];
                            const float b = fmaf(bscale, c.wn[e], fmaf(4.8e-7f, fabsf(z), p.abs_eps));
                            // NaN fails both comparisons; b < 1e30 keeps every
                            // partial sum of both logits far from overflow
                            sane = sane && fabsf(z) < 3.0e38f && b < 1.0e30f;
                            const float lo = z - b;
                            if (lo > kth) {
                                float cur = lo;
#pragma unroll
                                for (int i = 0; i < kMaxTopK; ++i) {
                                    const float big = fmaxf(top[i], cur);
                                    cur = fminf(top[i], cur);
                                    top[i] = big;
                                }
                                kth = top[kMaxTopK - 1];
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) c.top[sl][row][j] = top[j];
            // a non-finite or huge logit or bound sends the token to the full path
            c.insane[sl][row] = !sane || !(xn < 3.0e38f);
            const bool b2 = epi_barrier(c, 1u, abort_flag, p.status, lane);
            // the k-th largest lower end over all slices (each slice's list ends
            // with its k largest; the entries before them are padding)
#pragma unroll 1
            for (int o = 0; o < kCandSlices; ++o) {
                if (o == sl) continue;
#pragma unroll 1
                for (int jj = kMaxTopK - p.k; jj < kMaxTopK; ++jj) {
                    const float lo = c.top[o][row][jj];
                    if (lo > kth) {
                        float cur = lo;
#pragma unroll
                        for (int i = 0; i < kMaxTopK; ++i) {
                            const float big = fmaxf(top[i], cur);
                            cur = fminf(top[i], cur);
                            top[i] = big;
                        }
                        kth = top[kMaxTopK - 1];
                    }
                }
            }
            // pass 2: this slice's experts whose upper end reaches it, counted,
            // then written after the earlier slices' candidates
            int n = 0;
#pragma unroll
            for (int ch = 0; ch < kCandSliceCols / 32; ++ch) {
                if (e0 + ch * 32 < p.E) {
                    uint32_t v[32];
                    __syncwarp();
                    tmem_load_32cols(taddr + ch * 32, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int e = e0 + ch * 32 + j;
                        if (e < p.E) {
                            const float z = __uint_as_float(v[j]) + c.bias[e];
                            const float b = fmaf(bscale, c.wn[e], fmaf(4.8e-7f, fabsf(z), p.abs_eps));
                            n += z + b >= kth ? 1 : 0;
                        }
                    }
                }
            }
            c.ncand[sl][row] = n;
            const bool b3 = epi_barrier(c, 0u, abort_flag, p.status, lane);
            int base_n = 0, total = 0, bad = !(b2 && b3);
#pragma unroll
            for (int i = 0; i < kCandSlices; ++i) {
                const int ni = c.ncand[i][row];
                base_n += i < sl ? ni : 0;
                total += ni;
                bad |= c.insane[i][row];
            }
            const bool over = bad || total > kMaxCand || total < p.k;
            // the tensor-memory loads are warp-wide: the whole warp runs this
            // pass when any lane writes, and only the writing lanes store
            const bool write = !over && n > 0 && t < p.T;
            if (__any_sync(0xffffffffu, write)) {
                int m = base_n;
#pragma unroll
                for (int ch = 0; ch < kCandSliceCols / 32; ++ch) {
                    if (e0 + ch * 32 < p.E) {
                        uint32_t v[32];
                        __syncwarp();
                        tmem_load_32cols(taddr + ch * 32, v);
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int e = e0 + ch * 32 + j;
                            if (e < p.E) {
                                const float z = __uint_as_float(v[j]) + c.bias[e];
                                const float b = fmaf(bscale, c.wn[e], fmaf(4.8e-7f, fabsf(z), p.abs_eps));
                                if (write && z + b >= kth) p.cand[t * kMaxCand + m++] = static_cast<uint8_t>(e);
                            }
                        }
                    }
                }
            }
            if (sl == 0 && t < p.T) {
                if (over) {
                    p.cnt[t] = kOverflow;
                    p.ovf[atomicAdd(p.novf, 1u)] = static_cast<int32_t>(t);
                } else {
                    p.cnt[t] = static_cast<uint8_t>(total);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<1>(tmem, 256);
    }
}

// ------------------------------------------------------------ exact candidates
// A block takes p.bt consecutive tokens and lists their (token, candidate)
// pairs in groups of four of one token (a token's list is padded to a
// multiple of four with copies of its first candidate, summed and dropped).
// Consumer thread i takes the i-th of kExactConsumers nearly equal contiguous
// runs of groups, so every thread does the same work whatever the candidate
// counts, and sums the four pairs of a group as four interleaved chains
// sharing the token's x. A producer warp streams x and all E router weight
// rows through a ring of S chunks of 64 features (unpadded 128-byte rows) with
// TMA; consumer warps wait on each chunk's full barrier and release a chunk
// on its empty barrier when they no longer need it, with no block-wide
// barrier between chunks.
//
// Lane l of a quarter warp (pk = l mod 8) walks the features in windows of 64
// offset by 8 pk: window w covers features [64 (w - 1) + 8 pk, 64 w + 8 pk),
// so its j-th 16-byte piece sits at position (pk + j) mod 8 of its row, and
// the eight lanes of a quarter warp always read eight different bank groups,
// whichever rows (candidate experts) they read. The windows tile the feature
// axis in ascending order, so each logit is still one fused multiply-add per
// feature in ascending order. A window needs chunks w - 1 and w resident, so
// up to S - 2 chunks are in flight.
constexpr int kExactConsumers = 384;
constexpr int kExactThreads = kExactConsumers + 32;  // + the producer warp

struct ExactBars {
    uint64_t full[4];
    uint64_t empty[4];
    int abort;
};

__host__ __device__ constexpr size_t exact_tail_bytes(int BT)
{
    // zs [BT*64] f32, pexp [BT*64] u8, ptok [BT*16] u8, qbase [BT+1] i32, then
    // the barriers (8-byte aligned)
    return (static_cast<size_t>(BT) * kMaxCand * 5 + static_cast<size_t>(BT) * (kMaxCand / 4) +
            (static_cast<size_t>(BT) + 1) * 4 + 7) / 8 * 8 +
           sizeof(ExactBars);
}

template <int S>
__global__ void __launch_bounds__(kExactThreads, 1)
route_exact_kernel(const __grid_constant__ CUtensorMap tm_xr, const __grid_constant__ CUtensorMap tm_wr,
                   const FastParams p)
{
    extern __shared__ uint8_t ex_raw[];
    uint8_t *ring_p = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(ex_raw) + 1023) & ~uintptr_t(1023));
    const int NT = blockDim.x, BT = p.bt, E = p.E;
    const uint32_t stage_bytes = static_cast<uint32_t>(BT + E) * 128u;
    const uint32_t ring = smem_u32(ring_p);
    float *zs = reinterpret_cast<float *>(ring_p + S * stage_bytes);          // [BT*64] per pair
    uint8_t *pexp = reinterpret_cast<uint8_t *>(zs + BT * kMaxCand);         // [BT*64] per pair
    uint8_t *ptok = pexp + BT * kMaxCand;                                     // [BT*16] per group
    int *qbase = reinterpret_cast<int *>(ptok + BT * (kMaxCand / 4));         // [BT+1]
    ExactBars &bars = *reinterpret_cast<ExactBars *>(
        (reinterpret_cast<uintptr_t>(qbase + BT + 1) + 7) & ~uintptr_t(7));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, pk = tid & 7;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], kExactConsumers / 32);
        }
        bars.abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_xr);
        tma_prefetch_desc(&tm_wr);
    }
    pdl_wait();
    pdl_trigger();
    const long t0 = static_cast<long>(blockIdx.x) * BT;
    // groups per token, their exclusive scan (one warp), then the pair lists
    if (tid < 32) {
        int run = 0;
        for (int j0 = 0; j0 < BT; j0 += 32) {
            const int j = j0 + tid;
            int q = 0;
            if (j < BT && t0 + j < p.T) {
                const int cn = p.cnt[t0 + j];
                q = cn == kOverflow ? 0 : (cn + 3) / 4;
            }
            int inc = q;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, inc, o);
                if (tid >= o) inc += v;
            }
            if (j < BT) qbase[j] = run + inc - q;
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (tid == 0) qbase[BT] = run;
    }
    __syncthreads();
    for (int j = tid; j < BT; j += NT) {
        const long t = t0 + j;
        const int q0 = qbase[j], nq = qbase[j + 1] - q0;
        if (nq == 0) continue;
        const int n = p.cnt[t];
        const uint8_t *cl = p.cand + t * kMaxCand;
        for (int i = 0; i < 4 * nq; ++i) {
            pexp[4 * q0 + i] = cl[i < n ? i : 0];
            zs[4 * q0 + i] = 0.0f;
        }
        for (int q = 0; q < nq; ++q) ptok[q0 + q] = static_cast<uint8_t>(j);
    }
    __syncthreads();
    const int nchunks = (p.d + 63) / 64, nsub = p.d / 8;
    volatile int *abort_flag = &bars.abort;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int ch = 0; ch < nchunks; ++ch) {
                const int s = ch % S;
                const uint32_t ph = static_cast<uint32_t>(ch / S) & 1u;
                if (!mbar_wait(&bars.empty[s], ph ^ 1u, abort_flag, p.status, kWhereRouteTc, 7u, kCandWaitNs))
                    break;
                mbar_arrive_expect_tx(&bars.full[s], stage_bytes);
                const uint32_t bar = smem_u32(&bars.full[s]);
                tma_load_2d<1>(&tm_xr, bar, ring_p + s * stage_bytes, ch * 64, static_cast<int>(t0));
                tma_load_2d<1>(&tm_wr, bar, ring_p + s * stage_bytes + BT * 128, ch * 64, 0);
                ++issued;
            }
            // every load issued has landed before the CTA can exit (see the
            // candidate kernel's producer)
            for (int i = issued > S ? issued - S : 0; i < issued; ++i)
                if (!mbar_wait_drain(&bars.full[i % S], static_cast<uint32_t>(i / S) & 1u, kDrainNs))
                    report_failure(p.status, kStatusTimeout, kWhereRouteTc, 9u);
        }
        __syncwarp();
    } else {
        const int ctid = tid - 32;
        const int Q = qbase[BT];
        const int g_begin = static_cast<int>((static_cast<long>(Q) * ctid) / kExactConsumers);
        const int g_end = static_cast<int>((static_cast<long>(Q) * (ctid + 1)) / kExactConsumers);
        for (int w = 0; w <= nchunks; ++w) {
            if (w < nchunks) {
                const bool ready = mbar_wait(&bars.full[w % S], static_cast<uint32_t>(w / S) & 1u, abort_flag,
                                             p.status, kWhereRouteTc, 8u, kCandWaitNs);
                if (!__all_sync(0xffffffffu, ready)) break;
            }
            if (g_begin < g_end) {
                const int cl = w - 1;
                const uint32_t lo = ring + static_cast<uint32_t>((cl + S) % S) * stage_bytes;
                const uint32_t hi = ring + static_cast<uint32_t>(w % S) * stage_bytes;
                uint32_t off[8];
                unsigned vmask = 0;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int q = pk + jj;
                    const int g = 8 * cl + q;
                    off[jj] = (q < 8 ? lo : hi) + static_cast<uint32_t>((q & 7) << 4);
                    vmask |= (g >= 0 && g < nsub ? 1u : 0u) << jj;
                }
                uint4 xr[8];
                int cur = -1;
                for (int gq = g_begin; gq < g_end; ++gq) {
                    const int tok = ptok[gq];
                    if (tok != cur) {
                        cur = tok;
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            xr[jj] = ((vmask >> jj) & 1u) ? lds128(off[jj] + static_cast<uint32_t>(tok) * 128u)
                                                          : make_uint4(0u, 0u, 0u, 0u);
                    }
                    const uchar4 ex4 = *reinterpret_cast<const uchar4 *>(pexp + 4 * gq);
                    const uint32_t eo[4] = {static_cast<uint32_t>(BT + ex4.x) * 128u,
                                            static_cast<uint32_t>(BT + ex4.y) * 128u,
                                            static_cast<uint32_t>(BT + ex4.z) * 128u,
                                            static_cast<uint32_t>(BT + ex4.w) * 128u};
                    float4 a = *reinterpret_cast<const float4 *>(zs + 4 * gq);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        if ((vmask >> jj) & 1u) {
                            const uint4 w0 = lds128(off[jj] + eo[0]);
                            const uint4 w1 = lds128(off[jj] + eo[1]);
                            const uint4 w2 = lds128(off[jj] + eo[2]);
                            const uint4 w3 = lds128(off[jj] + eo[3]);
#pragma unroll
                            for (int g = 0; g < 8; ++g) {
                                const uint16_t xv = half_of(xr[jj], g);
                                a.x = fma_bf16x(xv, half_of(w0, g), a.x);
                                a.y = fma_bf16x(xv, half_of(w1, g), a.y);
                                a.z = fma_bf16x(xv, half_of(w2, g), a.z);
                                a.w = fma_bf16x(xv, half_of(w3, g), a.w);
                            }
                        }
                    }
                    *reinterpret_cast<float4 *>(zs + 4 * gq) = a;
                }
            }
            __syncwarp();
            if (w >= 1 && lane == 0) mbar_arrive(&bars.empty[(w - 1) % S]);  // chunk w - 1 is done here
        }
    }
    __syncthreads();
    if (*abort_flag) return;
    // selection: one thread per token over its n candidates (pairs 4 q0 ..)
    for (int j = tid; j < BT; j += NT) {
        const long t = t0 + j;
        if (t >= p.T) break;
        const int q0 = qbase[j];
        if (qbase[j + 1] == q0) continue;  // on the full path
        const int n = p.cnt[t];
        const float *z = zs + 4 * q0;
        const uint8_t *ids = pexp + 4 * q0;
        uint64_t taken = 0;
        float ev[16];
        float zmax = 0.0f;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) ev[jj] = 0.0f;
#pragma unroll
        for (int jj = 0; jj < kMaxTopK; ++jj) {
            if (jj < p.k) {
                float bv = -FLT_MAX;
                int bi = -1;
                for (int i = 0; i < n; ++i) {
                    const float zi = p.bias != nullptr ? z[i] + p.bias[ids[i]] : z[i];
                    if (!((taken >> i) & 1ull) && (bi < 0 || zi > bv)) {
                        bv = zi;
                        bi = i;
                    }
                }
                taken |= 1ull << bi;
                if (jj == 0) zmax = bv;
                ev[jj] = expf(bv - zmax);
                p.idx[t * p.k + jj] = ids[bi];
            }
        }
        const float den = butterfly_den(ev);
#pragma unroll
        for (int jj = 0; jj < kMaxTopK; ++jj)
            if (jj < p.k) p.gate[t * p.k + jj] = ev[jj] / den;
    }
}

// ------------------------------------------------------------ full path
// One block per listed token: thread e sums expert e's exact logit over the
// token's row (staged in shared memory); warp 0 then takes k rounds of a
// shuffle arg-max (ties to the lower expert) and the softmax of the k logits.
__global__ void __launch_bounds__(kFullThreads) route_full_kernel(const FastParams p)
{
    extern __shared__ __align__(16) uint8_t fx_raw[];
    uint16_t *xrow = reinterpret_cast<uint16_t *>(fx_raw);  // [d]
    __shared__ float lg[256];
    pdl_wait();
    pdl_trigger();
    const unsigned n = *p.novf;
    const int lane = threadIdx.x & 31;
    for (unsigned i = blockIdx.x; i < n; i += gridDim.x) {
        const long t = p.ovf[i];
        __syncthreads();  // the previous token's logits and row are no longer read
        for (int c8 = threadIdx.x * 8; c8 < p.d; c8 += kFullThreads * 8)
            *reinterpret_cast<uint4 *>(xrow + c8) = *reinterpret_cast<const uint4 *>(p.x + t * p.d + c8);
        __syncthreads();
        const int e = threadIdx.x;
        if (e < p.E) {
            const uint16_t *w = p.wr + static_cast<long>(e) * p.d;
            float a = 0.0f;
            for (int c8 = 0; c8 < p.d; c8 += 8)
                a = fma8(*reinterpret_cast<const uint4 *>(xrow + c8), *reinterpret_cast<const uint4 *>(w + c8), a);
            if (p.bias != nullptr) a = a + p.bias[e];
            lg[e] = a;
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            float v[8];
            uint32_t avail = 0;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int ee = lane + 32 * r;
                v[r] = ee < p.E ? lg[ee] : 0.0f;
                if (ee < p.E) avail |= 1u << r;
            }
            int sel_e = 0;
            float sel_v = 0.0f;
            for (int jj = 0; jj < p.k; ++jj) {
                float bv = -FLT_MAX;
                int be = INT_MAX;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int ee = lane + 32 * r;
                    if (((avail >> r) & 1u) && (be == INT_MAX || v[r] > bv)) {
                        bv = v[r];
                        be = ee;
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
                if (lane == jj) {
                    sel_e = be;
                    sel_v = bv;
                }
            }
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
}

// ------------------------------------------------------------ host side
size_t align_scratch(size_t v) { return (v + 255) / 256 * 256; }

struct ScratchLayout {
    size_t cand, cnt, ovf, novf, wn2, total;
};

ScratchLayout scratch_layout(long T, int E)
{
    ScratchLayout L{};
    size_t o = 0;
    L.cand = o;
    o = align_scratch(o + static_cast<size_t>(T) * kMaxCand);
    L.cnt = o;
    o = align_scratch(o + static_cast<size_t>(T));
    L.ovf = o;
    o = align_scratch(o + static_cast<size_t>(T) * 4);
    L.novf = o;
    o = align_scratch(o + 4);
    L.wn2 = o;
    o = align_scratch(o + static_cast<size_t>(E) * 4);
    L.total = o;
    return L;
}

constexpr size_t cand_smem_bytes()
{
    return 1024 + kCandStages * (kCandATile + kCandBTile) + sizeof(CandSmem);
}

size_t exact_smem_bytes(int S, int BT, int E)
{
    return 1024 + static_cast<size_t>(S) * (BT + E) * 128 + exact_tail_bytes(BT);
}

struct ExactPlan {
    int bt, stages;
};

ExactPlan exact_plan(long T, int E, int sms)
{
    ExactPlan pl{};
    long bt = (T + sms - 1) / sms;
    if (bt > kExactMaxBT) bt = kExactMaxBT;
    if (bt < 1) bt = 1;
    pl.bt = static_cast<int>(bt);
    pl.stages = exact_smem_bytes(4, pl.bt, E) <= kSmemLimit   ? 4
                : exact_smem_bytes(3, pl.bt, E) <= kSmemLimit ? 3
                                                              : 0;
    return pl;
}

bool make_map(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_outer, bool swizzle)
{
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kCandK), box_outer};
    const cuuint32_t estr[2] = {1, 1};
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// gamma_n(u) = n u / (1 - n u), rounded up to float
float gamma_of(double n, double u)
{
    const double g = n * u / (1.0 - n * u);
    return std::nextafter(static_cast<float>(g), INFINITY);
}

}  // namespace

size_t route_fast_scratch_bytes(long T, int E) { return scratch_layout(T, E).total; }

bool route_fast_supported(long T, int d, int E, int k)
{
    return T >= 1 && d >= 8 && d % 8 == 0 && d < (1 << 20) && k >= 1 && k <= kMaxTopK && E >= k &&
           E <= 256 && static_cast<size_t>(d) * 2 + 2048 <= kSmemLimit;
}

cudaError_t launch_route_fast(const RouteArgs &a, unsigned *status, void *scratch, size_t scratch_bytes,
                              cudaStream_t s)
{
    if (!route_fast_supported(a.T, a.d, a.E, a.k)) return cudaErrorNotSupported;
    const ScratchLayout L = scratch_layout(a.T, a.E);
    if (scratch == nullptr || status == nullptr || scratch_bytes < L.total ||
        (reinterpret_cast<uintptr_t>(scratch) & 255u))
        return cudaErrorInvalidValue;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorUnknown;
    const ExactPlan pl = exact_plan(a.T, a.E, sms);
    if (pl.stages == 0) return cudaErrorNotSupported;

    uint8_t *sc = static_cast<uint8_t *>(scratch);
    FastParams p{};
    p.x = a.x;
    p.wr = a.wr;
    p.bias = a.bias;
    p.idx = a.topk_idx;
    p.gate = a.topk_gate;
    p.status = status;
    p.cand = sc + L.cand;
    p.cnt = sc + L.cnt;
    p.ovf = reinterpret_cast<int32_t *>(sc + L.ovf);
    p.novf = reinterpret_cast<unsigned *>(sc + L.novf);
    p.wn2 = reinterpret_cast<float *>(sc + L.wn2);
    p.T = a.T;
    p.d = a.d;
    p.E = a.E;
    p.k = a.k;
    p.npad = (a.E + 15) / 16 * 16;
    p.bt = pl.bt;
    p.gamma = std::nextafter(gamma_of(a.d, std::ldexp(1.0, -24)) + gamma_of(a.d, std::ldexp(1.0, -21)),
                             static_cast<float>(INFINITY));
    p.abs_eps = static_cast<float>(std::ldexp(static_cast<double>(a.d), -120));

    // swizzled tiles for the candidate kernel's MMAs, plain rows for the exact kernel
    CUtensorMap tm_x, tm_w, tm_xr, tm_wr;
    if (!make_map(&tm_x, a.x, a.d, a.T, kCandM, true) || !make_map(&tm_w, a.wr, a.d, a.E, p.npad, true) ||
        !make_map(&tm_xr, a.x, a.d, a.T, pl.bt, false) || !make_map(&tm_wr, a.wr, a.d, a.E, a.E, false))
        return cudaErrorInvalidValue;

    struct CandTag {};
    struct Exact3Tag {};
    struct Exact4Tag {};
    struct FullTag {};
    cudaError_t e = once_per_device<CandTag>([](int) {
        return cudaFuncSetAttribute(route_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(cand_smem_bytes()));
    });
    if (e != cudaSuccess) return e;
    if (pl.stages == 4)
        e = once_per_device<Exact4Tag>([](int) {
            return cudaFuncSetAttribute(route_exact_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmemLimit));
        });
    else
        e = once_per_device<Exact3Tag>([](int) {
            return cudaFuncSetAttribute(route_exact_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmemLimit));
        });
    if (e != cudaSuccess) return e;
    e = once_per_device<FullTag>([](int) {
        return cudaFuncSetAttribute(route_full_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmemLimit - 2048));
    });
    if (e != cudaSuccess) return e;

    e = launch_pdl(route_wnorm_kernel, dim3(a.E), dim3(128), 0, s, p);
    if (e != cudaSuccess) return e;
    e = launch_pdl(route_cand_kernel, dim3((a.T + kCandM - 1) / kCandM), dim3(kCandThreads), cand_smem_bytes(),
                   s, tm_x, tm_w, p);
    if (e != cudaSuccess) return e;
    const dim3 eg((a.T + pl.bt - 1) / pl.bt);
    const size_t esm = exact_smem_bytes(pl.stages, pl.bt, a.E);
    e = pl.stages == 4 ? launch_pdl(route_exact_kernel<4>, eg, dim3(kExactThreads), esm, s, tm_xr, tm_wr, p)
                       : launch_pdl(route_exact_kernel<3>, eg, dim3(kExactThreads), esm, s, tm_xr, tm_wr, p);
    if (e != cudaSuccess) return e;
    const int fg = a.T < sms ? a.T : sms;
    return launch_pdl(route_full_kernel, dim3(fg), dim3(kFullThreads), static_cast<size_t>(a.d) * 2, s, p);
}

}  // namespace moe
