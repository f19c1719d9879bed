// grouped_gemm.cu -- the expert computation of one MoE layer as ONE persistent
// grouped GEMM over all experts (Xian et al., "X-Stage ...", section 2.2:
// Linear-1 -> SwiGLU -> Linear-2 per expert; Cui et al., "Fine-grained
// Computation-Communication Overlap ...", section 3.3.1: one rank-wide
// persistent kernel over a unified tile worklist with per-tile ready flags).
//
// Tiles. Rows of x_perm are expert-contiguous. A "scheduler row" is one band
// of 128 (single CTA) or 256 (CTA pair) token rows of one expert; the
// scheduler rows of all experts are concatenated in expert order (row p ->
// expert e(p), first row O_e), or, in the mixed order, the rows of experts
// that have a single row are spread evenly among the others' (see the
// prologue).
//   Linear-1 tile (p, n): h[rows, n*128 : n*128+128] =
//       bf16(silu(x W1[e]^T) * (x W3[e]^T)); the MMA is 128 x 256 x 16 with the
//       W1 tile stacked on the W3 tile, so one accumulator holds gate | up.
//   Linear-2 tile (p, n): y[rows, n*N2 : n*N2+N2] = bf16(h W2[e]^T).
// A Linear-2 tile of row p reads h rows that all Linear-1 tiles of row p write;
// each finished Linear-1 tile increments l1_done[p] (release) and the TMA
// producer of a Linear-2 tile waits (acquire, bounded) until it reaches P1.
// Each finished Linear-2 tile publishes its ready flag (= the call's epoch).
//
// h ring (optional, Xian et al., Algorithm 1's "destination ring slot"): h
// holds Q scheduler rows instead of all of them; row p lives in slot p mod Q.
// A Linear-1 tile of row p >= Q first waits (acquire, bounded) until every
// Linear-2 tile of row p - Q has finished (l2_done[p - Q] = CTAs per tile *
// P2), so the slot's previous rows have been read. With Q >= D + 2 * group
// every such Linear-2 tile comes earlier in the tile order than the waiting
// tile (see TileSource), so these waits cannot deadlock either.
//
// Fused combine (FC; Cui et al., section 3.3: a consumer polls the producer's
// per-tile signals and sends each finished block to its owner): two more warps
// per CTA consume scheduler rows as their Linear-2 tiles finish (the per-row
// Linear-2 counter reaches CTAs per tile * P2). A token is combined by the
// unit that holds its last row (in scheduler-row order) once its other rows'
// rows are finished too, and written to its owner segment; the epilogue warps
// join after their last tile. The consumers wait only on Linear-2 tiles, which
// never wait on them, and the fp32 sum runs in j order exactly as the combine
// kernel's, so the output bits are the same.
//
// Order (Xian et al., Algorithm 1): one cursor pair k1, k2 walks the Linear-1
// and Linear-2 tile streams; the Linear-2 tile at k2 goes out once its row
// trails the Linear-1 cursor's row by at least D, else the next Linear-1 tile.
// That gives ONE global tile sequence; the instances (CTAs or CTA pairs) take
// its tiles in order from a global ticket counter, so every tile is started
// by a CTA that is running, every dependency wait is on a tile with a smaller
// ticket, and the waits cannot deadlock whether or not the whole grid is
// resident (see TileSource). The expert-wave order (all Linear-1 tiles of a
// wave of experts, then its Linear-2 tiles) is kept as the comparison
// schedule. Both orders give bit-identical outputs.
//
// CTA roles (192 threads, 256 with the fused combine): warp 0 = TMA producer,
// warp 1 = tensor-memory allocator + single-thread MMA issuer, warps 2..5 =
// epilogue (warp w reads tensor-memory lanes 32*(w%4)...+31), warps 6..7 =
// combine consumers. Tensor memory holds two 128 x 256 fp32 accumulators (512
// columns).
//
// CTA pairs (CG = 2, the default): the two CTAs of a cluster compute 256-row
// tiles with tcgen05.mma.cta_group::2. Each CTA loads its own 128 rows of A and
// half of B (Linear-1: W1 in the first CTA, W3 in the second; Linear-2: half of
// the W2 rows), so a pipeline stage is 32 KiB and six stages fit, synchronised
// two at a time (kSync). The first CTA
// issues every MMA and multicasts each completion to both CTAs; both CTAs'
// TMA loads complete on the first CTA's stage barrier; both CTAs' epilogues
// release an accumulator by arriving on the first CTA's barrier. CG = 1 keeps
// one CTA per tile (4 stages of 48 KiB) for comparison.
//
// Tokens on the N side (TN, CTA pairs only). Above, tokens are the MMA's M
// rows, so every expert's last scheduler row is padded to 256 rows. With TN the
// operands swap: A (M, split between the pair) holds weight rows and B (N)
// holds the scheduler row's tokens, and the MMA width N is the expert's
// remaining tokens rounded up to 16, so an expert wastes at most 15 token
// columns. Linear-1: each CTA's A tile is 64 W1 rows over the same 64 W3
// rows (64 features; the pair covers 128 h columns), so tensor-memory lanes
// 0-63 hold gate and 64-127 up: the epilogue warps reading lanes q*32.. and
// (q+2)*32.. swap half of their 32-token slab through shared memory, the gate
// warp then finishing tokens 0-15 and the up warp tokens 16-31. Linear-2: each
// CTA's A tile is 128 W2 rows (256 y columns a pair). B of a tile of N tokens
// is split as the MMA wants it: the first CTA supplies tokens [0, N/2), the
// second [N/2, N). Each epilogue warp turns its (row, token) block around in
// its own shared-memory slab, so that lanes store tokens' contiguous outputs.
#include <climits>

#include "kernels.cuh"
#include "sm100.cuh"

namespace moe {
namespace {

constexpr int kBlockM = 128;  // rows per CTA
constexpr int kBlockK = 64;   // 64 bf16 = 128 B = one swizzle atom row
constexpr int kL1N = 128;     // h columns per Linear-1 tile (MMA N = 2 * 128)
constexpr int kATileBytes = kBlockM * kBlockK * 2;  // 16 KiB
constexpr int kMaxStages = 6;
// Stages per full/empty barrier: the producer arms and fills two stages at a
// time, and the MMA thread waits once and commits once per 8 MMAs instead of
// 4. The thread's loop of wait, MMAs and commit costs about as much as a
// full-width k-block of tensor work, so halving its waits and commits per MMA
// gave 3-5% less GEMM time on every workload (three stages a barrier left too
// little of the ring loading ahead and lost 7-12%).
constexpr int kSync = 2;
constexpr int kDefaultGroupRows = 32;  // raster group, in 128-row M-tiles
constexpr int kSmallExpertGroupRows = 16;  // ... when experts average under 4 scheduler rows
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr int kThreads = 192;
constexpr int kConsumerThreads = 64;  // two consumer warps with the fused combine
constexpr int kEpiThreads = 128;
constexpr int kTraceWords = 16;  // per-CTA counters when tracing is on
// per-tile timeline record (clock64 of the CTA's SM):
// 0 kind | row << 2 | n << 34, 1 producer start (after its dependency wait),
// 2 producer dependency-wait cycles, 3 MMA start (accumulator free), 4 MMA last
// issue, 5 MMA stage-wait cycles, 6 epilogue start (accumulator ready),
// 7 epilogue stores done
constexpr int kTileTraceWords = 8;
constexpr int kMaxMixedRows = 1024;  // scheduler rows the mixed order can hold
constexpr int kTileQueue = 8;        // tile descriptors in flight per CTA
constexpr bool kMixedByDefault = true;

template <int CG, bool TN = false>
struct Cfg {
    static constexpr int kStages = CG == 2 ? 6 : 4;
    static constexpr int kSlots = kStages / kSync;  // barrier pairs (two stages each)
    static constexpr int kBTileBytes = (256 / CG) * kBlockK * 2;  // this CTA's share of B
    // token rows of one scheduler row: the MMA's M rows with tokens on the M
    // side; up to 256 tokens (the widest MMA N) with tokens on the N side
    static constexpr int kTileRows = TN ? 256 : kBlockM * CG;
};

struct GemmParams {
    const int32_t *offsets;
    uint16_t *h;
    uint16_t *y;
    unsigned *l1_done;
    unsigned *l2_done;  // per scheduler row: finished Linear-2 tiles (h ring only)
    unsigned *ticket;   // next tile of the global order (zero at launch)
    unsigned *l2_flags;
    unsigned *status;
    int E, d, F, R;
    int P1, P2, N2;
    int kb1, kb2;
    int schedule, lead, group, cg;
    int ring;  // h ring slots in scheduler rows; 0 = h holds every row
    int mixed; // mixed row order: 0 off, 1 when single-row experts are >= 1/4 of the rows, 2 asked for
    int rows;  // token rows of one scheduler row
    int fc;    // fused combine: count finished Linear-2 tiles per row for the consumers
    const float *gate;
    const int32_t *row_of_slot;
    const int32_t *slot_of_row;
    int T, k, rows_per_seg;
    uint16_t *seg[kMaxSegments];
    int unmet_dependency;  // > 0 only in the failure-detection test: a wait nothing satisfies
    unsigned long long wait_ns;  // limit of every bounded wait
    unsigned epoch;
    unsigned long long *trace;
    unsigned long long *tile_trace;  // optional per-tile timeline: [CTA][cap][kTileTraceWords]
    int tile_trace_cap;
};

struct SmemCtl {
    uint64_t full[kMaxStages];   // barrier pair's stages loaded (used in the pair's first CTA)
    uint64_t empty[kMaxStages];  // barrier pair's stages consumed by the MMAs
    uint64_t tfull[2];           // accumulator ready for the epilogue
    uint64_t tempty[2];          // accumulator drained (every epilogue thread of the pair)
    uint64_t estore[2];          // this CTA's epilogue stores issued (publisher)
    uint64_t drain;              // every MMA this CTA issued has completed (teardown)
    uint64_t tq_full[kTileQueue];   // descriptor written (in each CTA of the pair)
    uint64_t tq_empty[kTileQueue];  // descriptor read by every reading role (in the CTA that publishes)
    uint64_t sched_go;              // pair scheduler: this CTA's producer took a descriptor
    int4 tq[kTileQueue];            // tile descriptors (pack_tile)
    uint32_t tmem_base;
    uint32_t p_uses;                 // barrier-pair loads this CTA's producer issued (teardown)
    uint32_t p_bytes[kMaxStages];    // this CTA's bytes in the latest load of each barrier pair
    int abort;
    int epi_fail;  // TN epilogue: a warp gave up (the warp pairs meet at barriers)
    int cunit;     // fused combine: next consumer unit of this CTA
    int nwaves;
    int offs[kMaxExperts + 1];       // expert row offsets (copy of expert_offsets)
    int row_start[kMaxExperts + 1];  // first scheduler row of each expert
    int wave_row[kMaxExperts + 1];   // wave w spans scheduler rows [wave_row[w], wave_row[w+1])
    int wave_tile[kMaxExperts + 1];  // first global tile index of wave w
    int mixed;                       // scheduler rows in the mixed order (mrow) instead of expert order
    int mrow[kMaxMixedRows];         // scheduler row -> expert | band << 9 (when the rows fit)
    int seg[kMaxMixedRows + 1];      // first ticket of each row block's segment (interleaved order)
};

// epilogue buffer per epilogue warp: tokens on the M side use 32 rows x 64
// bf16 (4 KiB); tokens on the N side two 2 KiB mailboxes and a 1 KiB slab
constexpr int kEpiStageBytes = 5 * 1024;
constexpr size_t kCtlBytes = (sizeof(SmemCtl) + 127) / 128 * 128;
template <int CG, bool TN>
constexpr size_t smem_bytes()
{
    return 1024 /*alignment slack*/ + size_t(Cfg<CG, TN>::kStages) * (kATileBytes + Cfg<CG, TN>::kBTileBytes) +
           kCtlBytes + 4 * kEpiStageBytes;
}

static_assert(smem_bytes<2, true>() <= 232448 && smem_bytes<1, false>() <= 232448,
              "shared memory of the grouped GEMM exceeds 227 KiB");

struct Tile {
    int kind;  // 0 = Linear-1, 1 = Linear-2, -1 = no more tiles
    int row;   // scheduler row
    int n;     // N-tile
    int e;     // expert owning the row
    int b0;    // the row's first token row (in x_perm / y_perm)
};

// Position k of a tile stream (Pn N-tiles per scheduler row) -> (row, n). Tiles
// of one expert occupy positions [row_start[e]*Pn, row_start[e+1]*Pn); inside
// the expert they run over groups of GM consecutive rows, N-tile-major within a
// group, so a weight tile is reused by the group's M-tiles back to back. Every
// tile of row p sits below position (p + GM) * Pn and at or above position
// (p - GM + 1) * Pn. In the mixed order the groups run over the global row
// sequence instead.
__device__ __forceinline__ int expert_of_row(const SmemCtl &c, int E, int row)
{
    if (c.row_start[E] <= kMaxMixedRows) return c.mrow[row] & 0x1FF;  // the table holds every row
    // the largest e with row_start[e] <= row (row < row_start[E]): experts
    // without rows share their row_start with the next expert
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (c.row_start[mid] <= row) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// first row and size of the raster group holding scheduler row m
__device__ __forceinline__ void group_of_row(const SmemCtl &c, int E, int GM, int m, int &g0, int &gs)
{
    if (c.mixed) {
        g0 = m - m % GM;
        gs = min(GM, c.row_start[E] - g0);
        return;
    }
    const int e = expert_of_row(c, E, m);
    const int r0 = c.row_start[e];
    g0 = m - (m - r0) % GM;
    gs = min(GM, c.row_start[e + 1] - g0);
}

__device__ Tile stream_tile(const SmemCtl &c, int E, int k, int Pn, int GM, int kind, int rows)
{
    Tile t;
    t.kind = kind;
    int g0, gs;
    group_of_row(c, E, GM, k / Pn, g0, gs);  // positions of a group: [g0 * Pn, (g0 + gs) * Pn)
    const int i = k - g0 * Pn;
    t.n = i / gs;
    t.row = g0 + i % gs;
    if (c.mixed || c.row_start[E] <= kMaxMixedRows) {
        const int packed = c.mrow[t.row];
        t.e = packed & 0x1FF;
        t.b0 = c.offs[t.e] + (packed >> 9) * rows;
    } else {
        t.e = expert_of_row(c, E, t.row);
        t.b0 = c.offs[t.e] + (t.row - c.row_start[t.e]) * rows;
    }
    return t;
}

// The tile order (Xian et al., Algorithm 1, taken as ONE sequence for the
// whole grid). Instances claim tickets 0, 1, 2, ... from a global counter, so
// every tile is started by a running CTA and in ticket order. Interleaved
// schedule: the Linear-1 and Linear-2 streams merged with lead D, i.e. the
// sequence one instance walking both streams with step 1 would emit. With
// m(k2) the largest row among Linear-2 positions <= k2 (the stream is in
// order, so a tile never passes an earlier one), the Linear-2 tile at k2 goes
// right before the Linear-1 tiles of row block K = min(m(k2) + D, P), or after
// all of them when K = P. The sequence is thus, for b = 0 .. P: the Linear-2
// tiles with K = b, then the P1 Linear-1 tiles of block b. Segment b starts at
// ticket S(b) = b * P1 + C(b - D - 1), C(m) = number of Linear-2 positions
// with m(k2) <= m (a closed form per raster group), so a ticket is decoded by
// a binary search over b.
//   Dependencies: a Linear-2 tile of row r waits for the Linear-1 tiles of
// row r, all in blocks < r + GM <= r + D <= K when D >= GM; a Linear-1 tile
// of row p in an h ring of Q rows waits for the Linear-2 tiles of row p - Q,
// whose K <= p - Q + GM - 1 + D <= p - GM + 1 (the first block holding
// tiles of row p) when Q >= D + 2 GM. So every wait is on a smaller ticket,
// claimed earlier by a CTA that is running, and the waits cannot deadlock
// however many CTAs are resident.
// Expert-wave schedule: ticket = position in the wave sequence (each wave:
// its Linear-1 tiles, then its Linear-2 tiles).
struct TileSource {
    int P, P1, P2, D, GM, mode, rows, tot1, tot2, E;

    __device__ TileSource(const SmemCtl &c, const GemmParams &p)
    {
        P = c.row_start[p.E];
        P1 = p.P1;
        P2 = p.P2;
        D = p.lead;
        GM = p.group;
        mode = p.schedule;
        rows = p.rows;
        tot1 = P * P1;
        tot2 = P * P2;
        E = p.E;
    }

    // C(m): Linear-2 positions whose largest row so far is <= m. Inside a
    // raster group (g0, gs) the first pass (n = 0) walks its rows one by
    // one, every later pass already holds the group's last row.
    __device__ int l2_count(const SmemCtl &c, int m) const
    {
        if (m < 0) return 0;
        if (m >= P - 1) return tot2;
        int g0, gs;
        group_of_row(c, E, GM, m, g0, gs);
        return m < g0 + gs - 1 ? g0 * P2 + (m - g0 + 1) : (g0 + gs) * P2;
    }

    __device__ Tile decode(const SmemCtl &c, unsigned q) const
    {
        Tile t;
        if (mode != 0) {
            if (q >= static_cast<unsigned>(c.wave_tile[c.nwaves])) {
                t.kind = -1;
                return t;
            }
            const int gi = static_cast<int>(q);
            int lo = 0, hi = c.nwaves - 1;  // the wave holding gi
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (c.wave_tile[mid] <= gi) lo = mid;
                else hi = mid - 1;
            }
            const int j = gi - c.wave_tile[lo];
            const int r0 = c.wave_row[lo];
            const int nr = c.wave_row[lo + 1] - r0;
            if (j < nr * P1) return stream_tile(c, E, r0 * P1 + j, P1, GM, 0, rows);
            return stream_tile(c, E, r0 * P2 + (j - nr * P1), P2, GM, 1, rows);
        }
        if (q >= static_cast<unsigned>(tot1 + tot2)) {
            t.kind = -1;
            return t;
        }
        const int qi = static_cast<int>(q);
        // the segment holding ticket q: the largest b in [0, P] with S(b) <= q
        int lo = 0, hi = P;
        if (P <= kMaxMixedRows) {
            while (lo < hi) {  // over the table the prologue built
                const int mid = (lo + hi + 1) >> 1;
                if (c.seg[mid] <= qi) lo = mid;
                else hi = mid - 1;
            }
        } else {
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (mid * P1 + l2_count(c, mid - D - 1) <= qi) lo = mid;
                else hi = mid - 1;
            }
        }
        const int b = lo;
        const int c0 = l2_count(c, b - D - 1);
        const int n2 = (b < P ? l2_count(c, b - D) : tot2) - c0;  // Linear-2 tiles of the segment
        const int off = qi - (b * P1 + c0);
        if (off < n2) return stream_tile(c, E, c0 + off, P2, GM, 1, rows);
        return stream_tile(c, E, b * P1 + (off - n2), P1, GM, 0, rows);
    }
};

// Tile descriptors pass from the producer that claims them to the CTA's other
// roles (and the peer CTA) through a small shared-memory queue.
__device__ __forceinline__ int4 pack_tile(const Tile &t)
{
    return make_int4(t.kind < 0 ? -1 : (t.kind | (t.n << 1)), t.row, t.e, t.b0);
}

__device__ __forceinline__ Tile unpack_tile(int4 v)
{
    Tile t;
    t.kind = v.x < 0 ? -1 : (v.x & 1);
    t.n = v.x < 0 ? 0 : (v.x >> 1);
    t.row = v.y;
    t.e = v.z;
    t.b0 = v.w;
    return t;
}

__device__ __forceinline__ bool wait_rows_ready(const unsigned *ctr, unsigned target,
                                                volatile int *cta_abort, unsigned *status,
                                                unsigned detail, unsigned long long limit_ns,
                                                unsigned where = kWhereProducerDep)
{
    if (ld_acquire_u32(ctr) >= target) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(128);
        if (ld_acquire_u32(ctr) >= target) return true;
        if ((it & 15u) == 0u) {
            if (*cta_abort) return false;
            if (ld_volatile_u32(status) != 0u) {
                *cta_abort = 1;
                return false;
            }
            if (globaltimer_ns() - t0 > limit_ns) {
                report_failure(status, kStatusTimeout, where, detail);
                *cta_abort = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ float silu_mul(float g, float u)
{
    return g * __fdividef(1.0f, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ float silu_mul(uint32_t g_bits, uint32_t u_bits)
{
    return silu_mul(__uint_as_float(g_bits), __uint_as_float(u_bits));
}

// MMA width (TN) of a scheduler row whose expert has `remaining` tokens from
// the row's first token on: the row's tokens rounded up to a multiple of 16
__device__ __forceinline__ int tile_tokens(int remaining, int rows)
{
    return (min(remaining, rows) + 15) & ~15;
}

// last index i in [0, n) with v[i] <= x (v non-decreasing, v[0] <= x)
__device__ __forceinline__ int last_le(const int *v, int n, int x)
{
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (v[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Fused combine, run by one warp: take this CTA's units from a shared counter
// (unit U = 32 rows of scheduler row U / units-per-row; CTA g owns U = g,
// g + gridDim.x, ... in increasing U, so every scheduler row's rows are spread
// over many CTAs), wait until the unit's row has all its Linear-2 tiles
// finished, and combine every token whose last row lies in the unit. False
// when a wait gave up.
template <int CG, bool TN>
__device__ bool combine_consumer(SmemCtl &c, const GemmParams &p, int lane, volatile int *abort_flag)
{
    constexpr int kTileRows = Cfg<CG, TN>::kTileRows;
    constexpr int kUnits = kTileRows / 32;
    const int E = p.E;
    const int P = c.row_start[E];
    const int total = P * kUnits;
    const int mine = total > static_cast<int>(blockIdx.x)
                         ? (total - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                               static_cast<int>(gridDim.x)
                         : 0;
    const unsigned target = static_cast<unsigned>(CG * p.P2);
    const int nvec = p.d / 8;
    for (;;) {
        int u = 0;
        if (lane == 0) u = atomicAdd(&c.cunit, 1);
        u = __shfl_sync(0xffffffffu, u, 0);
        if (u >= mine) return true;
        const int U = static_cast<int>(blockIdx.x) + u * static_cast<int>(gridDim.x);
        const int b = U / kUnits;
        const int e = last_le(c.row_start, E, b);
        const int band0 = c.offs[e] + (b - c.row_start[e]) * kTileRows;
        const int r0 = band0 + (U % kUnits) * 32;
        const int r1 = min(c.offs[e + 1], band0 + kTileRows);
        if (r0 >= r1) continue;
        bool ok = true;
        if (lane == 0)
            ok = wait_rows_ready(&p.l2_done[b], target, abort_flag, p.status,
                                 0x20000000u | static_cast<unsigned>(b), p.wait_ns, kWhereCombine);
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return false;
        __syncwarp();
        // lane i looks at row r0 + i: its token, the token's rows and their
        // scheduler rows; the token belongs here if b is the last of them
        const int r = r0 + lane;
        int t = 0, rows[kMaxTopK], rb[kMaxTopK];
        bool own = false;
        if (r < r1) {
            t = __ldg(p.slot_of_row + r) / p.k;
            int bmax = -1;
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                rows[j] = j < p.k ? __ldg(p.row_of_slot + static_cast<long>(t) * p.k + j) : -1;
                rb[j] = -1;
                if (rows[j] >= 0) {  // a slot without a row (bad expert id) adds no term
                    const int ej = last_le(c.offs, E, rows[j]);
                    rb[j] = c.row_start[ej] + (rows[j] - c.offs[ej]) / kTileRows;
                    bmax = max(bmax, rb[j]);
                }
            }
            own = bmax == b;
        }
        unsigned todo = __ballot_sync(0xffffffffu, own);
        while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const int tt = __shfl_sync(0xffffffffu, t, src);
            // the token's other rows must be finished as well
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                const int bj = __shfl_sync(0xffffffffu, rb[j], src);
                if (bj >= 0 && bj != b) {
                    bool okj = true;
                    if (lane == 0)
                        okj = wait_rows_ready(&p.l2_done[bj], target, abort_flag, p.status,
                                              0x20000000u | static_cast<unsigned>(bj), p.wait_ns,
                                              kWhereCombine);
                    if (!__shfl_sync(0xffffffffu, okj ? 1 : 0, 0)) return false;
                }
            }
            __syncwarp();
            const uint4 *src_rows[kMaxTopK];
            float g[kMaxTopK];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                const int rj = __shfl_sync(0xffffffffu, rows[j], src);
                src_rows[j] = rj >= 0 ? reinterpret_cast<const uint4 *>(p.y + static_cast<long>(rj) * p.d)
                                      : nullptr;
                g[j] = j < p.k ? __ldg(p.gate + static_cast<long>(tt) * p.k + j) : 0.0f;
            }
            uint4 *dst = reinterpret_cast<uint4 *>(p.seg[tt / p.rows_per_seg] +
                                                   static_cast<long>(tt % p.rows_per_seg) * p.d);
            for (int v = lane; v < nvec; v += 32) {
                uint4 val[kMaxTopK];
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j)
                    if (src_rows[j] != nullptr) val[j] = src_rows[j][v];
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j) {
                    if (src_rows[j] != nullptr) {
                        const uint32_t w[4] = {val[j].x, val[j].y, val[j].z, val[j].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            acc[2 * h] = fmaf(g[j], __uint_as_float(w[h] << 16), acc[2 * h]);
                            acc[2 * h + 1] = fmaf(g[j], __uint_as_float(w[h] & 0xFFFF0000u), acc[2 * h + 1]);
                        }
                    }
                }
                dst[v] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                    pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
            }
        }
    }
}

// Publish the tile of a claimed ticket as descriptor number tl: single CTA:
// by its producer; pair: by the second CTA's scheduler thread, into both CTAs'
// queues (`other` = the other CTA's rank). False when the wait for a free
// queue slot gave up.
template <int CG>
__device__ bool publish_tile(SmemCtl &c, const GemmParams &p, const TileSource &src, int tl, unsigned ticket,
                             Tile &out, volatile int *abort_flag, uint32_t other)
{
    const int q = tl % kTileQueue;
    const uint32_t ph = static_cast<uint32_t>(tl / kTileQueue) & 1u;
    out = src.decode(c, ticket);
    if (!mbar_wait_cluster(&c.tq_empty[q], ph ^ 1u, abort_flag, p.status, kWhereTileQueue,
                           static_cast<unsigned>(tl), p.wait_ns))
        return false;
    const int4 v = pack_tile(out);
    c.tq[q] = v;
    if constexpr (CG == 2) {
        st_shared_cluster_v4(map_to_cta(smem_u32(&c.tq[q]), other), v);
        mbar_arrive_cluster(map_to_cta(smem_u32(&c.tq_full[q]), other));
    }
    mbar_arrive(&c.tq_full[q]);
    return true;
}

// Every other role: wait for descriptor number tl and read it. False when
// the wait gave up.
__device__ __forceinline__ bool take_tile(SmemCtl &c, const GemmParams &p, int tl, Tile &out,
                                          volatile int *abort_flag)
{
    const int q = tl % kTileQueue;
    const uint32_t ph = static_cast<uint32_t>(tl / kTileQueue) & 1u;
    if (!mbar_wait_cluster(&c.tq_full[q], ph, abort_flag, p.status, kWhereTileQueue,
                           0x10000000u | static_cast<unsigned>(tl), p.wait_ns))
        return false;
    out = unpack_tile(c.tq[q]);
    return true;
}

// Give descriptor tl's queue slot back (once per reading role, after every
// thread of the role has read it). The slots are counted where the publisher
// runs: the single CTA, or the second CTA of a pair.
template <int CG>
__device__ __forceinline__ void release_tile(SmemCtl &c, int tl, uint32_t rank)
{
    const int q = tl % kTileQueue;
    if (CG == 1 || rank == 1) mbar_arrive(&c.tq_empty[q]);
    else mbar_arrive_cluster(map_to_cta(smem_u32(&c.tq_empty[q]), 1));
}

// Teardown, run by the producer thread of the pair's first CTA (or of a single
// CTA) once both producers have stopped: wait until every load still in flight
// has landed. Loads go out a barrier pair (kSync stages) at a time: use i (of
// either CTA) used pair i mod S in phase (i / S) mod 2, S = the number of
// pairs, and a producer only issues use i after use i - S was consumed, so
// only the last S uses can be in flight. With a CTA pair, the two producers
// may have stopped at different uses (each gives up on its own): a use the
// first CTA armed for both halves but the peer never loaded gets the peer's
// bytes counted here, and a use only the peer loaded gets its arrival and byte
// count here, so every such phase completes once the issued copies land. A
// wait that runs out is recorded in the status word.
template <int CG, int kSlots>
__device__ void drain_loads(SmemCtl &c, const GemmParams &p)
{
    constexpr unsigned long long kDrainLimitNs = 50000000ull;
    const uint32_t own = c.p_uses;
    uint32_t peer = own;
    if constexpr (CG == 2) peer = ld_shared_cluster_u32(map_to_cta(smem_u32(&c.p_uses), 1));
    const uint32_t n = own > peer ? own : peer;
    const uint32_t lo = n > static_cast<uint32_t>(kSlots) ? n - kSlots : 0u;
    for (uint32_t i = lo; i < n; ++i) {
        const int s = static_cast<int>(i % kSlots);
        const uint32_t par = (i / kSlots) & 1u;
        if constexpr (CG == 2) {
            if (i < own && i >= peer)
                mbar_complete_tx(&c.full[s], c.p_bytes[s]);
            else if (i >= own && i < peer)
                mbar_arrive_expect_tx(&c.full[s], ld_shared_cluster_u32(map_to_cta(smem_u32(&c.p_bytes[s]), 1)));
        }
        if (!mbar_wait_drain(&c.full[s], par, kDrainLimitNs))
            report_failure(p.status, kStatusTimeout, kWhereLoadDrain, static_cast<unsigned>(s));
    }
}

template <int CG, bool TN, bool FC>
__global__ void __launch_bounds__(FC ? kThreads + kConsumerThreads : kThreads, 1)
grouped_swiglu_gemm_kernel(const __grid_constant__ CUtensorMap tm_x,
                           const __grid_constant__ CUtensorMap tm_h,
                           const __grid_constant__ CUtensorMap tm_w1,
                           const __grid_constant__ CUtensorMap tm_w3,
                           const __grid_constant__ CUtensorMap tm_w2, const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    uint8_t *sA = reinterpret_cast<uint8_t *>(base);
    constexpr int kStages = Cfg<CG, TN>::kStages;
    constexpr int kBTileBytes = Cfg<CG, TN>::kBTileBytes;
    constexpr int kTileRows = Cfg<CG, TN>::kTileRows;
    uint8_t *sB = sA + kStages * kATileBytes;
    SmemCtl &c = *reinterpret_cast<SmemCtl *>(sB + kStages * kBTileBytes);
    uint8_t *s_epi = sB + kStages * kBTileBytes + kCtlBytes;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = p.E;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;  // CTA within the pair
    const bool leader = rank == 0;
    // tokens on the N side: weight rows (features) a tile covers in this CTA:
    // Linear-1 64 (64 W1 over the same 64 W3 rows), Linear-2 128 W2 rows
    constexpr int kTnL1 = 64, kTnL2 = kBlockM;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg<CG, TN>::kSlots; ++s) {
            mbar_init(&c.full[s], 1);
            mbar_init(&c.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&c.tfull[b], 1);
            mbar_init(&c.tempty[b], kEpiThreads * CG);
            mbar_init(&c.estore[b], kEpiThreads);
        }
        mbar_init(&c.drain, 1);
        for (int q = 0; q < kTileQueue; ++q) {
            mbar_init(&c.tq_full[q], 1);
            // readers of a descriptor: single CTA: the MMA thread and the four
            // epilogue warps (the producer publishes); pair: both producers, the
            // MMA thread and both CTAs' epilogue warps (the peer's scheduler
            // thread publishes)
            mbar_init(&c.tq_empty[q], CG == 2 ? 11 : 5);
        }
        mbar_init(&c.sched_go, 1);
        c.p_uses = 0;
        c.abort = 0;
        c.epi_fail = 0;
        c.cunit = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_h);
        tma_prefetch_desc(&tm_w1);
        tma_prefetch_desc(&tm_w3);
        tma_prefetch_desc(&tm_w2);
    }
    if (warp == 1) {
        tmem_alloc<CG>(&c.tmem_base, kTmemCols);
        tmem_relinquish<CG>();
        tc_fence_before();
    }
    // everything above overlaps the previous kernel's tail; what follows reads
    // its outputs (expert offsets, x_perm, counters)
    pdl_wait();
    pdl_trigger();
    if (warp == 2) {
        // expert offsets -> scheduler-row prefix (warp-parallel exclusive scan).
        // Offsets that are not a non-decreasing sequence from 0 to R are
        // reported and leave the kernel with no tiles (nothing is written).
        const int per = (E + 31) / 32;
        int local = 0;
        bool bad = false;
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e < E) {
                const int o0 = p.offsets[e], o1 = p.offsets[e + 1];
                c.offs[e] = o0;
                if (e == E - 1) c.offs[E] = o1;
                bad |= o1 < o0 || (e == 0 && o0 != 0) || (e == E - 1 && o1 != p.R);
                local += (o1 - o0 + kTileRows - 1) / kTileRows;
            }
        }
        const bool any_bad = __any_sync(0xffffffffu, bad);
        if (any_bad) {
            local = 0;
            if (lane == 0 && blockIdx.x == 0)
                report_failure(p.status, kStatusBadOffsets, kWhereGemmOffsets, 0);
        }
        int incl = local;
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        __syncwarp();  // offs[] written by other lanes above
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e < E) {
                c.row_start[e] = run;
                if (!any_bad) run += (c.offs[e + 1] - c.offs[e] + kTileRows - 1) / kTileRows;
            }
        }
        if (lane == 31) c.row_start[E] = incl;
        __syncwarp();
        // Mixed row order: experts with a single scheduler row ("light": their
        // tiles mostly stream weights) are spread evenly among the rows of the
        // other experts ("heavy": their tiles are compute-bound), so that the
        // tiles in flight at any time mix both. Light row i goes to position
        // ceil((i+1)P/l) - 1, heavy row j to the (j+1)-th remaining position
        // (Bresenham over P = h + l rows); positions of one raster group share
        // an N-tile, so the heavy rows still reuse their weight tiles.
        int mixed = 0;
        if (p.mixed && !any_bad) {
            int lc = 0, hc = 0;
            for (int i = 0; i < per; ++i) {
                const int e = lane * per + i;
                if (e < E) {
                    const int nb = c.row_start[e + 1] - c.row_start[e];
                    if (nb == 1) ++lc;
                    else hc += nb;
                }
            }
            int li = lc, hi = hc;
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, li, o);
                const int b = __shfl_up_sync(0xffffffffu, hi, o);
                if (lane >= o) {
                    li += a;
                    hi += b;
                }
            }
            const int l = __shfl_sync(0xffffffffu, li, 31), h = __shfl_sync(0xffffffffu, hi, 31);
            const int P = l + h;
            li -= lc;  // this lane's first light index / heavy row index
            hi -= hc;
            // worth it when single-row experts make up a quarter of the rows or
            // more (mid: 34%, -2.5% GEMM time); with few of them, groups that
            // straddle two large experts lose weight reuse (DiT: +2.7%)
            if (l > 0 && h > 0 && P <= kMaxMixedRows && (p.mixed == 2 || 4 * l >= P)) {
                mixed = 1;
                for (int i = 0; i < per; ++i) {
                    const int e = lane * per + i;
                    if (e >= E) break;
                    const int nb = c.row_start[e + 1] - c.row_start[e];
                    if (nb == 1) {
                        c.mrow[((li + 1) * P + l - 1) / l - 1] = e;
                        ++li;
                    } else {
                        for (int bnd = 0; bnd < nb; ++bnd, ++hi) {
                            // smallest x with x - floor(x l / P) >= hi + 1; the row sits at x - 1
                            int x = hi * P / h + 1;
                            while (x - x * l / P < hi + 1) ++x;
                            c.mrow[x - 1] = e | (bnd << 9);
                        }
                    }
                }
            }
        }
        if (!mixed && !any_bad && c.row_start[E] <= kMaxMixedRows) {
            // expert order: the same row table, read by the tile decode
            for (int i = 0; i < per; ++i) {
                const int e = lane * per + i;
                if (e >= E) break;
                for (int r = c.row_start[e]; r < c.row_start[e + 1]; ++r) c.mrow[r] = e | ((r - c.row_start[e]) << 9);
            }
        }
        if (lane == 0) c.mixed = mixed;
        __syncwarp();
        if (p.schedule == 0 && c.row_start[E] <= kMaxMixedRows) {
            // segment starts of the interleaved tile order, S(b) for b = 0 .. P
            const TileSource src(c, p);
            for (int b = lane; b <= src.P; b += 32) c.seg[b] = b * src.P1 + src.l2_count(c, b - src.D - 1);
        }
        __syncwarp();
        if (lane == 0) {
            // expert waves for the comparison schedule: consecutive experts until
            // the wave's Linear-1 tiles fill the grid once
            int nw = 0;
            int tiles = 0;
            c.wave_row[0] = 0;
            c.wave_tile[0] = 0;
            int wr = 0;
            for (int e = 0; e < E; ++e) {
                const int r1 = c.row_start[e + 1];
                if (static_cast<long>(r1 - wr) * p.P1 >= gridDim.x / CG || e == E - 1) {
                    tiles += (r1 - wr) * (p.P1 + p.P2);
                    ++nw;
                    c.wave_row[nw] = r1;
                    c.wave_tile[nw] = tiles;
                    wr = r1;
                }
            }
            c.nwaves = nw;
        }
    }
    __syncthreads();
    if constexpr (CG == 2) cluster_sync_all();  // the peer's barriers exist before any remote use
    tc_fence_after();
    const uint32_t tmem_base = c.tmem_base;
    volatile int *abort_flag = &c.abort;
    const bool tr = p.trace != nullptr;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const TileSource src(c, p);
            int s = 0;
            uint32_t ph = 0;
            uint32_t uses = 0;
            bool ok = true;
            unsigned long long w_empty = 0, w_rows = 0, t0 = tr ? clock64() : 0;
            // A single CTA claims and publishes the next tile itself, once a
            // few stages of the current one are queued (the claim and its
            // decode then overlap the wait for free stages). In a pair both
            // producers take the tiles the second CTA's scheduler thread
            // publishes, off this thread's path.
            Tile next;
            unsigned claimed = 0;  // single CTA: ticket of the next tile, claimed at the current tile's first stage
            if (CG == 1) ok = publish_tile<CG>(c, p, src, 0, atomicAdd(p.ticket, 1u), next, abort_flag, 0u);
            for (int tl = 0; ok; ++tl) {
                Tile t;
                if (CG == 1) {
                    t = next;
                } else if (take_tile(c, p, tl, t, abort_flag)) {
                    release_tile<CG>(c, tl, rank);
                    if (rank == 1) mbar_arrive(&c.sched_go);  // the scheduler may publish the next one
                } else {
                    break;
                }
                if (t.kind < 0) break;
                unsigned long long *rec =
                    (p.tile_trace && tl < p.tile_trace_cap)
                        ? p.tile_trace + (static_cast<long>(blockIdx.x) * p.tile_trace_cap + tl) * kTileTraceWords
                        : nullptr;
                unsigned long long dep0 = rec ? clock64() : 0;
                const int e = t.e;
                const int band0 = t.b0;
                // this CTA's 128 rows of the scheduler row (tokens on the M side)
                const int row0 = band0 + static_cast<int>(rank) * kBlockM;
                // this CTA's first token of B (tokens on the N side)
                const int brow = TN ? band0 + static_cast<int>(rank) *
                                                  (tile_tokens(c.offs[e + 1] - band0, kTileRows) >> 1)
                                    : 0;
                // h rows of this scheduler row: slot (row mod Q) of the ring, or in place
                const int hoff = p.ring ? (t.row % p.ring) * kTileRows - band0 : 0;
                if (t.kind == 0 && p.ring && t.row >= p.ring) {
                    // the slot's previous row must be read by all its Linear-2 tiles
                    const unsigned long long tw = tr ? clock64() : 0;
                    if (!wait_rows_ready(&p.l2_done[t.row - p.ring], static_cast<unsigned>(CG * p.P2),
                                         abort_flag, p.status, 0x40000000u | static_cast<unsigned>(t.row),
                                         p.wait_ns))
                        break;
                    if (tr) w_rows += clock64() - tw;
                }
                if (t.kind == 1) {
                    const unsigned long long tw = tr ? clock64() : 0;
                    if (!wait_rows_ready(&p.l1_done[t.row],
                                         static_cast<unsigned>(CG * p.P1 + p.unmet_dependency),
                                         abort_flag, p.status, static_cast<unsigned>(t.row),
                                         p.wait_ns))
                        break;
                    if (tr) w_rows += clock64() - tw;
                    fence_proxy_async_global();
                }
                if (rec) {
                    const unsigned long long now = clock64();
                    rec[0] = static_cast<unsigned long long>(t.kind) |
                             (static_cast<unsigned long long>(t.row) << 2) |
                             (static_cast<unsigned long long>(t.n) << 34);
                    rec[1] = now;
                    rec[2] = t.kind == 1 ? now - dep0 : 0;
                }
                const int nkb = t.kind == 0 ? p.kb1 : p.kb2;
                // bytes of one stage summed over the CTAs of the pair
                const uint32_t bytes =
                    CG * ((TN || t.kind == 0) ? kATileBytes + kBTileBytes
                                              : kATileBytes + (p.N2 / CG) * kBlockK * 2);
                constexpr int kSlots = Cfg<CG, TN>::kSlots;
                for (int kb0 = 0; kb0 < nkb; kb0 += kSync) {
                    const int ns = min(kSync, nkb - kb0);
                    const unsigned long long tw = tr ? clock64() : 0;
                    if (!mbar_wait(&c.empty[s], ph ^ 1u, abort_flag, p.status, kWhereProducerEmpty,
                                   static_cast<unsigned>(s), p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (tr) w_empty += clock64() - tw;
                    // the pair's loads all complete on the first CTA's barrier
                    if (leader) mbar_arrive_expect_tx(&c.full[s], bytes * ns);
                    const uint32_t bar = CG == 2 ? map_to_cta(smem_u32(&c.full[s]), 0)
                                                 : smem_u32(&c.full[s]);
                    for (int j = 0; j < ns; ++j) {
                        const int kb = kb0 + j;
                        uint8_t *a = sA + (s * kSync + j) * kATileBytes;
                        uint8_t *b = sB + (s * kSync + j) * kBTileBytes;
                        if constexpr (TN) {
                            if (t.kind == 0) {
                                const int f = t.n * (kTnL1 * CG) + static_cast<int>(rank) * kTnL1;
                                tma_load_3d<CG>(&tm_w1, bar, a, kb * kBlockK, f, e);
                                tma_load_3d<CG>(&tm_w3, bar, a + kATileBytes / 2, kb * kBlockK, f, e);
                                tma_load_2d<CG>(&tm_x, bar, b, kb * kBlockK, brow);
                            } else {
                                tma_load_3d<CG>(&tm_w2, bar, a, kb * kBlockK,
                                                t.n * p.N2 + static_cast<int>(rank) * kTnL2, e);
                                tma_load_2d<CG>(&tm_h, bar, b, kb * kBlockK, brow + hoff);
                            }
                        } else if (t.kind == 0) {
                            tma_load_2d<CG>(&tm_x, bar, a, kb * kBlockK, row0);
                            if (CG == 1 || rank == 0)
                                tma_load_3d<CG>(&tm_w1, bar, b, kb * kBlockK, t.n * kL1N, e);
                            if (CG == 1 || rank == 1)
                                tma_load_3d<CG>(&tm_w3, bar, CG == 1 ? b + kBTileBytes / 2 : b,
                                                kb * kBlockK, t.n * kL1N, e);
                        } else {
                            tma_load_2d<CG>(&tm_h, bar, a, kb * kBlockK, row0 + hoff);
                            tma_load_3d<CG>(&tm_w2, bar, b, kb * kBlockK,
                                            t.n * p.N2 + static_cast<int>(rank) * (p.N2 / CG), e);
                        }
                    }
                    c.p_bytes[s] = bytes / CG * ns;
                    ++uses;
                    if (++s == kSlots) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if constexpr (CG == 1) {
                        if (kb0 == 0) claimed = atomicAdd(p.ticket, 1u);
                        const int pk = min(3, nkb - 1);
                        if (pk >= kb0 && pk < kb0 + ns &&
                            !publish_tile<CG>(c, p, src, tl + 1, claimed, next, abort_flag, 0u)) {
                            ok = false;
                            break;
                        }
                    }
                }
            }
            c.p_uses = uses;
            if (tr) {
                unsigned long long *o = p.trace + blockIdx.x * kTraceWords;
                o[0] = w_empty;
                o[1] = w_rows;
                o[2] = clock64() - t0;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && leader) {
            int s = 0;
            uint32_t ph = 0;
            const uint32_t idesc1 = idesc_bf16_f32(kTileRows, 2 * kL1N);
            const uint32_t idesc2 = idesc_bf16_f32(kTileRows, p.N2);
            bool ok = true;
            unsigned long long w_full = 0, w_tmem = 0, t0 = tr ? clock64() : 0;
            Tile t_next;
            ok = take_tile(c, p, 0, t_next, abort_flag);
            if (ok) release_tile<CG>(c, 0, rank);
            for (int tl = 0; ok; ++tl) {
                const Tile t = t_next;
                if (t.kind < 0) break;
                const int b = tl & 1;
                const uint32_t aph = static_cast<uint32_t>(tl >> 1) & 1u;
                unsigned long long tw = tr ? clock64() : 0;
                if (!mbar_wait(&c.tempty[b], aph ^ 1u, abort_flag, p.status, kWhereMmaTmemEmpty,
                               static_cast<unsigned>(tl), p.wait_ns))
                    break;
                if (tr) w_tmem += clock64() - tw;
                unsigned long long *rec =
                    (p.tile_trace && tl < p.tile_trace_cap)
                        ? p.tile_trace + (static_cast<long>(blockIdx.x) * p.tile_trace_cap + tl) * kTileTraceWords
                        : nullptr;
                unsigned long long tile_wait = 0;
                if (rec) rec[3] = clock64();
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b) * kAccCols;
                uint32_t idesc = t.kind == 0 ? idesc1 : idesc2;
                if constexpr (TN) {
                    const int band0 = t.b0;
                    idesc = idesc_bf16_f32(kBlockM * CG, tile_tokens(c.offs[t.e + 1] - band0, kTileRows));
                }
                const int nkb = t.kind == 0 ? p.kb1 : p.kb2;
                constexpr int kSlots = Cfg<CG, TN>::kSlots;
                for (int kb0 = 0; kb0 < nkb; kb0 += kSync) {
                    const int ns = min(kSync, nkb - kb0);
                    tw = (tr || rec) ? clock64() : 0;
                    if (!mbar_wait(&c.full[s], ph, abort_flag, p.status, kWhereMmaFull,
                                   static_cast<unsigned>(s), p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (tr || rec) {
                        const unsigned long long dw = clock64() - tw;
                        w_full += dw;
                        tile_wait += dw;
                    }
                    tc_fence_after();
                    for (int j = 0; j < ns; ++j) {
                        const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sA + (s * kSync + j) * kATileBytes));
                        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sB + (s * kSync + j) * kBTileBytes));
#pragma unroll
                        for (int kk = 0; kk < kBlockK / 16; ++kk)
                            mma_bf16_ss<CG>(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc,
                                            ((kb0 + j) | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit<CG>(&c.empty[s]);
                    if (++s == kSlots) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (kb0 + ns >= nkb) {
                        // the next descriptor, read while this tile's last MMAs run
                        if (!take_tile(c, p, tl + 1, t_next, abort_flag)) {
                            ok = false;
                            break;
                        }
                        release_tile<CG>(c, tl + 1, rank);
                    }
                }
                if (rec) {
                    rec[4] = clock64();
                    rec[5] = tile_wait;
                }
                if (ok) mma_commit<CG>(&c.tfull[b]);
            }
            // every issued MMA must finish before tensor memory is freed, also
            // when the loop was left early
            mma_commit<CG>(&c.drain, 1);
            if (!mbar_wait_drain(&c.drain, 0, p.wait_ns))
                report_failure(p.status, kStatusTimeout, kWhereMmaDrain, static_cast<unsigned>(s));
            if (tr) {
                unsigned long long *o = p.trace + blockIdx.x * kTraceWords;
                o[3] = w_full;
                o[4] = w_tmem;
                o[5] = clock64() - t0;
            }
        } else if (CG == 2 && lane == 0) {
            // ------------------------------------------------------------ pair scheduler
            // The second CTA's MMA warp, otherwise idle, claims the tickets and
            // publishes their tiles to both CTAs: tile tl + 1 once this CTA's
            // producer has taken tile tl, so both producers find it long
            // before they need it and neither spends time on the claim.
            const TileSource src(c, p);
            for (int tl = 0;; ++tl) {
                if (tl > 0 && !mbar_wait_cluster(&c.sched_go, static_cast<uint32_t>(tl - 1) & 1u, abort_flag,
                                                 p.status, kWhereTileQueue, 0x20000000u | static_cast<unsigned>(tl),
                                                 p.wait_ns))
                    break;
                Tile t;
                if (!publish_tile<CG>(c, p, src, tl, atomicAdd(p.ticket, 1u), t, abort_flag, 0u)) break;
                if (t.kind < 0) break;
            }
        }
    } else if (FC && warp >= kThreads / 32) {
        // ------------------------------------------------------------ combine consumers
        combine_consumer<CG, TN>(c, p, lane, abort_flag);
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // tensor-memory lane quarter this warp may read
        const bool publisher = (warp == 2 && lane == 0);
        unsigned long long w_full = 0, w_work = 0, w_stores = 0, n1 = 0, n2 = 0;
        const unsigned long long t0 = tr ? clock64() : 0;
        if (tr && publisher) p.trace[blockIdx.x * kTraceWords + 12] = globaltimer_ns();
        for (int tl = 0;; ++tl) {
            Tile t;
            // every lane waits for the descriptor; once all have read it, lane 0
            // gives the slot back
            const bool got = take_tile(c, p, tl, t, abort_flag);
            __syncwarp();
            if (lane == 0 && got) release_tile<CG>(c, tl, rank);
            const int b = tl & 1;
            const uint32_t aph = static_cast<uint32_t>(tl >> 1) & 1u;
            unsigned long long tw = tr ? clock64() : 0;
            // the whole warp agrees before its warp-collective tensor-memory loads
            const bool ready = got && (t.kind < 0 || mbar_wait(&c.tfull[b], aph, abort_flag, p.status,
                                                               kWhereEpiTmemFull, static_cast<unsigned>(tl),
                                                               p.wait_ns));
            bool go = __all_sync(0xffffffffu, ready);
            if constexpr (TN) {
                // warp pairs meet at named barriers below, so all four epilogue
                // warps leave together or not at all (a flag only ever set, read
                // after a barrier every warp reaches in this iteration)
                if (!go && lane == 0) c.epi_fail = 1;
                named_bar_sync(1, kEpiThreads);
                go = *reinterpret_cast<volatile int *>(&c.epi_fail) == 0;
            }
            if (!go) break;
            if (t.kind < 0) break;  // every warp read the same end marker
            unsigned long long *rec =
                (publisher && p.tile_trace && tl < p.tile_trace_cap)
                    ? p.tile_trace + (static_cast<long>(blockIdx.x) * p.tile_trace_cap + tl) * kTileTraceWords
                    : nullptr;
            if (rec) rec[6] = clock64();
            if (tr) {
                const unsigned long long now = clock64();
                w_full += now - tw;
                tw = now;
                if (t.kind == 0) ++n1;
                else ++n2;
            }
            tc_fence_after();
            const int e = t.e;
            const int row0 = t.b0 + static_cast<int>(rank) * kBlockM;
            if constexpr (TN) {
                // accumulator: lane = weight row, column = token. Per 32-token
                // slab each warp works alone: Linear-1 lanes l and l+16 hold
                // gate and up of one feature, one shuffle gives lane l tokens
                // 0-15 and lane l+16 tokens 16-31 of that feature; the bf16
                // results go token-major into the warp's shared-memory slab,
                // and lane j stores token j's contiguous columns.
                const int band0 = t.b0;
                const int valid = min(kTileRows, c.offs[e + 1] - band0);
                uint8_t *wslab = s_epi + (warp - 2) * kEpiStageBytes;
                const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>(b) * kAccCols;
                const int nch = (valid + 31) >> 5;
                for (int ch = 0; ch < nch; ++ch) {
                    uint32_t v[32];
                    tmem_load_32cols(tb + ch * 32, v);
                    const long grow = static_cast<long>(band0) + ch * 32 + lane;  // token row of this lane
                    const bool store = ch * 32 + lane < valid;
                    if (t.kind == 0) {
                        // q < 2: gate of features 32q + lane, finishes tokens 0-15;
                        // q >= 2: up of features 32(q-2) + lane, finishes tokens 16-31.
                        // Each warp sends the other half through its double-buffered
                        // 2 KiB mailbox ([16 tokens][32 lanes] fp32), then one
                        // barrier of the warp pair.
                        const bool gate_w = q < 2;
                        float *mine = reinterpret_cast<float *>(wslab + (ch & 1) * 2048);
                        const int pw = (q ^ 2) < 2 ? (q ^ 2) + 4 : (q ^ 2);  // partner warp (quarter q ^ 2)
                        const float *theirs = reinterpret_cast<const float *>(
                            s_epi + (pw - 2) * kEpiStageBytes + (ch & 1) * 2048);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            mine[i * 32 + lane] = __uint_as_float(gate_w ? v[16 + i] : v[i]);
                        named_bar_sync(2 + (q & 1), 64);
                        float hv[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float other = theirs[i * 32 + lane];
                            hv[i] = gate_w ? silu_mul(__uint_as_float(v[i]), other)
                                           : silu_mul(other, __uint_as_float(v[16 + i]));
                        }
                        // bf16 pairs of adjacent features, token-major: even lane
                        // takes token 2i, odd lane token 2i+1 ([16 tokens][16 words])
                        uint32_t *sl = reinterpret_cast<uint32_t *>(wslab + 4096);
                        const bool ev = (lane & 1) == 0;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float r = __shfl_xor_sync(0xffffffffu, ev ? hv[2 * i + 1] : hv[2 * i], 1);
                            sl[(2 * i + (ev ? 0 : 1)) * 16 + (lane >> 1)] =
                                ev ? pack_bf16x2(hv[2 * i], r) : pack_bf16x2(r, hv[2 * i + 1]);
                        }
                        __syncwarp();
                        // two lanes a token, 32 bytes each
                        const int tk = (gate_w ? 0 : 16) + (lane >> 1);
                        const int half = lane & 1;
                        const int col = t.n * (kTnL1 * CG) + static_cast<int>(rank) * kTnL1 + (q & 1) * 32 +
                                        half * 16;
                        const long hrow = static_cast<long>(band0) + ch * 32 + tk +
                                          (p.ring ? (t.row % p.ring) * kTileRows - band0 : 0);
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int j = jj ^ ((lane >> 2) & 1);  // spread the lanes over the banks
                            const uint4 val = *reinterpret_cast<const uint4 *>(
                                reinterpret_cast<const uint8_t *>(sl) + (tk & 15) * 64 + half * 32 + j * 16);
                            if (ch * 32 + tk < valid && col + 8 * j < p.F)
                                *reinterpret_cast<uint4 *>(p.h + hrow * p.F + col + 8 * j) = val;
                        }
                    } else {
                        // even lane: (row, row+1) of token 2i; odd lane: of token 2i+1
                        const bool ev = (lane & 1) == 0;
                        uint32_t *sl = reinterpret_cast<uint32_t *>(wslab);  // [32 tokens][16 words]
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const uint32_t r = __shfl_xor_sync(0xffffffffu, ev ? v[2 * i + 1] : v[2 * i], 1);
                            const float lo_v = __uint_as_float(ev ? v[2 * i] : r);
                            const float hi_v = __uint_as_float(ev ? r : v[2 * i + 1]);
                            sl[(2 * i + (ev ? 0 : 1)) * 16 + (lane >> 1)] = pack_bf16x2(lo_v, hi_v);
                        }
                        __syncwarp();
                        const int col = t.n * p.N2 + static_cast<int>(rank) * kTnL2 + q * 32;
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int j = (jj + (lane >> 1)) & 3;  // spread the lanes over the banks
                            const uint4 val = *reinterpret_cast<const uint4 *>(wslab + lane * 64 + j * 16);
                            if (store && col + 8 * j < p.d)
                                *reinterpret_cast<uint4 *>(p.y + grow * p.d + col + 8 * j) = val;
                        }
                    }
                    __syncwarp();
                }
            } else {
                const int valid_rows = min(kBlockM, c.offs[e + 1] - row0);  // may be <= 0
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(b) * kAccCols;
                // 64 columns at a time: tensor memory -> registers (thread = row) ->
                // swizzled shared-memory transpose -> 16-byte stores that cover four
                // full 128-byte row segments per warp instruction.
                uint8_t *stg = s_epi + (warp - 2) * kEpiStageBytes;
                const int nchunks = t.kind == 0 ? kL1N / 64 : p.N2 / 64;
                // h rows go to the row's ring slot when the ring is on
                const long hoff = (t.kind == 0 && p.ring)
                                      ? static_cast<long>(t.row % p.ring) * kTileRows - t.b0
                                      : 0;
                uint16_t *const out_base = t.kind == 0 ? p.h + hoff * p.F : p.y;
                const int out_ld = t.kind == 0 ? p.F : p.d;
                const int col_base = t.kind == 0 ? t.n * kL1N : t.n * p.N2;
                for (int ch = 0; ch < nchunks; ++ch) {
                    uint32_t pk[32];
                    if (t.kind == 0) {
                        uint32_t g[64], u[64];
                        tmem_load_2x64cols(tbase + ch * 64, tbase + kL1N + ch * 64, g, u);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            pk[i] = pack_bf16x2(silu_mul(g[2 * i], u[2 * i]),
                                                silu_mul(g[2 * i + 1], u[2 * i + 1]));
                    } else {
                        uint32_t a[64];
                        tmem_load_64cols(tbase + ch * 64, a);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            pk[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
                    }
                    // row `lane` of the warp's 32-row slab: 8 pieces of 16 B, piece j at
                    // slot j ^ (lane & 7) (conflict-free writes and reads)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4 *>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    __syncwarp();
                    const int piece = lane & 7;
                    const int col = col_base + ch * 64 + piece * 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = i * 4 + (lane >> 3);  // row within the warp's slab
                        const uint4 v =
                            *reinterpret_cast<const uint4 *>(stg + r * 128 + ((piece ^ (r & 7)) << 4));
                        if (q * 32 + r < valid_rows && col < out_ld)
                            *reinterpret_cast<uint4 *>(out_base + (static_cast<long>(row0) + q * 32 + r) *
                                                                      out_ld + col) = v;
                    }
                    __syncwarp();
                }
            }
            // this thread's stores before any later TMA read of them (other CTAs)
            fence_proxy_async_global();
            tc_fence_before();
            mbar_arrive(&c.estore[b]);
            if constexpr (CG == 2)
                mbar_arrive_cluster(map_to_cta(smem_u32(&c.tempty[b]), 0));
            else
                mbar_arrive(&c.tempty[b]);
            if (tr) {
                const unsigned long long now = clock64();
                w_work += now - tw;
                tw = now;
            }
            if (publisher) {
                // all 128 epilogue threads have stored: publish the tile
                const bool stored = mbar_wait(&c.estore[b], aph, abort_flag, p.status,
                                              kWhereEpiTmemFull, 0x80000000u | static_cast<unsigned>(tl),
                                              p.wait_ns);
                if (tr) w_stores += clock64() - tw;
                if (rec) rec[7] = clock64();
                if (stored) {
                    __threadfence();
                    if (t.kind == 0) {
                        red_release_add_u32(&p.l1_done[t.row], 1u);
                    } else {
                        st_release_u32(
                            &p.l2_flags[(static_cast<long>(t.row) * p.P2 + t.n) * CG + rank],
                            p.epoch);
                        if (p.ring || p.fc) red_release_add_u32(&p.l2_done[t.row], 1u);
                    }
                }
            }
            __syncwarp();
        }
        // with the fused combine, the epilogue warps turn consumers once their
        // tiles are done (unless a wait gave up)
        if constexpr (FC)
            if (!*abort_flag && ld_volatile_u32(p.status) == 0u)
                combine_consumer<CG, TN>(c, p, lane, abort_flag);
        if (tr && publisher) {
            unsigned long long *o = p.trace + blockIdx.x * kTraceWords;
            o[6] = w_full;
            o[7] = w_work;
            o[8] = w_stores;
            o[9] = clock64() - t0;
            o[10] = n1;
            o[11] = n2;
            o[13] = globaltimer_ns();
        }
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync_all();  // both producers have stopped issuing loads
    // every TMA load the CTA (pair) issued has landed before its shared memory
    // is released: on the normal path the MMA thread consumed them all and
    // these waits return at once; after an early exit they cover the loads
    // still in flight
    if (warp == 0 && lane == 0 && leader) drain_loads<CG, Cfg<CG, TN>::kSlots>(c, p);
    __syncwarp();
    if constexpr (CG == 2) cluster_sync_all();  // the peer stays until its loads have landed too
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, kTmemCols);
    }
}

bool make_map_2d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer)
{
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_3d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t mid, uint64_t outer,
                 uint32_t box_inner, uint32_t box_mid)
{
    const cuuint64_t dims[3] = {inner, mid, outer};
    const cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
    const cuuint32_t box[3] = {box_inner, box_mid, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int ffn_l2_block_n(int d, int requested)
{
    if (requested >= 64 && requested <= 256 && requested % 64 == 0) return requested;
    // fewest tiles, then fewest padded columns: a k-block costs about the same
    // for any tile width up to 256 (the loop is paced by delivering and issuing
    // stages, not by the MMA width), so a narrower tile only adds k-blocks
    int best = 256;
    long best_tiles = LONG_MAX, best_pad = LONG_MAX;
    for (int n = 256; n >= 64; n -= 64) {
        const long tiles = (d + n - 1) / n;
        const long pad = tiles * n - d;
        if (tiles < best_tiles || (tiles == best_tiles && pad < best_pad)) {
            best_tiles = tiles;
            best_pad = pad;
            best = n;
        }
    }
    return best;
}

long ffn_max_rows(long R, int E)
{
    // 128-row M-tiles: sum_e ceil(c_e / 128) <= R / 128 + E; CTA pairs use
    // (R / 256 + E) scheduler rows with two flags per Linear-2 tile
    return R / kBlockM + 2L * E + 2;
}

namespace {

template <int CG, bool TN, bool FC>
cudaError_t launch_cg(const FfnArgs &a, GemmParams p, cudaStream_t stream)
{
    constexpr size_t smem = smem_bytes<CG, TN>();
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(FC ? kThreads + kConsumerThreads : kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // once per device: the shared-memory attribute, and how many instances
    // (CTAs or CTA pairs) can be resident at once -- every CTA of the
    // persistent grid must be (the Linear-2 tiles wait on Linear-1 tiles of
    // other CTAs)
    struct Tag {};
    static int max_inst[kOnceDevices];
    auto init = [&](int dev) -> cudaError_t {
        cudaError_t err = cudaFuncSetAttribute(grouped_swiglu_gemm_kernel<CG, TN, FC>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        int clusters = 0;
        cudaLaunchConfig_t occ = cfg;
        occ.gridDim = dim3(static_cast<unsigned>(sms / CG * CG), 1, 1);
        err = cudaOccupancyMaxActiveClusters(&clusters, grouped_swiglu_gemm_kernel<CG, TN, FC>, &occ);
        if (err != cudaSuccess) return err;
        const int m = clusters < sms / CG ? clusters : sms / CG;
        if (m <= 0) return cudaErrorInvalidConfiguration;
        if (dev >= 0 && dev < kOnceDevices) max_inst[dev] = m;
        return cudaSuccess;
    };
    const cudaError_t ierr = once_per_device<Tag>(init);
    if (ierr != cudaSuccess) return ierr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    int max_instances = 0;
    if (dev >= 0 && dev < kOnceDevices) {
        max_instances = max_inst[dev];
    } else {
        // no cached slot: query again (the attribute was set just now)
        int clusters = 0;
        cudaLaunchConfig_t occ = cfg;
        occ.gridDim = dim3(static_cast<unsigned>(sms / CG * CG), 1, 1);
        const cudaError_t err =
            cudaOccupancyMaxActiveClusters(&clusters, grouped_swiglu_gemm_kernel<CG, TN, FC>, &occ);
        if (err != cudaSuccess) return err;
        max_instances = clusters < sms / CG ? clusters : sms / CG;
        if (max_instances <= 0) return cudaErrorInvalidConfiguration;
    }
    int instances = max_instances;
    if (a.num_ctas > 0) {
        const int want = a.num_ctas / CG > 0 ? a.num_ctas / CG : 1;
        if (want < instances) instances = want;
    }
    // lead of Linear-1 over Linear-2 (scheduler rows). The minimum is a raster
    // group (every tile of a row sits below position (row + group) * P1) plus
    // the rows the instances have in flight; tiles finish out of order, and
    // below about twice that Linear-2 producers start to wait, so the default
    // is twice the minimum plus one row. Never below the group size: that
    // bound keeps the dependency waits deadlock-free.
    p.lead = a.lead > 0 ? a.lead : 2 * (p.group + (instances + p.P1 - 1) / p.P1) + 1;
    if (p.lead < p.group) p.lead = p.group;
    if (p.ring) {
        // a ring of Q rows bounds the lead: Q >= D + 2 * group (see TileSource)
        if (p.ring < 3 * p.group || p.schedule != 0) return cudaErrorInvalidConfiguration;
        if (p.lead > p.ring - 2 * p.group) p.lead = p.ring - 2 * p.group;
    }

    const long R = a.R;
    CUtensorMap tx, th, tw1, tw3, tw2;
    // token boxes: the A rows with tokens on the M side, this CTA's B rows (all
    // of a single CTA's up to 256 tokens, half of a pair's) on the N side
    const uint32_t tok_box = TN ? 256 / CG : kBlockM;
    if (!make_map_2d(&tx, a.x_perm, a.d, R, kBlockK, tok_box) ||
        !make_map_2d(&th, a.h, a.F, p.ring ? static_cast<long>(p.ring) * Cfg<CG, TN>::kTileRows : R, kBlockK,
                     tok_box) ||
        !make_map_3d(&tw1, a.w1, a.d, a.F, a.E, kBlockK, TN ? kL1N / 2 : kL1N) ||
        !make_map_3d(&tw3, a.w3, a.d, a.F, a.E, kBlockK, TN ? kL1N / 2 : kL1N) ||
        !make_map_3d(&tw2, a.w2, a.F, a.d, a.E, kBlockK, TN ? kBlockM : p.N2 / CG))
        return cudaErrorInvalidValue;

    if (!a.counters_zeroed) {
        // l1_done, l2_done right after it, then the tile ticket
        cudaError_t err = cudaMemsetAsync(a.l1_done, 0, sizeof(unsigned) * (2 * a.max_rows + 1), stream);
        if (err != cudaSuccess) return err;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(instances * CG), 1, 1);
    cfg.numAttrs = 2;  // + programmatic dependent launch (the occupancy query used the cluster alone)
    return cudaLaunchKernelEx(&cfg, grouped_swiglu_gemm_kernel<CG, TN, FC>, tx, th, tw1, tw3, tw2, p);
}

}  // namespace

cudaError_t launch_ffn(const FfnArgs &a, cudaStream_t stream)
{
    if (a.R == 0) return cudaSuccess;
    GemmParams p;
    p.offsets = a.offsets;
    p.h = a.h;
    p.y = a.y;
    p.l1_done = a.l1_done;
    p.l2_done = a.l1_done + a.max_rows;
    p.ticket = a.l1_done + 2 * a.max_rows;
    p.ring = a.h_ring_rows;
    // mixed row order: asked for (or by default) with the interleaved schedule;
    // not with the fused combine, whose consumers walk rows in expert order
    // 2 = asked for: taken whenever both kinds of experts exist; 1 = default:
    // taken when single-row experts are a quarter of the rows or more
    p.mixed = (a.schedule == 0 && a.gate == nullptr)
                  ? (a.row_order == 2 ? 2 : (a.row_order == 0 && kMixedByDefault) ? 1 : 0)
                  : 0;
    p.l2_flags = a.l2_flags;
    p.status = a.status;
    p.E = a.E;
    p.d = a.d;
    p.F = a.F;
    p.R = a.R;
    // CTA pairs halve the operand traffic per MMA. With tokens on the M side
    // they pad every expert to 256-row tiles, so below ~1024 rows per expert
    // single CTAs win there; with tokens on the N side an expert pads to 16
    // tokens. Tokens go on the N side unless Linear-2's 256-wide weight tiles
    // would pad y (d not a multiple of 256) on large experts.
    const bool big_experts = a.R / a.E >= 1024;
    bool tn;
    if (a.orientation == 2)
        tn = true;
    else if (a.orientation == 1 || a.cta_group == 1)
        tn = false;
    else
        tn = a.d % 256 == 0 || !big_experts;
    if (tn)
        p.cg = a.cta_group == 1 ? 1 : 2;
    else if (a.cta_group == 1 || a.cta_group == 2)
        p.cg = a.cta_group;
    else
        p.cg = big_experts ? 2 : 1;
    p.rows = tn ? 256 : p.cg * kBlockM;
    p.N2 = tn ? p.cg * kBlockM : ffn_l2_block_n(a.d, a.l2_block_n);
    const int l1n = tn ? 64 * p.cg : kL1N;  // h columns per Linear-1 tile
    p.P1 = (a.F + l1n - 1) / l1n;
    p.P2 = (a.d + p.N2 - 1) / p.N2;
    p.kb1 = (a.d + kBlockK - 1) / kBlockK;
    p.kb2 = (a.F + kBlockK - 1) / kBlockK;
    p.schedule = a.schedule;
    p.epoch = a.epoch;
    p.trace = a.trace;
    p.tile_trace = a.tile_trace;
    p.tile_trace_cap = a.tile_trace_cap;
    p.wait_ns = a.wait_limit_us > 0 ? 1000ull * static_cast<unsigned long long>(a.wait_limit_us)
                                    : kWaitLimitNs;
    p.unmet_dependency = a.unmet_dependency > 0 ? 1 : 0;
    // raster group (128-row M-tiles): with few rows per expert a smaller group
    // keeps fewer experts' weight tiles in flight in L2 (fine, E = 256 with two
    // 256-token rows per expert: 1.9-4% less GEMM time; with 8-16 rows per
    // expert the default group is as fast or faster)
    const long rows_per_expert = static_cast<long>(a.R) / (static_cast<long>(a.E) * 256);
    const int group = a.group_rows > 0 ? a.group_rows
                                       : (rows_per_expert < 4 ? kSmallExpertGroupRows : kDefaultGroupRows);
    p.group = (group + p.cg - 1) / p.cg;                                     // scheduler rows
    p.fc = a.gate != nullptr ? 1 : 0;
    if (p.fc) {
        p.gate = a.gate;
        p.row_of_slot = a.row_of_slot;
        p.slot_of_row = a.slot_of_row;
        p.T = a.T;
        p.k = a.k;
        p.rows_per_seg = a.T / a.S;
        for (int i = 0; i < kMaxSegments; ++i) p.seg[i] = i < a.S ? a.seg[i] : nullptr;
        if (tn) return p.cg == 1 ? launch_cg<1, true, true>(a, p, stream) : launch_cg<2, true, true>(a, p, stream);
        if (p.cg == 1) return launch_cg<1, false, true>(a, p, stream);
        return launch_cg<2, false, true>(a, p, stream);
    }
    if (tn) return p.cg == 1 ? launch_cg<1, true, false>(a, p, stream) : launch_cg<2, true, false>(a, p, stream);
    if (p.cg == 1) return launch_cg<1, false, false>(a, p, stream);
    return launch_cg<2, false, false>(a, p, stream);
}

}  // namespace moe
