// gemm_dec.cu -- the dequant-fused GEMM for one token tile of at most 160
// rows (the decode step of a block), with the dequantised weights in TMEM.
//
// Computes exactly what gemm.cu's kernel computes: Y = act(X W^T + bias) +
// residual with W stored 4-bit in groups of 64 along k and every weight
// dequantised on chip to w^ = fp16(fma(c, scale, min)) ("FlexGen 完全拆解",
// compression section: stored tensors are dequantised to FP16 before
// compute).  Same operand mapping: 128 weight rows are the MMA's M, the
// block's rows (nt <= 160) its N, so each weight tile is fetched from HBM and
// dequantised once per block.  What differs, and why (measured on GB300):
//
//  * A (the dequantised 128 x 128 weight tile of a stage) is written from
//    registers straight into TMEM (tcgen05.st) and the MMAs read it there.
//    With both operands in shared memory a 128 x 144 x 16 MMA takes 117
//    cycles (shared-memory bandwidth); with A in TMEM it takes 72.
//  * A stage is 128 k: 8 MMAs per barrier wait and commit.  Each wait and
//    commit costs ~150 cycles of the issuing warp that the MMAs do not hide at
//    this N (the MMA queue is about one deep).
//  * The MMA loop runs on the whole warp (warp-uniform control flow and
//    descriptors, advanced by additions) and lane 0 alone issues the MMAs and
//    commits: the warp shares its sub-partition with three dequantising
//    warps, and an issue loop inside a one-lane branch measured ~65 cycles
//    per MMA there, against ~45 for the MMA itself at small N.
//  * Three dequantising groups of four warps (one warp per TMEM lane
//    quarter: a warp can only reach the 32 lanes of its sub-partition) work
//    on three stages at once; the exact fp32 dequantisation runs at about 25
//    weights per cycle per SM, the throughput that bounds this kernel.
//  * Two accumulators in TMEM: the epilogue of one segment overlaps the main
//    loop of the next.
//  * Work is split evenly over persistent 2-CTA clusters (1 CTA per SM).  The
//    unit is (a pair of adjacent 128-row weight tiles, one 256-k codes box);
//    the units are dealt out as contiguous ranges, so every SM does the same
//    number of boxes whatever the tile count.  The two CTAs of a cluster take
//    the two tiles of a pair and share each activation stage through TMA
//    multicast.  A tile whose boxes fall to several clusters is summed in a
//    fixed order: the cluster holding the tile's first box keeps its part in
//    TMEM and, after its last box, adds the later parts in k order (each
//    written once to global memory by the cluster that computed it, behind a
//    release/acquire flag tagged with the launch's epoch), then runs the
//    epilogue.  The split depends on (N, K) and the number of clusters only,
//    never on M, so every row's result is independent of the other rows.
//  * The residual (out and fc2 projections) reaches the epilogue as a tile
//    in shared memory, loaded by TMA while the segment's main loop runs:
//    read by each thread from global memory, 2 bytes at a time and late in
//    the segment, it cost 7-10 % of those launches (measured by leaving the
//    loads out).
//
// Warp roles (640 threads): warp 0 = TMA producer of codes boxes and their
// (min, scale); warp 1 = TMEM allocator and the single MMA-issuing thread;
// warp 2 = TMA producer of this CTA's slice of the activation stages
// (multicast to the cluster); warp 3 = TMA producer of residual tiles;
// warps 4-7 = epilogue, one per TMEM lane quarter; warps 8-19 =
// dequantisers, group g = warps 8+4g .. 11+4g, the warp of lane quarter q
// owning weight rows 32q..32q+31 (one row per thread).
//
// Every wait (mbarrier or flag) is bounded; a wait that expires flags the CTA
// to stop, records a timeout in the device status word, waits for its own
// copies and MMAs in flight, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "fg_internal.cuh"

namespace {

using namespace fgd;

constexpr int kTileF = 128;             // weight rows per CTA (MMA M)
constexpr int kBoxK = 256;              // k per codes box (128 code bytes per row)
constexpr int kStageK = 128;            // k per pipeline stage (8 MMAs of k 16)
constexpr int kACols = kStageK / 2;     // TMEM columns of one A stage (two fp16 per column)
constexpr int kMaxNt = 144;             // activation rows (MMA N) this kernel takes
constexpr int kAccStride = 144;         // TMEM columns per accumulator
constexpr int kABase = 2 * kAccStride;  // first TMEM column of the A ring
constexpr int kNS = 3;                  // stages: A in TMEM, B in shared memory
constexpr int kG = 3;                   // dequant groups in flight
constexpr int kSC = 4;                  // codes boxes in flight
constexpr int kDecMinUnits = 3;         // units (256-k boxes of a tile pair) per cluster, at least
constexpr int kThreads = 32 * (8 + 4 * kG);
constexpr uint32_t kCBytes = kTileF * kBoxK / 2;      // 16 KB of packed codes
constexpr uint32_t kMBytes = kTileF * (kBoxK / 64) * 8;   // 4 KB of (min, scale)
constexpr uint32_t kRBytes = kMaxNt * kTileF * 2;         // the residual tile of a Y segment
static_assert(kABase + kNS * kACols <= 512, "TMEM columns");
static_assert(kMaxNt <= kAccStride, "accumulator width");
// A parity wait on an mbarrier tells the current phase from the previous one
// only: a dequant group jumps kG stages at a time, so the A ring needs at
// least kG stages (its previous stage then keeps the barrier at most one
// phase behind).  Codes boxes: a group's previous stage is at most two boxes
// back, so kSC >= 2 suffices.
static_assert(kNS >= kG && kSC >= 2, "parity rule");

struct DecParams {
    const __half* bias;        // [N] or null
    const __half* residual;    // [M][N] or null
    __half* Y;                 // [M][N]
    float* partial;            // [Q * c][nt][128] fp32 (parts of split tiles)
    unsigned long long* flags; // [Q * c][4 lane quarters]: epoch once that part is written
    unsigned long long epoch;
    long long units;           // pairs * nbox
    int M, N, K;
    int nt;                    // MMA N (activation rows, multiple of 16)
    int c;                     // CTAs per cluster (1 or 2)
    int nbox;                  // K / 256
    int Q;                     // clusters
    int act;
    int* status;
    unsigned long long wait_ns;
    int drop_arrive;
};

// Units [lo, hi) of cluster q: an even split of `units` over Q clusters.
__device__ __forceinline__ long long range_lo(long long units, int Q, int q) {
    return units * q / Q;
}

// Segments of a cluster's range: maximal runs of units in one tile pair.
struct SegIter {
    long long u, hi;
    int nbox;
    int t, b0, b1;   // current segment: pair t, boxes [b0, b1)
    __device__ bool next() {
        if (u >= hi) return false;
        t = static_cast<int>(u / nbox);
        b0 = static_cast<int>(u - static_cast<long long>(t) * nbox);
        const long long end = static_cast<long long>(t + 1) * nbox;
        const long long e = hi < end ? hi : end;
        b1 = static_cast<int>(e - static_cast<long long>(t) * nbox);
        u = e;
        return true;
    }
};

// Shared memory (offsets from a 1024-aligned base):
//   B ring  [kNS][2 halves][nt][128 B]   (k 0-63 and 64-127 of the stage,
//                                          128-byte swizzled, K-major)
//   codes   [kSC][128 rows][128 B]       (128-byte swizzled)
//   meta    [kSC][128 rows][4][2] fp32
//   resid   [nt][128] fp16                 (residual rows of the current Y tile)
//   barriers, TMEM address slot, abort flag
struct Smem {
    uint32_t base, b0, c0, m0, r0, bars;
    uint32_t half_bytes;   // nt * 128
    __device__ uint32_t b(int s) const { return b0 + static_cast<uint32_t>(s) * 2u * half_bytes; }
    __device__ uint32_t c(int s) const { return c0 + static_cast<uint32_t>(s) * kCBytes; }
    __device__ uint32_t m(int s) const { return m0 + static_cast<uint32_t>(s) * kMBytes; }
    __device__ uint32_t full(int s) const { return bars + 8u * s; }
    __device__ uint32_t empty(int s) const { return bars + 8u * (kNS + s); }
    __device__ uint32_t c_full(int s) const { return bars + 8u * (2 * kNS + s); }
    __device__ uint32_t c_empty(int s) const { return bars + 8u * (2 * kNS + kSC + s); }
    __device__ uint32_t acc_full(int a) const { return bars + 8u * (2 * kNS + 2 * kSC + a); }
    __device__ uint32_t acc_empty(int a) const { return bars + 8u * (2 * kNS + 2 * kSC + 2 + a); }
    __device__ uint32_t drain() const { return bars + 8u * (2 * kNS + 2 * kSC + 4); }
    __device__ uint32_t res_full() const { return bars + 8u * (2 * kNS + 2 * kSC + 5); }
    __device__ uint32_t res_empty() const { return bars + 8u * (2 * kNS + 2 * kSC + 6); }
    __device__ uint32_t res_last() const { return bars + 8u * (2 * kNS + 2 * kSC + 7); }
    __device__ uint32_t end() const { return bars + 8u * (2 * kNS + 2 * kSC + 8); }
};

// res: the launch has a residual (its tiles are staged in shared memory);
// without one the L1 cache keeps those 36 KB.
__host__ __device__ constexpr size_t dec_smem_bytes(int nt, bool res) {
    return 1024 + static_cast<size_t>(kNS) * 2 * nt * 128 + kSC * (kCBytes + kMBytes) + (res ? kRBytes : 0) +
           8 * (2 * kNS + 2 * kSC + 8) + 16;
}
static_assert(dec_smem_bytes(kMaxNt, true) <= 227 * 1024, "shared memory");

__global__ void __launch_bounds__(kThreads, 1)
    gemm_dec_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmM, const __grid_constant__ CUtensorMap tmR,
                    const DecParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Smem sm;
    sm.base = (raw + 1023u) & ~1023u;
    sm.half_bytes = static_cast<uint32_t>(p.nt) * 128u;
    sm.b0 = sm.base;
    sm.c0 = sm.b0 + kNS * 2u * sm.half_bytes;
    sm.m0 = sm.c0 + kSC * kCBytes;
    sm.r0 = sm.m0 + kSC * kMBytes;
    sm.bars = sm.r0 + (p.residual != nullptr ? kRBytes : 0u);
    uint8_t* const gen = smem_raw - raw;   // generic pointer = gen + shared address
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gen + sm.end());
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = p.c;
    const uint32_t crank = cluster_ctarank();
    const uint16_t cmask = static_cast<uint16_t>((1u << c) - 1u);
    const int q = static_cast<int>(blockIdx.x) / c;   // cluster index
    SegIter proto;
    proto.u = range_lo(p.units, p.Q, q);
    proto.hi = range_lo(p.units, p.Q, q + 1);
    proto.nbox = p.nbox;
    const int nstages = static_cast<int>(2 * (proto.hi - proto.u));
    const uint64_t lim = p.wait_ns;
    // The weights (codes and (min, scale)) never change during a step: their
    // loads and dequantisation start at once, possibly while the previous
    // kernel of the stream still runs; the roles that read activations,
    // residuals, partial sums or flags, or write Y, first wait for it.
    griddep_launch();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            // full: the activation producer's arrive (+ B bytes) and the 4 warps
            // of the dequant group that wrote the stage's A into TMEM
            mbar_init(sm.full(s), 1 + 4);
            // empty: one MMA commit from every CTA of the cluster (frees the
            // local A and the multicast B of the stage)
            mbar_init(sm.empty(s), c);
        }
        for (int s = 0; s < kSC; ++s) {
            mbar_init(sm.c_full(s), 1);
            mbar_init(sm.c_empty(s), 2 * 4);   // both stages of the box, 4 warps each
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(sm.acc_full(a), 1);
            mbar_init(sm.acc_empty(a), 4);     // the 4 epilogue warps
        }
        mbar_init(sm.drain(), 1);
        mbar_init(sm.res_full(), 1);
        mbar_init(sm.res_empty(), 4);   // the 4 epilogue warps, after each Y segment
        mbar_init(sm.res_last(), 1);
        // A wait that expired earlier (status not yet cleared by fg_check)
        // makes every later cluster skip its work instead of waiting again.
        *abort_flag = (p.status != nullptr && *reinterpret_cast<volatile int*>(p.status) != 0);
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmC);
        prefetch_tmap(&tmM);
        if (p.residual != nullptr) prefetch_tmap(&tmR);
    }
    __syncthreads();
    // Every barrier of every CTA in the cluster exists before any multicast.
    cluster_sync_all();
    {
        // the skip decision of rank 0 holds for the whole cluster
        const uint32_t f0 = ld_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), 0));
        if (f0 != 0) {
            cluster_sync_all();   // nobody reads rank 0's flag after it leaves
            return;               // uniform across the cluster: nothing issued yet
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        *abort_flag = 1;
        report(p.status, fg::kDevTimeout);
    };
    // The flags' tag: the launch's own value, changed by the count of errors
    // fg_check has cleared, so flags left set by a launch that timed out can
    // never match a later replay of it.
    const unsigned long long epoch =
        p.epoch ^ (p.status != nullptr
                       ? static_cast<unsigned long long>(
                             static_cast<uint32_t>(reinterpret_cast<volatile int*>(p.status)[1]) & 0xFFFFu)
                             << 32
                       : 0ull);

    // Later parts of the tile whose first part ends this cluster's range:
    // computed by clusters q + 1, q + 2, ... (in k order), each published by
    // a flag per lane quarter.  Returns how many there are (0: the tile is
    // whole here); clears ok on a timeout.
    auto wait_parts = [&](int t, int b1, int qq, bool& ok) -> int {
        if (b1 >= p.nbox) return 0;
        int nparts = 0;
        const long long tile_end = static_cast<long long>(t + 1) * p.nbox;
        for (int r = q + 1; r < p.Q; ++r) {
            const unsigned long long* f = p.flags + (r * c + static_cast<int>(crank)) * 4 + qq;
            const uint64_t t0 = globaltimer();
            bool got = true;
            while (ld_acquire_u64(f) != epoch) {
                if (*abort_flag || globaltimer() - t0 > lim) {
                    got = false;
                    break;
                }
            }
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                return nparts;
            }
            ++nparts;
            if (range_lo(p.units, p.Q, r + 1) >= tile_end) break;
        }
        return nparts;
    };
    // Y = act(acc + later parts + bias) + residual for one weight row n per
    // thread (the TMEM lanes of its quarter), 8-column chunks c_first,
    // c_first + c_step, ...  The residual comes from the segment's tile in
    // shared memory; every partial-sum load of a round is issued before the
    // first add, so their latencies overlap; the parts are added in k order.
    const __half* rbuf = reinterpret_cast<const __half*>(gen + sm.r0);
    auto y_epilogue = [&](uint32_t acc, int n, int row, int nparts, int c_first, int c_step) {
        const float bias = (p.bias != nullptr && n < p.N) ? __half2float(p.bias[n]) : 0.0f;
        const bool nv = n < p.N;
        if (nparts >= 2) {
            // Several later parts: one 8-column chunk per round with up to
            // three parts' loads in flight together (one L2 round trip for
            // three parts instead of three).
            for (int c0 = 8 * c_first; c0 < p.nt; c0 += 8 * c_step) {
                uint32_t r0[8];
                __syncwarp();
                tmem_ld8(acc + static_cast<uint32_t>(c0), r0);
                tmem_wait_ld();
                if (!nv) continue;
                float v0[8], res0[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    res0[j] = (p.residual != nullptr && c0 + j < p.M)
                                  ? __half2float(rbuf[(c0 + j) * kTileF + row])
                                  : 0.0f;
                    v0[j] = __uint_as_float(r0[j]);
                }
                for (int u0 = 0; u0 < nparts; u0 += 3) {
                    float pv[3][8];
#pragma unroll
                    for (int u = 0; u < 3; ++u) {
                        const bool has = u0 + u < nparts;
                        const float* src =
                            p.partial +
                            static_cast<size_t>(has ? (q + 1 + u0 + u) * c + static_cast<int>(crank) : 0) *
                                p.nt * kTileF +
                            row + c0 * kTileF;
#pragma unroll
                        for (int j = 0; j < 8; ++j) pv[u][j] = has ? __ldcg(src + j * kTileF) : 0.0f;
                    }
#pragma unroll
                    for (int u = 0; u < 3; ++u)
                        if (u0 + u < nparts) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) v0[j] = __fadd_rn(v0[j], pv[u][j]);
                        }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int m = c0 + j;
                    if (m >= p.M) break;
                    float x = __fadd_rn(v0[j], bias);
                    if (p.act == FG_ACT_RELU) x = fmaxf(x, 0.0f);
                    if (p.residual) x = __fadd_rn(x, res0[j]);
                    p.Y[static_cast<int64_t>(m) * p.N + n] = __float2half_rn(x);
                }
            }
            return;
        }
        // At most one later part: two 8-column chunks per round (c0 and
        // c0 + 8 c_step), the part's loads of both issued before the first
        // add, so a round costs one L2 round trip for 16 columns.
        for (int c0 = 8 * c_first; c0 < p.nt; c0 += 16 * c_step) {
            const int c1 = c0 + 8 * c_step;
            const bool two = c1 < p.nt;            // warp-uniform
            uint32_t r0[8], r1[8];
            __syncwarp();   // the stores of the previous round diverge
            tmem_ld8(acc + static_cast<uint32_t>(c0), r0);
            if (two) tmem_ld8(acc + static_cast<uint32_t>(c1), r1);
            tmem_wait_ld();
            if (!nv) continue;
            float v0[8], v1[8], res0[8], res1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const bool has_r = p.residual != nullptr;
                res0[j] = (has_r && c0 + j < p.M)
                              ? __half2float(rbuf[(c0 + j) * kTileF + row])
                              : 0.0f;
                res1[j] = (has_r && two && c1 + j < p.M)
                              ? __half2float(rbuf[(c1 + j) * kTileF + row])
                              : 0.0f;
                v0[j] = __uint_as_float(r0[j]);
                v1[j] = two ? __uint_as_float(r1[j]) : 0.0f;
            }
            // the later parts, in k order (the first one's loads go out with
            // the residual's)
            for (int u = 0; u < nparts; ++u) {
                const float* src =
                    p.partial +
                    static_cast<size_t>((q + 1 + u) * c + static_cast<int>(crank)) * p.nt * kTileF + row;
                float pv0[8], pv1[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    pv0[j] = __ldcg(src + (c0 + j) * kTileF);
                    pv1[j] = two ? __ldcg(src + (c1 + j) * kTileF) : 0.0f;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    v0[j] = __fadd_rn(v0[j], pv0[j]);
                    v1[j] = __fadd_rn(v1[j], pv1[j]);
                }
            }
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                if (h2 == 1 && !two) break;
                const int cb = h2 ? c1 : c0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int m = cb + j;
                    if (m >= p.M) break;
                    float x = __fadd_rn(h2 ? v1[j] : v0[j], bias);
                    if (p.act == FG_ACT_RELU) x = fmaxf(x, 0.0f);
                    if (p.residual) x = __fadd_rn(x, h2 ? res1[j] : res0[j]);
                    p.Y[static_cast<int64_t>(m) * p.N + n] = __float2half_rn(x);
                }
            }
        }
    };
    int last_nparts = 0;   // epilogue warps: parts consumed by the last segment

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- codes + (min, scale) TMA producer: one box per unit
            int issued_last[kSC];
            for (int s = 0; s < kSC; ++s) issued_last[s] = -1;
            SegIter it = proto;
            int bc = 0;
            bool stop = false;
            while (!stop && it.next()) {
                const int row0 = (it.t * c + static_cast<int>(crank)) * kTileF;
                for (int b = it.b0; b < it.b1; ++b, ++bc) {
                    const int s = bc % kSC;
                    if (!mbar_wait(sm.c_empty(s), ((bc / kSC) & 1) ^ 1u, abort_flag, lim)) {
                        fail();
                        stop = true;
                        break;
                    }
                    if (p.drop_arrive && bc == 0) continue;   // test knob: never arm box 0
                    mbar_arrive_expect_tx(sm.c_full(s), kCBytes + kMBytes);
                    tma_load_2d(sm.c(s), &tmC, b * (kBoxK / 2), row0, sm.c_full(s));
                    tma_load_2d(sm.m(s), &tmM, b * (kBoxK / 64) * 2, row0, sm.c_full(s));
                    issued_last[s] = bc;
                }
            }
            for (int j = 0; j < kSC; ++j)   // no copy may land after this CTA leaves
                if (issued_last[j] >= 0)
                    mbar_wait(sm.c_full(j), (issued_last[j] / kSC) & 1, nullptr, lim);
        }
    } else if (warp == 2) {
        if (lane == 0) {
            // ---------------- activation TMA producer: this CTA's 1/c slice of
            // the rows of each stage (both 64-k halves), multicast to the cluster
            griddep_wait();
            const int srows = p.nt / c;
            const uint32_t soff = crank * static_cast<uint32_t>(srows) * 128u;
            int issued_last[kNS];
            for (int s = 0; s < kNS; ++s) issued_last[s] = -1;
            SegIter it = proto;
            int i = 0;
            bool stop = false;
            while (!stop && it.next()) {
                for (int b = it.b0; b < it.b1 && !stop; ++b) {
                    for (int h = 0; h < 2; ++h, ++i) {
                        const int s = i % kNS;
                        if (!mbar_wait(sm.empty(s), ((i / kNS) & 1) ^ 1u, abort_flag, lim)) {
                            fail();
                            stop = true;
                            break;
                        }
                        mbar_arrive_expect_tx(sm.full(s), 2u * sm.half_bytes);
                        const int k0 = b * kBoxK + h * kStageK;
                        const int r0 = static_cast<int>(crank) * srows;
                        tma_load_2d_mc(sm.b(s) + soff, &tmX, k0, r0, sm.full(s), cmask);
                        tma_load_2d_mc(sm.b(s) + sm.half_bytes + soff, &tmX, k0 + 64, r0,
                                       sm.full(s), cmask);
                        issued_last[s] = i;
                    }
                }
            }
            // no copy may land after this CTA leaves: wait for each stage's last
            // phase (its completion needs every slice, ours included)
            for (int j = 0; j < kNS; ++j)
                if (issued_last[j] >= 0)
                    mbar_wait(sm.full(j), (issued_last[j] / kNS) & 1, nullptr, lim);
        }
    } else if (warp == 3) {
        if (lane == 0 && p.residual != nullptr) {
            // ---------------- residual TMA producer: the residual rows of each
            // segment that ends in the Y epilogue (a whole tile or a tile's
            // first part), one [nt][128] tile at a time, loaded as soon as
            // the previous one has been read
            griddep_wait();
            SegIter it = proto;
            int ny = 0, issued = -1;
            bool last_y = false;
            while (it.next()) {
                last_y = false;
                if (it.b0 != 0) continue;
                if (!mbar_wait(sm.res_empty(), (ny & 1) ^ 1u, abort_flag, lim)) {
                    fail();
                    break;
                }
                mbar_arrive_expect_tx(sm.res_full(), static_cast<uint32_t>(p.nt) * kTileF * 2u);
                tma_load_2d(sm.r0, &tmR, (it.t * c + static_cast<int>(crank)) * kTileF, 0, sm.res_full());
                issued = ny++;
                last_y = it.u >= it.hi;
            }
            // no copy may land after this CTA leaves; the dequant warps that
            // share the last Y epilogue wait for its rows here
            if (issued >= 0 && mbar_wait(sm.res_full(), issued & 1, nullptr, lim) && last_y)
                mbar_arrive(sm.res_last());
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer.  The whole warp runs the loop (its
        // control flow and descriptors are warp-uniform); lane 0 issues each
        // stage's 8 MMAs (A from TMEM, B from shared memory) and the commit
        // that frees the stage cluster-wide, and per segment the commit that
        // hands the accumulator to the epilogue.  (A commit tracks the MMAs of
        // the thread that issues it, so lane 0 issues them all.)
        const uint32_t idesc = idesc_f16_f32(kTileF, p.nt);
        const uint64_t bdesc0 = sw128_desc(sm.b(0));
        const uint32_t bstep = (2u * sm.half_bytes) >> 4;   // descriptor units per stage
        const uint32_t bhalf = sm.half_bytes >> 4;
        SegIter it = proto;
        int i = 0, sg = 0;
        int s = 0;
        uint32_t ph = 0;
        bool stop = false;
        while (!stop && it.next()) {
            const int a = sg & 1;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(sm.acc_empty(a), ((sg >> 1) & 1) ^ 1u, abort_flag, lim))) {
                if (lane == 0) fail();
                break;
            }
            tc_fence_after();
            const uint32_t acc = tmem + static_cast<uint32_t>(a * kAccStride);
            const int nst = 2 * (it.b1 - it.b0);
            for (int j = 0; j < nst; ++j, ++i) {
                if (!__all_sync(0xffffffffu, mbar_wait(sm.full(s), ph, abort_flag, lim))) {
                    if (lane == 0) fail();
                    stop = true;
                    break;
                }
                tc_fence_after();
                const uint32_t ta = tmem + static_cast<uint32_t>(kABase + s * kACols);
                const uint64_t bd0 = bdesc0 + static_cast<uint64_t>(s) * bstep;
                const uint64_t bd1 = bd0 + bhalf;
                if (lane == 0) {
                    mma_f16_ta(acc, ta, bd0, idesc, j != 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 1; kk < kStageK / 16; ++kk)
                        mma_f16_ta(acc, ta + 8 * kk, (kk < 4 ? bd0 : bd1) + 2 * (kk & 3), idesc, 1u);
                    mma_commit_mc(sm.empty(s), cmask);
                }
                __syncwarp();
                if (++s == kNS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (stop) break;
            if (lane == 0) mma_commit(sm.acc_full(a));
            __syncwarp();
            ++sg;
        }
        // also on abort: every MMA issued completes before TMEM is freed
        if (lane == 0) {
            mma_commit(sm.drain());
            mbar_wait(sm.drain(), 0, nullptr, lim);
        }
        __syncwarp();
    } else if (warp >= 8) {
        // ---------------- dequantisers: group g takes stages g, g + kG, ...;
        // thread = weight row 32q + lane of its lane quarter q.  A stage is
        // half of a codes box: 64 code bytes and two (min, scale) per row ->
        // 128 fp16 = 64 TMEM columns, written by two 32-column stores.
        const int g = (warp - 8) >> 2, qq = warp & 3;
        const int row = qq * 32 + lane;
        const uint32_t tl = static_cast<uint32_t>(qq * 32) << 16;
        const uint32_t rx = static_cast<uint32_t>(row & 7);
        bool failed = false;
        for (int i = g; i < nstages; i += kG) {
            const int bc = i >> 1, h = i & 1;
            const int cs = bc % kSC;
            if (!__all_sync(0xffffffffu, mbar_wait(sm.c_full(cs), (bc / kSC) & 1, abort_flag, lim))) {
                fail();
                failed = true;
                break;
            }
            // 16-byte units 4h..4h+3 of the 128-byte codes row, stored at
            // unit ^ (row % 8); (min, scale) of chunks 2h and 2h + 1
            const uint8_t* crow = gen + sm.c(cs) + row * 128;
            uint4 w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                w[j] = *reinterpret_cast<const uint4*>(crow + (((4u * h + j) ^ rx) << 4));
            const float4 mm = *reinterpret_cast<const float4*>(gen + sm.m(cs) + row * 32 + h * 16);
            // The box is released only after the proxy fence: TMA (the async
            // proxy) writes the next box into the slot, and an mbarrier
            // release alone does not order these generic reads before it.
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.c_empty(cs));
            const int s = i % kNS;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(sm.empty(s), ((i / kNS) & 1) ^ 1u, abort_flag, lim))) {
                fail();
                failed = true;
                break;
            }
            tc_fence_after();   // the MMAs that read this A stage have completed
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float mn = hh ? mm.z : mm.x, scl = hh ? mm.w : mm.y;
                const float S = scl * 16777216.0f, S16 = scl * 1048576.0f;
                const uint32_t wd[8] = {w[2 * hh].x,     w[2 * hh].y,     w[2 * hh].z,
                                        w[2 * hh].w,     w[2 * hh + 1].x, w[2 * hh + 1].y,
                                        w[2 * hh + 1].z, w[2 * hh + 1].w};
                uint32_t r[32];
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 v = dequant8_x2(wd[cc], S, S16, mn);
                    r[4 * cc] = v.x;
                    r[4 * cc + 1] = v.y;
                    r[4 * cc + 2] = v.z;
                    r[4 * cc + 3] = v.w;
                }
                __syncwarp();
                tmem_st32(tmem + tl + static_cast<uint32_t>(kABase + s * kACols + 32 * hh), r);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.full(s));
        }
        // The CTA's last segment, when it ends in the Y epilogue (this CTA
        // holds the tile's first part), is on the kernel's critical tail: the
        // dequantisers, idle by then, share it with the epilogue warp of
        // their lane quarter (8-column chunks 1 + g, 5 + g, ...).
        if (!failed) {
            griddep_wait();
            SegIter it = proto;
            int nseg = 0, lt = 0, lb0 = 0, lb1 = 0;
            while (it.next()) {
                ++nseg;
                lt = it.t;
                lb0 = it.b0;
                lb1 = it.b1;
            }
            if (nseg > 0 && lb0 == 0) {
                const int a = (nseg - 1) & 1;
                if (__all_sync(0xffffffffu, mbar_wait(sm.acc_full(a), ((nseg - 1) >> 1) & 1, abort_flag, lim))) {
                    tc_fence_after();
                    bool ok = true;
                    const int nparts = wait_parts(lt, lb1, qq, ok);
                    if (ok && p.residual != nullptr)
                        ok = __all_sync(0xffffffffu, mbar_wait(sm.res_last(), 0, abort_flag, lim));
                    if (ok)
                        y_epilogue(tmem + tl + static_cast<uint32_t>(a * kAccStride),
                                   (lt * c + static_cast<int>(crank)) * kTileF + row, row, nparts,
                                   1 + g, 4);
                    else
                        fail();
                } else {
                    fail();
                }
            }
        }
    } else if (warp >= 4) {
        // ---------------- epilogue, warps 4-7 = TMEM lane quarters 0-3
        griddep_wait();
        const int qq = warp & 3;
        const int row = qq * 32 + lane;
        const uint32_t tl = static_cast<uint32_t>(qq * 32) << 16;
        const int slot = q * c + static_cast<int>(crank);
        SegIter it = proto;
        int sg = 0, ny = 0;
        while (it.next()) {
            const bool last = it.u >= it.hi;
            const int a = sg & 1;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(sm.acc_full(a), (sg >> 1) & 1, abort_flag, lim))) {
                fail();
                break;
            }
            tc_fence_after();
            const uint32_t acc = tmem + tl + static_cast<uint32_t>(a * kAccStride);
            const int n = (it.t * c + static_cast<int>(crank)) * kTileF + row;
            bool ok = true;
            if (it.b0 > 0) {
                // A later part of a split tile: stored once for the cluster
                // holding the tile's first box, then published (one flag per
                // lane quarter, so no warp waits for another).
                float* dst = p.partial + static_cast<size_t>(slot) * p.nt * kTileF + row;
                for (int c0 = 0; c0 < p.nt; c0 += 16) {
                    uint32_t r[16];
                    __syncwarp();
                    tmem_ld16(acc + static_cast<uint32_t>(c0), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) dst[(c0 + j) * kTileF] = __uint_as_float(r[j]);
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_u64(p.flags + slot * 4 + qq, epoch);
            } else {
                // The tile's first part (or the whole tile); in the last
                // segment shared with the dequantisers (chunks 0, 4, 8, ...).
                const int nparts = wait_parts(it.t, it.b1, qq, ok);
                if (ok && p.residual != nullptr)
                    ok = __all_sync(0xffffffffu, mbar_wait(sm.res_full(), ny & 1, abort_flag, lim));
                if (ok) {
                    y_epilogue(acc, n, row, nparts, 0, last ? 4 : 1);
                    if (p.residual != nullptr) {
                        // the next tile's TMA (async proxy) overwrites what
                        // these generic reads saw
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(sm.res_empty());
                    }
                    ++ny;
                    if (last) last_nparts = nparts;
                } else {
                    fail();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.acc_empty(a));
            if (!ok) break;
            ++sg;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
    // The flags consumed by the last segment (read by all four warps of a
    // lane quarter, now past the barrier) go back to 0, so that a replay of
    // this launch (same epoch, e.g. from a CUDA graph) waits for them again.
    if (warp >= 4 && warp < 8 && lane == 0)
        for (int pi = 0; pi < last_nparts; ++pi)
            p.flags[((q + 1 + pi) * c + static_cast<int>(crank)) * 4 + (warp & 3)] = 0ull;
    // No CTA leaves while a peer may still multicast into it or arrive on its
    // barriers.
    cluster_sync_all();
    if (*abort_flag && threadIdx.x == 0) {
        // after an expired wait, give any stray multicast copy time to land
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {
        }
    }
}

}  // namespace

namespace fg {

namespace {

// Clusters of c CTAs that can be resident at once (one CTA per SM), for the
// largest tile this kernel takes, so that the plan -- and with it every
// output's summation order -- is the same for every M.  Every cluster of a
// launch is then resident together, which the in-kernel fixup relies on (its
// flag waits are bounded all the same).
int dec_max_clusters(int c) {
    static std::mutex mu;
    static int cache[64][3];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev][c] == 0) {
        const size_t smem = dec_smem_bytes(kMaxNt, true);
        if (cudaFuncSetAttribute(gemm_dec_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(c * num_sms()), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_dec_kernel, &cfg) != cudaSuccess || n <= 0)
            return 0;
        cache[dev][c] = n;
    }
    return cache[dev][c];
}

// Launch tags for the fixup flags: unique per launch, with a fixed upper half
// so that uninitialised workspace memory is never mistaken for a flag.
std::atomic<unsigned long long> g_epoch{0};

}  // namespace

bool plan_gemm_dec(int64_t M, int64_t N, int64_t K, int64_t plan_rows, GemmPlan& pl) {
    if (plan_rows > kMaxNt || M > kMaxNt || M <= 0 || K % kBoxK != 0 || N <= 0) return false;
    const int F = static_cast<int>(cdiv(N, kTileF));
    const int c = F % 2 == 0 ? 2 : 1;
    const int qmax = dec_max_clusters(c);
    if (qmax <= 0) return false;
    pl = GemmPlan{};
    pl.dec = 1;
    pl.nt = static_cast<int>(cdiv(M, 16) * 16);
    pl.tok_tiles = 1;
    pl.feat_tiles = F;
    pl.splits = 1;
    pl.dec_c = c;
    pl.dec_nbox = static_cast<int>(K / kBoxK);
    pl.dec_units = static_cast<long long>(F / c) * pl.dec_nbox;
    // at least kDecMinUnits units per cluster: a small projection (few units)
    // runs on fewer clusters, so its tiles are split fewer ways and the
    // tile-finishing epilogues add fewer parts (measured on the small
    // workloads; the large projections have tens of units per cluster)
    long long nq = pl.dec_units / kDecMinUnits;
    if (nq < 1) nq = 1;
    if (nq > qmax) nq = qmax;
    pl.dec_Q = static_cast<int>(nq);
    const size_t slots = static_cast<size_t>(pl.dec_Q) * c;
    pl.dec_part_bytes = (slots * pl.nt * kTileF * sizeof(float) + 255) & ~static_cast<size_t>(255);
    pl.ws_bytes = pl.dec_part_bytes + slots * 4 * sizeof(unsigned long long);
    pl.ws_min = pl.ws_bytes;
    return true;
}

fg_status launch_gemm_dec(const __half* X, int64_t M, const fg_q4* W, const __half* bias,
                          const __half* residual, int act, __half* Y, void* ws, size_t ws_bytes,
                          cudaStream_t st, const GemmPlan& pl) {
    const int64_t N = W->rows, K = W->cols;
    if (ws == nullptr || ws_bytes < pl.ws_bytes || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return set_error(FG_ERR_WORKSPACE, "dequant_gemm: workspace %zu < %zu bytes or misaligned",
                         ws_bytes, pl.ws_bytes);
    const int c = pl.dec_c;
    CUtensorMap tmX, tmC, tmM, tmR;
    // activations: this CTA's nt / c rows of a 64-k half stage (rows >= M read as 0)
    fg_status s = make_tmap(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K, M, 64, pl.nt / c,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != FG_OK) return s;
    // codes: one box = 128 rows x 128 bytes (256 k), 128-byte swizzle
    s = make_tmap(&tmC, W->codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, N, kBoxK / 2, kTileF,
                  CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != FG_OK) return s;
    // (min, scale): 128 rows x 4 groups x 2 fp32 per box
    s = make_tmap(&tmM, W->meta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (K / 64) * 2, N,
                  (kBoxK / 64) * 2, kTileF, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (s != FG_OK) return s;
    // residual: the [nt][128] tile of a Y segment (rows >= M, columns >= N read as 0)
    if (residual != nullptr) {
        s = make_tmap(&tmR, residual, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, N, M, kTileF, pl.nt,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
        if (s != FG_OK) return s;
    } else {
        tmR = tmX;   // never read
    }
    DecParams p{};
    p.bias = bias;
    p.residual = residual;
    p.Y = Y;
    p.partial = static_cast<float*>(ws);
    p.flags = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + pl.dec_part_bytes);
    p.epoch = 0xF1A6000000000000ull | (++g_epoch & 0x0000FFFFFFFFFFFFull);
    p.units = pl.dec_units;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.nt = pl.nt;
    p.c = c;
    p.nbox = pl.dec_nbox;
    p.Q = pl.dec_Q;
    p.act = act;
    p.status = device_status_ptr();
    p.wait_ns = wait_limit_ns();
    p.drop_arrive = take_drop_arrive();
    // one CTA per SM whatever nt; the attribute allows the largest launch (a
    // graph may hold both kinds), each launch asks for what it uses
    const size_t smem = dec_smem_bytes(kMaxNt, residual != nullptr);
    cudaError_t e = cudaFuncSetAttribute(gemm_dec_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(dec_smem_bytes(kMaxNt, true)));
    if (e != cudaSuccess) return cuda_error(e, "gemm_dec smem attribute");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.dec_Q * c), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    fg::add_pdl_attr(cfg, attr, 1);
    const double Md = M, Nd = N, Kd = K;
    // algorithmic traffic: the weight once (codes + (min, scale)), X once, Y once
    // (+ residual); the partial sums of split tiles stay in L2
    TraceScope ts(FG_TRACE_GEMM_DECODE, st, 2.0 * Md * Nd * Kd,
                  Nd * Kd * 0.625 + Md * Kd * 2.0 + Md * Nd * 2.0 * (residual ? 2.0 : 1.0));
    e = cudaLaunchKernelEx(&cfg, gemm_dec_kernel, tmX, tmC, tmM, tmR, p);
    if (e != cudaSuccess) return cuda_error(e, "gemm_dec launch");
    return cuda_error(cudaGetLastError(), "gemm_dec launch");
}

}  // namespace fg
