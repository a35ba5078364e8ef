// gemm.cu -- dequant-fused GEMM on the 5th-generation tensor cores.
//
// Y[m][n] = act(sum_k X[m][k] * W^[n][k] + bias[n]) + residual[m][n], where W
// is stored 4-bit in groups of 64 along k and dequantised to fp16 on chip
// ("FlexGen 完全拆解", compression section: stored tensors are dequantised to
// FP16 before compute).  This serves every projection of the decoder.
//
// Mapping (operands swapped so that a block of bls sequences is one MMA):
//   MMA A operand = 128 dequantised weight rows (output features) x 64 k,
//   MMA B operand = nt activation rows (tokens) x 64 k,  nt <= 256,
//   accumulator   = 128 x nt fp32 in TMEM (lane = feature, column = token).
// At decode, nt = bls: each weight tile is fetched from HBM and dequantised
// exactly once per block, which is the block schedule's weight reuse.
//
// Clusters of c = 1, 2 or 4 CTAs (consecutive feature tiles, one token tile)
// share each activation tile: every CTA loads 1/c of it and multicasts the
// slice to the whole cluster, so the activations cross L2 once per cluster
// instead of once per CTA.
//
// Warp roles (416 threads, 13 warps): warp 0 = TMA producer of the weight
// side (packed codes, 4 K-chunks per 128-byte-swizzled box, or fp16 A tiles);
// warp 2 = TMA producer of this CTA's activation slices; warp 1 = TMEM
// allocator and the single MMA-issuing thread, alone on its sub-partition
// during the mainloop (warps 5 and 9 idle until the epilogue); warps 3, 4, 6,
// 7, 8, 10, 11, 12 = dequantisers in four groups of two, group g owning K
// chunks g, g+4, ... (two weight rows per thread: 32 code bytes + (min,
// scale) -> 64 fp16 each, written in the 128-byte-swizzled K-major layout the
// MMA descriptor reads).  Warps 3-10 then run the epilogue (tcgen05.ld of the
// accumulator, bias / ReLU / residual, fp16 store -- or fp32 partial sums when
// K is split).  Tiles are visited in groups of 16 feature tiles x all token
// tiles, and each group of 4 feature tiles starts its K walk at its own
// offset, so L2 sees neither re-reads nor hot spots.
//
// Every mbarrier wait is bounded; a wait that expires flags the CTA to stop,
// records a timeout in the device status word, waits for its own copies and
// MMAs in flight, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "fg_internal.cuh"

namespace {

using namespace fgd;

constexpr int kThreads = 416;        // 13 warps
constexpr int kDeqWarps = 8;         // warps 3,4,6,7,8,10,11,12 (none on sub-partition 1)
constexpr int kDeqGroups = 4;        // groups of 2 warps; group g owns chunks i = g (mod 4)
constexpr int kRasterGroup = 16;     // feature tiles per rasterisation group
constexpr int kRotBlock = 4;         // feature tiles sharing one K-walk offset
constexpr int kTileF = 128;          // output features per CTA (MMA M)
// Planned rows from which the weights are dequantised once into fp16 for the
// whole launch instead of once per 256-row token tile (the prefill).
constexpr int64_t kF16WeightRows = 8192;
constexpr int kChunk = 64;           // k per A/B stage: one 128-byte swizzle row of fp16
constexpr int kCodeSpan = 4;         // K chunks per codes box (128 code bytes per row)
constexpr uint32_t kABytes = kTileF * kChunk * 2;                // 16 KB
constexpr uint32_t kCBytes = kTileF * kChunk / 2 * kCodeSpan;    // 16 KB of packed codes
constexpr int kCStages = 3;          // codes ring, at most (12 K chunks ahead)
constexpr int kMaxStages = 8;        // A+B stage ring
constexpr int kMaxBars = 2 * (kCStages + kMaxStages) + 1;
constexpr int kSmemLimit = 227 * 1024;
static_assert(kDeqGroups == kCodeSpan, "one chunk of every codes box per dequant group");
// A parity wait on an mbarrier can only tell the current phase from the one
// before it, so no thread may start waiting for a phase two ahead of the
// barrier.  A dequant group jumps kDeqGroups chunks at a time; its previous
// chunk guarantees the stage it waits for is at most one phase behind only if
// the stage ring has at least kDeqGroups stages.  (With fewer, a group can
// pass a wait early, overwrite a stage still being read and over-arrive on its
// barrier.)  The host never launches the dequant kernel with fewer stages.
constexpr int kMinStagesDq = kDeqGroups;

struct GemmParams {
    const float2* meta;       // [N][K/64] (min, scale); dequant mode
    const __half* bias;       // [N] or null
    const __half* residual;   // [M][N] or null
    __half* Y;                // [M][N] fp16
    float* Yf;                // [M][N] fp32 (fp16-weight mode)
    float* partial;           // [splits][M][N] fp32 when splits > 1
    int M, N, K;
    int nt;                   // activation rows per tile (MMA N)
    int feat_tiles, tok_tiles;
    int cluster;              // CTAs per cluster sharing the activation tile
    int kchunks;              // K / 64
    int kc_per_split;         // multiple of kCodeSpan
    int act;
    int ns, sc;               // ring depths (A+B stages, codes boxes)
    int* status;
    unsigned long long wait_ns;
    int drop_arrive;
};

// Dequantiser index 0..7 of a warp (-1 for other warps).  Sub-partition 1
// (warps 1, 5, 9) is left to the single MMA-issuing thread during the
// mainloop: every instruction on its path is latency-critical.
__device__ __forceinline__ int deq_index(int w) {
    switch (w) {
        case 3: return 0;
        case 4: return 1;
        case 6: return 2;
        case 7: return 3;
        case 8: return 4;
        case 10: return 5;
        case 11: return 6;
        case 12: return 7;
        default: return -1;
    }
}

// Shared-memory carve-up, all offsets from a 1024-aligned base:
//   stage ring [ns][A 16 KB | B nt*128 B]   (both 128B-swizzled K-major MMA
//                                            operands; one full and one empty
//                                            barrier per stage)
//   codes ring [sc][16 KB]                  (packed codes of 4 K chunks)
//   barriers, TMEM address slot, abort flag
struct Smem {
    uint32_t base, st0, c0, bars;
    int ns, sc;
    uint32_t b_bytes, st_bytes;
    // stage s = [A: 16 KB][B: nt*128 B]
    __device__ uint32_t a(int s) const { return st0 + static_cast<uint32_t>(s) * st_bytes; }
    __device__ uint32_t b(int s) const { return a(s) + kABytes; }
    __device__ uint32_t c(int s) const { return c0 + static_cast<uint32_t>(s) * kCBytes; }
    __device__ uint32_t full(int s) const { return bars + 8u * s; }
    __device__ uint32_t empty(int s) const { return bars + 8u * (ns + s); }
    __device__ uint32_t c_full(int s) const { return bars + 8u * (2 * ns + s); }
    __device__ uint32_t c_empty(int s) const { return bars + 8u * (2 * ns + sc + s); }
    __device__ uint32_t acc() const { return bars + 8u * (2 * ns + 2 * sc); }
    __device__ uint32_t end() const { return acc() + 8u; }
};

template <bool kDequant, bool kF32Out>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Smem sm;
    sm.base = (raw + 1023u) & ~1023u;
    sm.ns = p.ns;
    sm.sc = kDequant ? p.sc : 0;
    sm.b_bytes = static_cast<uint32_t>(p.nt) * 128u;
    sm.st_bytes = kABytes + sm.b_bytes;
    sm.st0 = sm.base;
    sm.c0 = sm.st0 + sm.ns * sm.st_bytes;
    sm.bars = sm.c0 + sm.sc * kCBytes;
    uint8_t* const gen = smem_raw - raw;   // generic pointer = gen + shared address
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gen + sm.end());
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ccount = p.cluster;
    const uint32_t crank = cluster_ctarank();
    const uint16_t cmask = static_cast<uint16_t>((1u << ccount) - 1u);
    // grouped rasterisation: within a group of kRasterGroup feature tiles the
    // feature tile varies fastest, then the token tile (a cluster is c
    // consecutive feature tiles of one token tile)
    int feat_tile, tok_tile;
    {
        const int id = blockIdx.x;
        const int per_group = kRasterGroup * p.tok_tiles;
        const int grp = id / per_group;
        const int f0 = grp * kRasterGroup;
        const int gf = min(kRasterGroup, p.feat_tiles - f0);
        const int r = id - grp * per_group;
        feat_tile = f0 + r % gf;
        tok_tile = r / gf;
    }
    const int feat0 = feat_tile * kTileF;
    const int tok0 = tok_tile * p.nt;
    const int kc0 = blockIdx.z * p.kc_per_split;
    const int kc1 = min(p.kchunks, kc0 + p.kc_per_split);
    const int nk = kc1 - kc0;
    // Each block of kRotBlock feature tiles walks its K chunks from its own
    // offset (whole codes boxes), so the CTAs sharing an activation tile do
    // not all fetch the same chunk at once.  The offset depends on the
    // feature tile only: the summation order of every output -- hence its
    // value -- does not depend on M, the cluster size or the other rows.
    const int nbox = nk / kCodeSpan;
    const int rot = (nk % kCodeSpan == 0 && nbox > 0)
                        ? kCodeSpan * static_cast<int>((static_cast<long long>(feat_tile / kRotBlock) * 37) % nbox)
                        : 0;
    auto chunk_at = [&](int i) { return kc0 + (i + rot) % nk; };
    const uint32_t ncols = p.nt <= 32 ? 32u : (p.nt <= 64 ? 64u : (p.nt <= 128 ? 128u : 256u));
    const uint64_t lim = p.wait_ns;
    // The weight side (4-bit codes and (min, scale), or the fp16 token
    // embedding of the LM head) never changes during a step: it is fetched
    // and dequantised at once, possibly while the previous kernel of the
    // stream still runs; the activation producer and the epilogue first wait
    // for that kernel.
    griddep_launch();

    if (threadIdx.x == 0) {
        for (int s = 0; s < sm.ns; ++s) {
            // full: the activation producer's arrive (+ B bytes), and either
            // the 2 dequant warps owning the chunk or the fp16 A producer (+ A bytes)
            mbar_init(sm.full(s), 1 + (kDequant ? kDeqWarps / kDeqGroups : 1));
            // empty: one MMA commit from every CTA of the cluster (frees the
            // local A and the multicast B of the stage)
            mbar_init(sm.empty(s), ccount);
        }
        for (int s = 0; s < sm.sc; ++s) {
            mbar_init(sm.c_full(s), 1);
            mbar_init(sm.c_empty(s), kDeqWarps);   // every dequant warp reads one chunk per box
        }
        mbar_init(sm.acc(), 1);
        // A wait that expired earlier (status not yet cleared by fg_check)
        // makes every later cluster skip its work instead of waiting again.
        *abort_flag = (p.status != nullptr && *reinterpret_cast<volatile int*>(p.status) != 0);
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
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
        tmem_alloc(smem_u32(tmem_slot), ncols);
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

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- weight-side TMA producer
            if (kDequant) {
                // one box = 128 rows x 128 code bytes = 4 K chunks
                const int nboxes = (nk + kCodeSpan - 1) / kCodeSpan;
                int issued_last[kCStages];
                for (int s = 0; s < kCStages; ++s) issued_last[s] = -1;
                const int SC = sm.sc;
                int s = 0;
                uint32_t ph = 0;
                for (int t = 0; t < nboxes; ++t, s = (s + 1 == SC) ? 0 : s + 1,
                         ph ^= (s == 0) ? 1u : 0u) {
                    if (!mbar_wait(sm.c_empty(s), ph ^ 1u, abort_flag, lim)) {
                        fail();
                        break;
                    }
                    if (p.drop_arrive && t == 0) continue;  // test knob: never arm box 0
                    mbar_arrive_expect_tx(sm.c_full(s), kCBytes);
                    tma_load_2d(sm.c(s), &tmW, chunk_at(kCodeSpan * t) * (kChunk / 2), feat0,
                                sm.c_full(s));
                    issued_last[s] = t;
                }
                for (int j = 0; j < SC; ++j)   // no copy may land after this CTA leaves
                    if (issued_last[j] >= 0)
                        mbar_wait(sm.c_full(j), (issued_last[j] / SC) & 1, nullptr, lim);
            } else {
                int issued_last[kMaxStages];
                for (int s = 0; s < kMaxStages; ++s) issued_last[s] = -1;
                const int NS = sm.ns;
                int s = 0;
                uint32_t ph = 0;
                for (int i = 0; i < nk; ++i, s = (s + 1 == NS) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
                    if (!mbar_wait(sm.empty(s), ph ^ 1u, abort_flag, lim)) {
                        fail();
                        break;
                    }
                    mbar_arrive_expect_tx(sm.full(s), kABytes);
                    tma_load_2d(sm.a(s), &tmW, chunk_at(i) * kChunk, feat0, sm.full(s));
                    issued_last[s] = i;
                }
                for (int j = 0; j < NS; ++j)
                    if (issued_last[j] >= 0)
                        mbar_wait(sm.full(j), (issued_last[j] / NS) & 1, nullptr, lim);
            }
        }
    } else if (warp == 2) {
        if (lane == 0) {
            // ---------------- activation TMA producer: this CTA's 1/c slice of
            // each B tile, multicast to every CTA of the cluster
            griddep_wait();
            const int srows = p.nt / ccount;
            const uint32_t soff = crank * static_cast<uint32_t>(srows) * 128u;
            int issued_last[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) issued_last[s] = -1;
            const int NS = sm.ns;
            int s = 0;
            uint32_t ph = 0;
            for (int i = 0; i < nk; ++i, s = (s + 1 == NS) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
                if (!mbar_wait(sm.empty(s), ph ^ 1u, abort_flag, lim)) {
                    fail();
                    break;
                }
                mbar_arrive_expect_tx(sm.full(s), sm.b_bytes);
                tma_load_2d_mc(sm.b(s) + soff, &tmX, chunk_at(i) * kChunk,
                               tok0 + static_cast<int>(crank) * srows, sm.full(s), cmask);
                issued_last[s] = i;
            }
            // no copy may land after this CTA leaves: wait for this stage's
            // last phase (its completion needs every slice, ours included)
            for (int j = 0; j < NS; ++j)
                if (issued_last[j] >= 0)
                    mbar_wait(sm.full(j), (issued_last[j] / NS) & 1, nullptr, lim);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            // The issue loop is kept minimal: it shares its sub-partition with
            // busy warps, so every instruction on this path costs many cycles.
            // Ring positions advance incrementally; descriptors are built once
            // and advanced by adding encoded byte offsets (address >> 4) to the
            // start-address field (no carry: shared addresses < 2^18).
            const uint32_t idesc = idesc_f16_f32(kTileF, p.nt);
            const int NS = sm.ns;
            const uint64_t ad0 = sw128_desc(sm.a(0)), bd0 = sw128_desc(sm.b(0));
            const uint32_t step = sm.st_bytes >> 4;
            uint32_t fb = sm.full(0), eb = sm.empty(0), off = 0, ph = 0;
            int s = 0;
            for (int i = 0; i < nk; ++i) {
                if (!mbar_wait(fb, ph, abort_flag, lim)) {
                    fail();
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk)
                    mma_f16(tmem, ad0 + off + 2 * kk, bd0 + off + 2 * kk, idesc,
                            (i | kk) != 0 ? 1u : 0u);
                mma_commit_mc(eb, cmask);   // frees the stage (A here, B cluster-wide)
                if (++s == NS) {
                    s = 0;
                    ph ^= 1u;
                    off = 0;
                    fb = sm.full(0);
                    eb = sm.empty(0);
                } else {
                    off += step;
                    fb += 8u;
                    eb += 8u;
                }
            }
            mma_commit(sm.acc());  // also on abort: lets the epilogue drain the MMAs in flight
        }
    } else {
        const int dqi = deq_index(warp);
        if (kDequant && dqi >= 0) {
            // ---------------- dequantisers: group dg (2 warps) owns chunks
            // i = dg, dg + 4, ... (chunk dg of every codes box); thread r0 of
            // the group owns weight rows r0 and r0 + 64.  Four chunks are in
            // flight at once, one per group.
            const int dg = dqi >> 1, r0 = (dqi & 1) * 32 + lane;
            const int n0 = feat0 + r0, n1 = n0 + 64;
            const bool v0 = n0 < p.N, v1 = n1 < p.N;
            const float2* mrow0 = p.meta + static_cast<int64_t>(n0) * p.kchunks;
            const float2* mrow1 = p.meta + static_cast<int64_t>(n1) * p.kchunks;
            const int nmine = nk > dg ? (nk - dg + kDeqGroups - 1) / kDeqGroups : 0;
            constexpr int kRing = 8;
            float2 ring0[kRing], ring1[kRing];
#pragma unroll
            for (int j = 0; j < kRing; ++j) {
                const int kc = j < nmine ? chunk_at(dg + j * kDeqGroups) : 0;
                ring0[j] = (v0 && j < nmine) ? __ldg(mrow0 + kc) : make_float2(0.f, 0.f);
                ring1[j] = (v1 && j < nmine) ? __ldg(mrow1 + kc) : make_float2(0.f, 0.f);
            }
            // this chunk's 32 code bytes of a row are 16-byte units 2*dg and
            // 2*dg+1 of the 128-byte row, stored at unit ^ (row % 8)
            const uint32_t u0 = ((2u * dg) ^ (r0 & 7)) << 4, u1 = ((2u * dg + 1) ^ (r0 & 7)) << 4;
            const int NS = sm.ns;
            int sc = 0, sa = dg % NS;       // chunk i = dg + 4*it: codes box it, stage i % NS
            uint32_t pc = 0, pa = (dg / NS) & 1;
            bool stop = false;
            for (int i0 = 0; i0 < nmine && !stop; i0 += kRing) {
#pragma unroll
                for (int j = 0; j < kRing; ++j) {
                    const int it = i0 + j;
                    if (it >= nmine || stop) break;
                    const float2 mm0 = ring0[j], mm1 = ring1[j];
                    if (it + kRing < nmine) {
                        const int kc = chunk_at(dg + (it + kRing) * kDeqGroups);
                        if (v0) ring0[j] = __ldg(mrow0 + kc);
                        if (v1) ring1[j] = __ldg(mrow1 + kc);
                    }
                    // every lane waits; the outcome is made warp-uniform so no
                    // lane can leave the loop while others sit in __syncwarp
                    if (!__all_sync(0xffffffffu, mbar_wait(sm.c_full(sc), pc, abort_flag, lim))) {
                        fail();
                        stop = true;
                        break;
                    }
                    const uint8_t* c0p = gen + sm.c(sc) + r0 * 128;
                    const uint8_t* c1p = c0p + 64 * 128;
                    const uint4 wa0 = *reinterpret_cast<const uint4*>(c0p + u0);
                    const uint4 wb0 = *reinterpret_cast<const uint4*>(c0p + u1);
                    const uint4 wa1 = *reinterpret_cast<const uint4*>(c1p + u0);
                    const uint4 wb1 = *reinterpret_cast<const uint4*>(c1p + u1);
                    // The codes box is released only after the proxy fence
                    // below: the next box is written into the slot by TMA (the
                    // async proxy), and an mbarrier release alone does not
                    // order these generic reads before that write -- with an
                    // arrive right here, runs with thousands of boxes per CTA
                    // dequantised codes the TMA had already replaced.
                    if (!__all_sync(0xffffffffu, mbar_wait(sm.empty(sa), pa ^ 1u, abort_flag, lim))) {
                        fail();
                        stop = true;
                        break;
                    }
                    const float S0 = mm0.y * 16777216.0f, S160 = mm0.y * 1048576.0f;
                    const float S1 = mm1.y * 16777216.0f, S161 = mm1.y * 1048576.0f;
                    const uint32_t w0[8] = {wa0.x, wa0.y, wa0.z, wa0.w, wb0.x, wb0.y, wb0.z, wb0.w};
                    const uint32_t w1[8] = {wa1.x, wa1.y, wa1.z, wa1.w, wb1.x, wb1.y, wb1.z, wb1.w};
                    uint8_t* a0p = gen + sm.a(sa) + r0 * 128;
                    uint8_t* a1p = a0p + 64 * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t off = (c ^ (r0 & 7)) << 4;
                        *reinterpret_cast<uint4*>(a0p + off) = dequant8(w0[c], S0, S160, mm0.x);
                        *reinterpret_cast<uint4*>(a1p + off) = dequant8(w1[c], S1, S161, mm1.x);
                    }
                    // one fence orders this warp's generic smem accesses before
                    // the async proxy: the A stores before the MMA reads them,
                    // and the codes reads before TMA overwrites the box
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(sm.full(sa));
                        mbar_arrive(sm.c_empty(sc));
                    }
                    // next chunk of this group: codes box +1, stage +4 (mod NS)
                    if (++sc == sm.sc) { sc = 0; pc ^= 1u; }
                    sa += kDeqGroups;
                    while (sa >= NS) { sa -= NS; pa ^= 1u; }
                }
            }
        }
        if (warp > 10) goto done;   // warps 11 and 12 only dequantise
        {
        // ---------------- epilogue, warps 3..10 (the accumulator barrier is
        // also the drain of every MMA issued, so it does not stop early on the
        // abort flag)
        // Lanes may leave the backed-off wait at different times: __all_sync
        // makes the outcome uniform and reconverges the warp before the
        // .sync.aligned TMEM loads below.
        griddep_wait();
        const bool ok = __all_sync(0xffffffffu, mbar_wait_sleepy(sm.acc(), 0, lim));
        if (!ok && lane == 0) report(p.status, fg::kDevTimeout);
        tc_fence_after();
        const int q = warp & 3;                    // TMEM lane quarter this warp may read
        const int colq = warp < 7 ? 0 : 1;  // two warps per quarter split the columns
        const int row = q * 32 + lane;
        const int n = feat0 + row;
        const bool live = ok && !*abort_flag;
        float bias = 0.0f;
        if (!kF32Out && live && p.bias != nullptr && n < p.N && gridDim.z == 1)
            bias = __half2float(p.bias[n]);
        for (int c0 = 16 * colq; c0 < p.nt; c0 += 32) {
            uint32_t r[16];
            __syncwarp();   // the stores of the previous round diverge
            tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, r);
            tmem_wait_ld();
            if (!live || n >= p.N) continue;
            // residual loads are all issued before the first store (the
            // residual never aliases Y), so their latencies overlap
            float res[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = tok0 + c0 + j;
                res[j] = (!kF32Out && gridDim.z == 1 && p.residual != nullptr && m < p.M)
                             ? __half2float(__ldg(p.residual + static_cast<int64_t>(m) * p.N + n))
                             : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = tok0 + c0 + j;
                if (m >= p.M) break;
                const float acc = __uint_as_float(r[j]);
                const int64_t idx = static_cast<int64_t>(m) * p.N + n;
                if (kF32Out) {
                    p.Yf[idx] = acc;
                } else if (gridDim.z > 1) {
                    p.partial[static_cast<int64_t>(blockIdx.z) * p.M * p.N + idx] = acc;
                } else {
                    float v = __fadd_rn(acc, bias);
                    if (p.act == FG_ACT_RELU) v = fmaxf(v, 0.0f);
                    if (p.residual) v = __fadd_rn(v, res[j]);
                    p.Y[idx] = __float2half_rn(v);
                }
            }
        }
        }
    }
done:
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, ncols);
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

// Fixed-order sum of the K-split partials, then the epilogue.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ partial,
                                                            int splits, int64_t M, int64_t N,
                                                            const __half* __restrict__ bias,
                                                            const __half* __restrict__ residual,
                                                            int act, __half* __restrict__ Y) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    griddep_wait();
    griddep_launch();
    const int64_t nv = M * N / 4;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nv;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t e = i * 4;
        float4 acc = reinterpret_cast<const float4*>(partial)[i];
        for (int z = 1; z < splits; ++z) {
            const float4 v = reinterpret_cast<const float4*>(partial + z * M * N)[i];
            acc.x = __fadd_rn(acc.x, v.x);
            acc.y = __fadd_rn(acc.y, v.y);
            acc.z = __fadd_rn(acc.z, v.z);
            acc.w = __fadd_rn(acc.w, v.w);
        }
        float a[4] = {acc.x, acc.y, acc.z, acc.w};
        const int64_t n0 = e % N;
        __half o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float v = a[j];
            if (bias) v = __fadd_rn(v, __half2float(bias[n0 + j]));
            if (act == FG_ACT_RELU) v = fmaxf(v, 0.0f);
            if (residual) v = __fadd_rn(v, __half2float(residual[e + j]));
            o[j] = __float2half_rn(v);
        }
        *reinterpret_cast<uint2*>(Y + e) = *reinterpret_cast<const uint2*>(o);
    }
}

// ---------------------------------------------------------------- host side

struct Rings {
    int ns, sc;
    size_t smem;
};

Rings rings_for(int nt, bool dq) {
    // every barrier must fit the space reserved for kMaxBars
    static_assert(2 * (kCStages + kMaxStages) + 1 <= kMaxBars, "barrier space");
    Rings r{};
    const size_t per = kABytes + static_cast<size_t>(nt) * 128;
    // dequant mode: as many codes boxes as leave kMinStagesDq stages (the
    // parity rule), preferring 3 boxes in flight
    for (int sc = dq ? kCStages : 0; sc >= 0; --sc) {
        const size_t fixed = 1024 + static_cast<size_t>(sc) * kCBytes + 8 * kMaxBars + 16;
        int ns = static_cast<int>((kSmemLimit - fixed) / per);
        if (ns > kMaxStages) ns = kMaxStages;
        r.sc = sc;
        r.ns = ns;
        r.smem = fixed + static_cast<size_t>(ns) * per;
        if (!dq || ns >= kMinStagesDq) break;
    }
    return r;
}

// CTAs per cluster sharing one activation tile: the largest of 4, 2, 1 that
// divides the feature tiles and leaves slices of whole 8-row swizzle atoms.
int cluster_for(int feat_tiles, int nt) {
    for (int c = 4; c > 1; c >>= 1)
        if (feat_tiles % c == 0 && nt % c == 0 && (nt / c) % 8 == 0) return c;
    return 1;
}

template <bool kDequant, bool kF32Out>
fg_status run_gemm(const void* X, const CUtensorMap& tmW, GemmParams& p, const fg::GemmPlan& plan,
                   cudaStream_t st) {
    const Rings rg = rings_for(plan.nt, kDequant);
    if (rg.ns < (kDequant ? kMinStagesDq : 2) || (kDequant && rg.sc < 1))
        return fg::set_error(FG_ERR_UNSUPPORTED, "gemm: tile of %d rows does not fit", plan.nt);
    p.ns = rg.ns;
    p.sc = rg.sc;
    p.cluster = cluster_for(plan.feat_tiles, plan.nt);
    p.feat_tiles = plan.feat_tiles;
    p.tok_tiles = plan.tok_tiles;
    CUtensorMap tmX;
    fg_status s = fg::make_tmap(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.K, p.M, kChunk,
                            plan.nt / p.cluster, CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != FG_OK) return s;
    auto kern = gemm_tc_kernel<kDequant, kF32Out>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(rg.smem));
    if (e != cudaSuccess) return fg::cuda_error(e, "gemm smem attribute");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.feat_tiles * plan.tok_tiles, 1, plan.splits);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = rg.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    fg::add_pdl_attr(cfg, attr, 1);
    const double M = p.M, N = p.N, K = p.K;
    // algorithmic traffic: the weight once (4-bit codes + fp32 (min, scale) per
    // 64, or fp16), X once, Y once (+ residual, or fp32 partials / logits)
    const double wbytes = kDequant ? N * K * 0.625 : N * K * 2.0;
    const double ybytes = kF32Out ? M * N * 4.0
                                  : (plan.splits > 1 ? plan.splits * M * N * 4.0
                                                     : M * N * 2.0 * (p.residual ? 2.0 : 1.0));
    // the LM head (fp32 logits) is traced with the small kernels; the
    // projections by their size, whichever form the weights take
    const int cls = kF32Out ? FG_TRACE_OTHER
                            : (p.M > 256 ? FG_TRACE_GEMM_PREFILL : FG_TRACE_GEMM_DECODE);
    fg::TraceScope ts(cls, st, 2.0 * M * N * K, wbytes + M * K * 2.0 + ybytes);
    e = cudaLaunchKernelEx(&cfg, kern, tmX, tmW, p);
    if (e != cudaSuccess) return fg::cuda_error(e, "gemm launch");
    return fg::cuda_error(cudaGetLastError(), "gemm launch");
}

}  // namespace

namespace fg {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

fg_status make_tmap(CUtensorMap* tm, const void* ptr, CUtensorMapDataType dt, int esize,
                    uint64_t cols, uint64_t rows, uint32_t bx, uint32_t by,
                    CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return fg::set_error(FG_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * static_cast<uint64_t>(esize)};
    cuuint32_t box[2] = {bx, by};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fg::set_error(FG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return FG_OK;
}


// Tile plan.  It depends on M only through the number of 256-row activation
// tiles, and the K split only on (N, K) -- and is used only when all rows fit
// one tile -- so every row's result is independent of M and of the other rows
// (the row-by-row and zig-zag block orders must agree bit for bit).
GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int64_t plan_rows, bool dequant) {
    GemmPlan pl{};
    if (plan_rows < M) plan_rows = M;
    if (dequant && plan_gemm_dec(M, N, K, plan_rows, pl)) return pl;
    pl.tok_tiles = static_cast<int>(cdiv(M, 256));
    if (pl.tok_tiles < 1) pl.tok_tiles = 1;
    int64_t rows = cdiv(M, pl.tok_tiles);
    pl.nt = static_cast<int>(cdiv(rows, 16) * 16);
    if (pl.nt < 16) pl.nt = 16;
    pl.feat_tiles = static_cast<int>(cdiv(N, kTileF));
    pl.splits = 1;
    const int64_t kchunks = K / kChunk;
    if (plan_rows <= 256) {   // one token tile: split K to fill the SMs
        const int sms = num_sms();
        int s = sms / pl.feat_tiles;
        if (s > 8) s = 8;
        if (s > kchunks / 8) s = static_cast<int>(kchunks / 8);
        if (s < 1) s = 1;
        pl.splits = s;
    }
    pl.kc_per_split = static_cast<int>(kchunks);
    if (pl.splits > 1) {
        // equal ranges of whole codes boxes (4 K chunks); drop empty splits
        const int64_t per = cdiv(cdiv(kchunks, pl.splits), kCodeSpan) * kCodeSpan;
        pl.splits = static_cast<int>(cdiv(kchunks, per));
        pl.kc_per_split = static_cast<int>(per);
    }
    pl.ws_bytes = pl.splits > 1 ? static_cast<size_t>(pl.splits) * M * N * sizeof(float) : 0;
    pl.ws_min = pl.ws_bytes;
    if (dequant && plan_rows >= kF16WeightRows) {   // splits == 1 here
        pl.f16w = 1;
        pl.ws_bytes = static_cast<size_t>(N) * K * sizeof(__half);
    }
    return pl;
}

fg_status launch_gemm_g4(const __half* X, int64_t M, const fg_q4* W, const __half* bias,
                         const __half* residual, int act, __half* Y, void* ws, size_t ws_bytes,
                         cudaStream_t st, int64_t plan_rows) {
    if (M == 0) return FG_OK;
    const int64_t N = W->rows, K = W->cols;
    const GemmPlan pl = plan_gemm(M, N, K, plan_rows);
    if (pl.ws_min > 0 && (ws == nullptr || ws_bytes < pl.ws_min))
        return set_error(FG_ERR_WORKSPACE, "dequant_gemm: workspace %zu < %zu bytes", ws_bytes,
                         pl.ws_min);
    if (pl.dec) return launch_gemm_dec(X, M, W, bias, residual, act, Y, ws, ws_bytes, st, pl);
    // prefill-sized blocks with room for the fp16 weights take the fp16
    // pipeline; otherwise the fused dequantisation below
    if (pl.f16w && ws != nullptr && ws_bytes >= pl.ws_bytes) {
        // dequantise the weights once (exactly: fp16(fma(code, scale, min)),
        // the values the fused path computes per tile), then the fp16 GEMM on
        // CTA pairs (gemm_pf.cu)
        __half* w16 = static_cast<__half*>(ws);
        fg_status s = launch_dequant_g4(W->codes, W->meta, N * K / kGroup, w16, st,
                                        FG_TRACE_GEMM_PREFILL);
        if (s != FG_OK) return s;
        return launch_gemm_pf(X, M, w16, N, K, bias, residual, act, Y, st);
    }
    // codes: one box = 128 rows x 128 bytes (4 K chunks), 128-byte swizzle
    CUtensorMap tmC;
    fg_status s = make_tmap(&tmC, W->codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, N,
                            kCodeSpan * kChunk / 2, kTileF, CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != FG_OK) return s;
    GemmParams p{};
    p.meta = reinterpret_cast<const float2*>(W->meta);
    p.bias = bias;
    p.residual = residual;
    p.Y = Y;
    p.partial = static_cast<float*>(ws);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.nt = pl.nt;
    p.kchunks = static_cast<int>(K / kChunk);
    p.kc_per_split = pl.kc_per_split;
    p.act = act;
    p.status = device_status_ptr();
    p.wait_ns = wait_limit_ns();
    p.drop_arrive = take_drop_arrive();
    s = run_gemm<true, false>(X, tmC, p, pl, st);
    if (s != FG_OK || pl.splits == 1) return s;
    const int64_t nv = M * N / 4;
    int64_t blocks = cdiv(nv, 256);
    if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, pl.splits * M * N * 4.0 + M * N * 4.0);
    {
        const cudaError_t le_ = fg::launch_pdl(splitk_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
            p.partial, pl.splits, M, N, bias, residual, act, Y);
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "splitk_reduce_kernel launch");
    }
    return cuda_error(cudaGetLastError(), "splitk reduce launch");
}

fg_status launch_gemm_f16_f32out(const __half* X, int64_t M, const __half* W, int64_t N,
                                 int64_t K, float* Y, cudaStream_t st) {
    if (M == 0) return FG_OK;
    GemmPlan pl = plan_gemm(M, N, K, M, false);
    pl.splits = 1;
    CUtensorMap tmW;
    fg_status s = make_tmap(&tmW, W, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K, N, kChunk, kTileF,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != FG_OK) return s;
    GemmParams p{};
    p.Yf = Y;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.nt = pl.nt;
    p.kchunks = static_cast<int>(K / kChunk);
    p.kc_per_split = p.kchunks;
    p.status = device_status_ptr();
    p.wait_ns = wait_limit_ns();
    return run_gemm<false, true>(X, tmW, p, pl, st);
}

}  // namespace fg
