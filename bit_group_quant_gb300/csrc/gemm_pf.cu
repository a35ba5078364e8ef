// gemm_pf.cu -- the prefill projection GEMM over fp16 weights, on CTA pairs.
//
// Y[m][n] = act(sum_k X[m][k] * W[n][k] + bias[n]) + residual[m][n] with W the
// projection's weights already dequantised once into fp16 (w^ = fp16(fma(q,
// scale, min)), "FlexGen 完全拆解", compression section: stored tensors are
// dequantised to FP16 before compute).  It serves a prefill-sized block
// (thousands of rows: bls sequences x s prompt tokens), where the projections
// are dense contractions that dominate the step's time.
//
// Mapping.  A tile is 256 weight rows x 256 activation rows.  A 2-CTA cluster
// (one SM pair) computes it with tcgen05 MMAs of M = 256, N = 256, K = 16
// (cta_group::2): each CTA holds its 128 weight rows (A) and 128 of the 256
// activation rows (B) of every 64-k stage, the even CTA issues the MMAs, and
// each CTA's TMEM receives its 128 weight rows x 256 activation columns.  Per
// SM and stage that is 16 KB of A and 16 KB of B written by TMA and read by
// the tensor core once -- half the shared-memory traffic per FLOP of a
// one-SM 128 x 256 tile, whose operand traffic alone saturates shared memory.
//
// Persistent: one pair per two SMs, tiles dealt round robin; two 256-column
// accumulators in TMEM, so a tile's epilogue (TMEM -> registers, bias, ReLU,
// residual, fp16 stores) overlaps the next tile's MMAs.  Tiles are ordered in
// blocks of 8 weight-row tiles x all activation tiles, and every tile walks K
// from 0, so the tiles running at one time share their weight and activation
// panels as they stream through L2.  Every row's result depends on K and the
// tile walk only, never on M or the row's position.
//
// Warp roles (384 threads): warp 0 = TMA producer (both CTAs; each loads its
// own A and B halves, completion counted on the even CTA's barrier); warp 1 =
// TMEM allocator (both) and MMA issuer (even CTA); warps 4-11 = epilogue, two
// per TMEM lane quarter (each half of the 256 columns).
//
// Every wait is bounded; a wait that expires flags the CTA to stop, records a
// timeout in the device status word, drains what it issued, frees TMEM and
// returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "fg_internal.cuh"

namespace {

using namespace fgd;

constexpr int kThreads = 384;                 // 12 warps
constexpr int kHalf = 128;                    // weight rows / activation rows per CTA per tile
constexpr int kTile = 256;                    // weight rows and activation rows per pair tile
constexpr int kChunk = 64;                    // k per stage (one 128-byte swizzle row of fp16)
constexpr uint32_t kOpBytes = kHalf * kChunk * 2;      // 16 KB: one CTA's A or B of a stage
constexpr uint32_t kStageBytes = 2 * kOpBytes;         // A then B
constexpr int kNS = 6;                        // stages
constexpr int kAccCols = 256;                 // TMEM columns per accumulator
constexpr int kFeatBlock = 8;                 // weight-row tiles per raster block
constexpr int kEpiWarp0 = 4;                  // first epilogue warp
constexpr int kEpiWarps = 8;
constexpr int kNumBars = 2 * kNS + 5;
constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kNS) * kStageBytes + 8 * kNumBars + 16;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(2 * kAccCols <= 512, "TMEM columns");

struct PfParams {
    const __half* bias;       // [N] or null
    const __half* residual;   // [M][N] or null
    __half* Y;                // [M][N]
    int M, N, K;
    int kchunks;              // K / 64
    int act;
    int ft, tt;               // weight-row tiles (of 256), activation tiles (of 256)
    int tiles;                // ft * tt
    int Q;                    // clusters (pairs)
    int* status;
    unsigned long long wait_ns;
    int drop_arrive;
};

// Tile id -> (weight-row tile, activation tile): blocks of kFeatBlock
// weight-row tiles; inside a block the weight-row tile varies fastest.
__device__ __forceinline__ void tile_coords(int id, int ft, int tt, int& f, int& t) {
    const int per = kFeatBlock * tt;
    const int blk = id / per;
    const int r = id - blk * per;
    const int f0 = blk * kFeatBlock;
    const int fw = min(kFeatBlock, ft - f0);
    t = r / fw;
    f = f0 + r % fw;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_pf_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const PfParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + kNS * kStageBytes;
    // barriers: full[kNS] (even CTA: the stage's four TMA loads of the pair),
    // empty[kNS] (the MMAs that read the stage are done), acc_full[2],
    // acc_empty[2] (even CTA: the 16 epilogue warps of the pair), drain
    auto full = [&](int s) { return bars + 8u * static_cast<uint32_t>(s); };
    auto empty = [&](int s) { return bars + 8u * static_cast<uint32_t>(kNS + s); };
    auto acc_full = [&](int a) { return bars + 8u * static_cast<uint32_t>(2 * kNS + a); };
    auto acc_empty = [&](int a) { return bars + 8u * static_cast<uint32_t>(2 * kNS + 2 + a); };
    const uint32_t drain = bars + 8u * (2 * kNS + 4);
    auto a_smem = [&](int s) { return base + static_cast<uint32_t>(s) * kStageBytes; };
    auto b_smem = [&](int s) { return a_smem(s) + kOpBytes; };
    uint8_t* const gen = smem_raw - raw;   // generic pointer = gen + shared address
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gen + bars + 8u * kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const bool leader = crank == 0;
    const int q = static_cast<int>(blockIdx.x) >> 1;    // pair index
    const int ntiles = q < p.tiles ? (p.tiles - 1 - q) / p.Q + 1 : 0;
    const uint64_t lim = p.wait_ns;
    // Both operands come from earlier kernels (the weights from the
    // dequantisation launched just before): the producer and the epilogue
    // wait for them; the set-up below overlaps the previous kernel's tail.
    griddep_launch();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(full(s), 1);      // the even CTA's arrive (+ both CTAs' bytes)
            mbar_init(empty(s), 1);     // one commit of the even CTA's MMA thread
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), 2 * kEpiWarps);
        }
        mbar_init(drain, 1);
        // A wait that expired earlier (status not yet cleared by fg_check)
        // makes every later pair skip its work instead of waiting again.
        *abort_flag = (p.status != nullptr && *reinterpret_cast<volatile int*>(p.status) != 0);
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    __syncthreads();
    // Every barrier of both CTAs exists before any remote arrive or load.
    cluster_sync_all();
    {
        // the skip decision of the even CTA holds for the pair
        const uint32_t f0 = ld_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), 0));
        if (f0 != 0) {
            cluster_sync_all();   // nobody reads the even CTA's flag after it leaves
            return;               // uniform across the pair: nothing issued yet
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), 2 * kAccCols);
        tmem_relinquish_pair();
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
            // ---------------- TMA producer: this CTA's A (weight rows) and B
            // (activation rows) of every stage, counted on the even CTA's full
            // barrier, which expects the bytes of both CTAs
            griddep_wait();
            int issued_last[kNS];
            for (int s = 0; s < kNS; ++s) issued_last[s] = -1;
            int s = 0, i = 0;
            uint32_t ph = 0;
            bool stop = false;
            for (int j = 0; j < ntiles && !stop; ++j) {
                int f, t;
                tile_coords(q + j * p.Q, p.ft, p.tt, f, t);
                const int arow = f * kTile + static_cast<int>(crank) * kHalf;
                const int brow = t * kTile + static_cast<int>(crank) * kHalf;
                for (int kc = 0; kc < p.kchunks; ++kc, ++i) {
                    if (!mbar_wait(empty(s), ph ^ 1u, abort_flag, lim)) {
                        fail();
                        stop = true;
                        break;
                    }
                    // test knob: the even CTA never arms its first stage
                    const bool drop = p.drop_arrive && i == 0 && leader;
                    if (!drop) {
                        if (leader) mbar_arrive_expect_tx(full(s), 2 * kStageBytes);
                        const uint32_t fb = mapa_shared(full(s), 0);
                        tma_load_2d_pair(a_smem(s), &tmA, kc * kChunk, arow, fb);
                        tma_load_2d_pair(b_smem(s), &tmB, kc * kChunk, brow, fb);
                        issued_last[s] = i;
                    }
                    if (++s == kNS) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // no copy may land after the pair leaves: the even CTA waits for the
            // last phase of every stage it armed (which counts both CTAs' bytes)
            if (leader)
                for (int j = 0; j < kNS; ++j)
                    if (issued_last[j] >= 0)
                        mbar_wait(full(j), (issued_last[j] / kNS) & 1, nullptr, lim);
        }
    } else if (warp == 1) {
        if (leader) {
            // ---------------- MMA issuer (even CTA).  The whole warp runs the
            // loop; lane 0 issues the 4 MMAs of a stage and the commit that
            // frees the stage in both CTAs, and per tile the commit that hands
            // the accumulator to both CTAs' epilogues.
            const uint32_t idesc = idesc_f16_f32(kTile, kTile);
            const uint64_t ad0 = sw128_desc(a_smem(0)), bd0 = sw128_desc(b_smem(0));
            const uint32_t step = kStageBytes >> 4;
            int s = 0;
            uint32_t ph = 0;
            bool stop = false;
            for (int j = 0; j < ntiles && !stop; ++j) {
                const int a = j & 1;
                if (!__all_sync(0xffffffffu,
                                mbar_wait_cluster(acc_empty(a), ((j >> 1) & 1) ^ 1u, abort_flag, lim))) {
                    if (lane == 0) fail();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(a * kAccCols);
                for (int kc = 0; kc < p.kchunks; ++kc) {
                    if (!__all_sync(0xffffffffu, mbar_wait(full(s), ph, abort_flag, lim))) {
                        if (lane == 0) fail();
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint64_t off = static_cast<uint64_t>(s) * step;
#pragma unroll
                        for (int kk = 0; kk < kChunk / 16; ++kk)
                            mma_f16_pair(d, ad0 + off + 2 * kk, bd0 + off + 2 * kk, idesc,
                                         (kc | kk) != 0 ? 1u : 0u);
                        mma_commit_pair_mc(empty(s), 3);
                    }
                    __syncwarp();
                    if (++s == kNS) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (stop) break;
                if (lane == 0) mma_commit_pair_mc(acc_full(a), 3);
                __syncwarp();
            }
            // also on abort: every MMA issued completes before TMEM is freed
            if (lane == 0) {
                mma_commit_pair_mc(drain, 1);
                mbar_wait(drain, 0, nullptr, lim);
            }
            __syncwarp();
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
        // ---------------- epilogue: warp w reads TMEM lane quarter w % 4 (its
        // 32 weight rows) and half ch of the 256 activation columns
        const int qq = warp & 3;
        const int ch = (warp - kEpiWarp0) >> 2;
        const int row = qq * 32 + lane;
        const uint32_t tl = static_cast<uint32_t>(qq * 32) << 16;
        const uint32_t empty_remote0 = mapa_shared(acc_empty(0), 0);
        griddep_wait();
        for (int j = 0; j < ntiles; ++j) {
            const int a = j & 1;
            int f, t;
            tile_coords(q + j * p.Q, p.ft, p.tt, f, t);
            if (!__all_sync(0xffffffffu, mbar_wait(acc_full(a), (j >> 1) & 1, abort_flag, lim))) {
                fail();
                break;
            }
            tc_fence_after();
            const int n = f * kTile + static_cast<int>(crank) * kHalf + row;
            const bool nv = n < p.N;
            const float bias = (nv && p.bias != nullptr) ? __half2float(p.bias[n]) : 0.0f;
            const int tok0 = t * kTile;
            for (int c0 = ch * kHalf; c0 < (ch + 1) * kHalf; c0 += 16) {
                uint32_t r[16];
                __syncwarp();   // the stores of the previous round diverge
                tmem_ld16(tmem + tl + static_cast<uint32_t>(a * kAccCols + c0), r);
                tmem_wait_ld();
                const int m0 = tok0 + c0;
                if (!nv || m0 >= p.M) continue;
                // residual loads all issued before the first store (the residual
                // never aliases Y), so their latencies overlap
                float res[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    res[jj] = (p.residual != nullptr && m0 + jj < p.M)
                                  ? __half2float(__ldg(p.residual + static_cast<int64_t>(m0 + jj) * p.N + n))
                                  : 0.0f;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int m = m0 + jj;
                    if (m >= p.M) break;
                    float v = __fadd_rn(__uint_as_float(r[jj]), bias);
                    if (p.act == FG_ACT_RELU) v = fmaxf(v, 0.0f);
                    if (p.residual) v = __fadd_rn(v, res[jj]);
                    p.Y[static_cast<int64_t>(m) * p.N + n] = __float2half_rn(v);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(empty_remote0 + 8u * static_cast<uint32_t>(a));
        }
    }
    tc_fence_before();
    __syncthreads();
    // both CTAs are past their last TMEM access and the even CTA's MMAs have
    // drained before the pair frees its TMEM
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 2 * kAccCols);
    cluster_sync_all();
    if (*abort_flag && threadIdx.x == 0) {
        // after an expired wait, give any stray copy time to land
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {
        }
    }
}

// Pairs that can be resident at once, per device (the grid is persistent).
int max_pairs() {
    static std::mutex mu;
    static int cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] == 0) {
        if (cudaFuncSetAttribute(gemm_pf_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes)) != cudaSuccess)
            return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * 76, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_pf_kernel, &cfg) != cudaSuccess || n <= 0)
            return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace

namespace fg {

fg_status launch_gemm_pf(const __half* X, int64_t M, const __half* W16, int64_t N, int64_t K,
                         const __half* bias, const __half* residual, int act, __half* Y,
                         cudaStream_t st) {
    if (M == 0) return FG_OK;
    CUtensorMap tmA, tmB;
    fg_status s = make_tmap(&tmA, W16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K, N, kChunk, kHalf,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != FG_OK) return s;
    s = make_tmap(&tmB, X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K, M, kChunk, kHalf,
                  CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != FG_OK) return s;
    const int pairs = max_pairs();
    if (pairs <= 0) return set_error(FG_ERR_CUDA, "gemm_pf: no resident CTA pair");
    PfParams p{};
    p.bias = bias;
    p.residual = residual;
    p.Y = Y;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.kchunks = static_cast<int>(K / kChunk);
    p.act = act;
    p.ft = static_cast<int>(cdiv(N, kTile));
    p.tt = static_cast<int>(cdiv(M, kTile));
    p.tiles = p.ft * p.tt;
    p.Q = p.tiles < pairs ? p.tiles : pairs;
    p.status = device_status_ptr();
    p.wait_ns = wait_limit_ns();
    p.drop_arrive = take_drop_arrive();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * p.Q), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    fg::add_pdl_attr(cfg, attr, 1);
    const double Md = M, Nd = N, Kd = K;
    // algorithmic traffic: the fp16 weights once, X once, Y once (+ residual)
    TraceScope ts(FG_TRACE_GEMM_PREFILL, st, 2.0 * Md * Nd * Kd,
                  Nd * Kd * 2.0 + Md * Kd * 2.0 + Md * Nd * 2.0 * (residual ? 2.0 : 1.0));
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_pf_kernel, tmA, tmB, p);
    if (e != cudaSuccess) return cuda_error(e, "gemm_pf launch");
    return cuda_error(cudaGetLastError(), "gemm_pf launch");
}

}  // namespace fg
