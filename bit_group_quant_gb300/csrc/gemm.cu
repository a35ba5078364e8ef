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
// Warp roles (320 threads): warp 0 = TMA producer (activations and packed
// codes into a ring of shared-memory stages); warp 1 = TMEM allocator and
// the single MMA-issuing thread; warps 2-9 = dequantisers (two threads per
// weight row, each 16 code bytes from shared memory + (min, scale) -> 32
// fp16 written in the 128-byte-swizzled K-major layout the MMA descriptor
// reads), then the epilogue (tcgen05.ld of the accumulator, bias / ReLU /
// residual, fp16 store) -- or fp32 partial sums when K is split.
// CTAs walk the output tiles in groups of 16 feature tiles x all token
// tiles, so weight and activation tiles are reused from L2.
//
// Every mbarrier wait is bounded; a wait that expires flags the CTA to stop,
// records a timeout in the device status word, waits for its own copies and
// MMAs in flight, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "fg_internal.cuh"

namespace {

using namespace fgd;

constexpr int kThreads = 320;
constexpr int kDeqThreads = 256;
constexpr int kRasterGroup = 16;     // feature tiles per rasterisation group
constexpr int kTileF = 128;          // output features per CTA (MMA M)
constexpr int kChunk = 64;           // k per stage: one 128-byte swizzle row of fp16
constexpr uint32_t kABytes = kTileF * kChunk * 2;   // 16 KB
constexpr uint32_t kCBytes = kTileF * kChunk / 2;   // 4 KB of packed codes
constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 227 * 1024;

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
    int kchunks;              // K / 64
    int kc_per_split;
    int act;
    int stages;
    int* status;
    unsigned long long wait_ns;
    int drop_arrive;
};

__device__ __forceinline__ uint32_t stage_bytes(int nt, bool dq) {
    return kABytes + static_cast<uint32_t>(nt) * 128u + (dq ? kCBytes : 0u);
}

// 8 codes (one 32-bit word, element 0 in the lowest nibble) -> 8 fp16
// m + c*s as four half2 words in element order.  (1024 + c) is exact in fp16
// when the code is OR-ed into the mantissa of 1024; subtracting 1024 leaves c
// exactly, and one fused half2 multiply-add applies scale and min.
__device__ __forceinline__ uint4 dequant8(uint32_t w, __half2 s2, __half2 m2) {
    const uint32_t kMagic = 0x64006400u;  // half2(1024, 1024)
    const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    uint32_t t[4];
    t[0] = (w & 0x000F000Fu) | kMagic;          // (c0, c4)
    t[1] = ((w >> 4) & 0x000F000Fu) | kMagic;   // (c1, c5)
    t[2] = ((w >> 8) & 0x000F000Fu) | kMagic;   // (c2, c6)
    t[3] = ((w >> 12) & 0x000F000Fu) | kMagic;  // (c3, c7)
    uint32_t y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 c = __hsub2(*reinterpret_cast<__half2*>(&t[i]), k1024);
        __half2 v = __hfma2(c, s2, m2);
        y[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    uint4 r;
    r.x = __byte_perm(y[0], y[1], 0x5410);  // (c0, c1)
    r.y = __byte_perm(y[2], y[3], 0x5410);  // (c2, c3)
    r.z = __byte_perm(y[0], y[1], 0x7632);  // (c4, c5)
    r.w = __byte_perm(y[2], y[3], 0x7632);  // (c6, c7)
    return r;
}

template <bool kDequant, bool kF32Out>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    const int S = p.stages;
    const uint32_t b_bytes = static_cast<uint32_t>(p.nt) * 128u;
    const uint32_t sbytes = stage_bytes(p.nt, kDequant);
    const uint32_t bars = base + static_cast<uint32_t>(S) * sbytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto deq_bar = [&](int s) { return bars + 8u * (S + s); };
    auto empty_bar = [&](int s) { return bars + 8u * (2 * S + s); };
    const uint32_t acc_bar = bars + 8u * (3 * S);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + S * sbytes + 8 * (3 * S + 1));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto a_smem = [&](int s) { return base + static_cast<uint32_t>(s) * sbytes; };
    auto b_smem = [&](int s) { return a_smem(s) + kABytes; };
    auto c_smem = [&](int s) { return b_smem(s) + b_bytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grouped rasterisation: within a group of kRasterGroup feature tiles the
    // feature tile varies fastest, then the token tile
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
    const uint32_t ncols = p.nt <= 32 ? 32u : (p.nt <= 64 ? 64u : (p.nt <= 128 ? 128u : 256u));
    const uint64_t lim = p.wait_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(deq_bar(s), kDeqThreads);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(acc_bar, 1);
        // A wait that expired earlier (status not yet cleared by fg_check)
        // makes every later CTA skip its work instead of waiting again.
        *abort_flag = (p.status != nullptr && *reinterpret_cast<volatile int*>(p.status) != 0);
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    __syncthreads();
    if (*abort_flag) return;  // uniform across the CTA: nothing allocated yet
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int issued_last[kMaxStages];
            for (int s = 0; s < S; ++s) issued_last[s] = -1;
            for (int i = 0; i < nk; ++i) {
                const int s = i % S;
                const uint32_t ph = (i / S) & 1;
                if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, lim)) {
                    *abort_flag = 1;
                    report(p.status, fg::kDevTimeout);
                    break;
                }
                if (p.drop_arrive && i == 0) continue;  // test knob: never arm stage 0
                const uint32_t bytes = b_bytes + (kDequant ? kCBytes : kABytes);
                mbar_arrive_expect_tx(full_bar(s), bytes);
                const int kc = kc0 + i;
                tma_load_2d(b_smem(s), &tmX, kc * kChunk, tok0, full_bar(s));
                if (kDequant)
                    tma_load_2d(c_smem(s), &tmW, kc * (kChunk / 2), feat0, full_bar(s));
                else
                    tma_load_2d(a_smem(s), &tmW, kc * kChunk, feat0, full_bar(s));
                issued_last[s] = i;
            }
            // Never leave with copies in flight into this CTA's shared memory.
            for (int s = 0; s < S; ++s)
                if (issued_last[s] >= 0)
                    mbar_wait(full_bar(s), (issued_last[s] / S) & 1, nullptr, lim);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc = idesc_f16_f32(kTileF, p.nt);
            for (int i = 0; i < nk; ++i) {
                const int s = i % S;
                const uint32_t ph = (i / S) & 1;
                bool ok = mbar_wait(full_bar(s), ph, abort_flag, lim);
                if (ok && kDequant) ok = mbar_wait(deq_bar(s), ph, abort_flag, lim);
                if (!ok) {
                    *abort_flag = 1;
                    report(p.status, fg::kDevTimeout);
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk) {
                    const uint64_t ad = sw128_desc(a_smem(s) + kk * 32);
                    const uint64_t bd = sw128_desc(b_smem(s) + kk * 32);
                    mma_f16(tmem, ad, bd, idesc, (i | kk) != 0 ? 1u : 0u);
                }
                mma_commit(empty_bar(s));
            }
            mma_commit(acc_bar);  // also on abort: lets the epilogue drain the MMAs in flight
        }
    } else {
        const int dt = threadIdx.x - 64;  // 0..255
        if (kDequant) {
            // ---------------- dequantisers: thread dt owns half hf of weight row rw
            const int rw = dt >> 1, hf = dt & 1;
            const int n = feat0 + rw;
            const bool nvalid = n < p.N;
            const float2* mrow = p.meta + static_cast<int64_t>(n) * p.kchunks + kc0;
            float2 ring[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                ring[j] = (nvalid && j < nk) ? __ldg(mrow + j) : make_float2(0.f, 0.f);
            bool stop = false;
            for (int i0 = 0; i0 < nk && !stop; i0 += 4) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = i0 + j;
                    if (i >= nk || stop) break;
                    const float2 mm = ring[j];
                    if (nvalid && i + 4 < nk) ring[j] = __ldg(mrow + i + 4);
                    const int s = i % S;
                    const uint32_t ph = (i / S) & 1;
                    if (!mbar_wait(full_bar(s), ph, abort_flag, lim)) {
                        *abort_flag = 1;
                        report(p.status, fg::kDevTimeout);
                        stop = true;
                        break;
                    }
                    const __half2 s2 = __float2half2_rn(mm.y);
                    const __half2 m2 = __float2half2_rn(mm.x);
                    const uint4 w = *reinterpret_cast<const uint4*>(
                        base_ptr + (c_smem(s) - base) + rw * 32 + hf * 16);
                    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
                    uint8_t* arow = base_ptr + (a_smem(s) - base) + rw * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int chunk = hf * 4 + c;
                        const uint4 v = dequant8(words[c], s2, m2);
                        *reinterpret_cast<uint4*>(arow + ((chunk ^ (rw & 7)) << 4)) = v;
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(deq_bar(s));
                }
            }
        }
        // ---------------- epilogue (the accumulator barrier is also the drain
        // of every MMA issued, so it does not stop early on the abort flag)
        const bool ok = mbar_wait(acc_bar, 0, nullptr, lim);
        if (!ok) report(p.status, fg::kDevTimeout);
        tc_fence_after();
        const int q = warp & 3;               // TMEM lane quarter this warp may read
        const int colhalf = (warp - 2) >> 2;  // two warps per quarter split the columns
        const int row = q * 32 + lane;
        const int n = feat0 + row;
        const bool live = ok && !*abort_flag;
        float bias = 0.0f;
        if (!kF32Out && live && p.bias != nullptr && n < p.N && gridDim.z == 1)
            bias = __half2float(p.bias[n]);
        for (int c0 = 16 * colhalf; c0 < p.nt; c0 += 32) {
            uint32_t r[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, r);
            tmem_wait_ld();
            if (!live || n >= p.N) continue;
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
                    if (p.residual) v = __fadd_rn(v, __half2float(p.residual[idx]));
                    p.Y[idx] = __float2half_rn(v);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, ncols);
}

// Fixed-order sum of the K-split partials, then the epilogue.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ partial,
                                                            int splits, int64_t M, int64_t N,
                                                            const __half* __restrict__ bias,
                                                            const __half* __restrict__ residual,
                                                            int act, __half* __restrict__ Y) {
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

// 2-D row-major tensor [rows][cols] of `esize`-byte elements; box = {bx, by}.
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

int stages_for(int nt, bool dq) {
    const int per = static_cast<int>(kABytes + nt * 128 + (dq ? kCBytes : 0));
    int s = (kSmemLimit - 1024 - 8 * (3 * kMaxStages + 1) - 16) / per;
    if (s > kMaxStages) s = kMaxStages;
    return s;
}

size_t smem_for(int nt, bool dq, int stages) {
    return 1024 + static_cast<size_t>(stages) * (kABytes + nt * 128 + (dq ? kCBytes : 0)) +
           8 * (3 * stages + 1) + 16;
}

template <bool kDequant, bool kF32Out>
fg_status run_gemm(const CUtensorMap& tmX, const CUtensorMap& tmW, GemmParams& p,
                   const fg::GemmPlan& plan, cudaStream_t st) {
    p.stages = stages_for(plan.nt, kDequant);
    const size_t smem = smem_for(plan.nt, kDequant, p.stages);
    auto kern = gemm_tc_kernel<kDequant, kF32Out>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return fg::cuda_error(e, "gemm smem attribute");
    dim3 grid(plan.feat_tiles * plan.tok_tiles, 1, plan.splits);
    p.feat_tiles = plan.feat_tiles;
    p.tok_tiles = plan.tok_tiles;
    const double M = p.M, N = p.N, K = p.K;
    // algorithmic traffic: the weight once (4-bit codes + fp32 (min, scale) per
    // 64, or fp16), X once, Y once (+ residual, or fp32 partials / logits)
    const double wbytes = kDequant ? N * K * 0.625 : N * K * 2.0;
    const double ybytes = kF32Out ? M * N * 4.0
                                  : (plan.splits > 1 ? plan.splits * M * N * 4.0
                                                     : M * N * 2.0 * (p.residual ? 2.0 : 1.0));
    const int cls = !kDequant ? FG_TRACE_OTHER
                              : (p.M > 256 ? FG_TRACE_GEMM_PREFILL : FG_TRACE_GEMM_DECODE);
    fg::TraceScope ts(cls, st, 2.0 * M * N * K, wbytes + M * K * 2.0 + ybytes);
    kern<<<grid, kThreads, smem, st>>>(tmX, tmW, p);
    return fg::cuda_error(cudaGetLastError(), "gemm launch");
}

}  // namespace

namespace fg {

// Tile plan.  It depends on M only through the number of 256-row activation
// tiles, and the K split only on (N, K) -- and is used only when all rows fit
// one tile -- so every row's result is independent of M and of the other rows
// (the row-by-row and zig-zag block orders must agree bit for bit).
GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K) {
    GemmPlan pl{};
    pl.tok_tiles = static_cast<int>(cdiv(M, 256));
    if (pl.tok_tiles < 1) pl.tok_tiles = 1;
    int64_t rows = cdiv(M, pl.tok_tiles);
    pl.nt = static_cast<int>(cdiv(rows, 16) * 16);
    if (pl.nt < 16) pl.nt = 16;
    pl.feat_tiles = static_cast<int>(cdiv(N, kTileF));
    pl.splits = 1;
    const int64_t kchunks = K / kChunk;
    if (pl.tok_tiles == 1) {
        const int sms = num_sms();
        int s = sms / pl.feat_tiles;
        if (s > 8) s = 8;
        if (s > kchunks / 8) s = static_cast<int>(kchunks / 8);
        if (s < 1) s = 1;
        pl.splits = s;
    }
    if (pl.splits > 1) {
        // equalise the chunk ranges; drop splits that would be empty
        const int64_t per = cdiv(kchunks, pl.splits);
        pl.splits = static_cast<int>(cdiv(kchunks, per));
    }
    pl.ws_bytes = pl.splits > 1 ? static_cast<size_t>(pl.splits) * M * N * sizeof(float) : 0;
    return pl;
}

fg_status launch_gemm_g4(const __half* X, int64_t M, const fg_q4* W, const __half* bias,
                         const __half* residual, int act, __half* Y, void* ws, size_t ws_bytes,
                         cudaStream_t st) {
    if (M == 0) return FG_OK;
    const int64_t N = W->rows, K = W->cols;
    const GemmPlan pl = plan_gemm(M, N, K);
    if (pl.ws_bytes > 0 && (ws == nullptr || ws_bytes < pl.ws_bytes))
        return set_error(FG_ERR_WORKSPACE, "dequant_gemm: workspace %zu < %zu bytes", ws_bytes,
                         pl.ws_bytes);
    CUtensorMap tmX, tmC;
    fg_status s = make_tmap(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K, M, kChunk, pl.nt,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != FG_OK) return s;
    s = make_tmap(&tmC, W->codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, N, kChunk / 2, kTileF,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
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
    p.kc_per_split = static_cast<int>(cdiv(p.kchunks, pl.splits));
    p.act = act;
    p.status = device_status_ptr();
    p.wait_ns = wait_limit_ns();
    p.drop_arrive = take_drop_arrive();
    s = run_gemm<true, false>(tmX, tmC, p, pl, st);
    if (s != FG_OK || pl.splits == 1) return s;
    const int64_t nv = M * N / 4;
    int64_t blocks = cdiv(nv, 256);
    if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, pl.splits * M * N * 4.0 + M * N * 4.0);
    splitk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        p.partial, pl.splits, M, N, bias, residual, act, Y);
    return cuda_error(cudaGetLastError(), "splitk reduce launch");
}

fg_status launch_gemm_f16_f32out(const __half* X, int64_t M, const __half* W, int64_t N,
                                 int64_t K, float* Y, cudaStream_t st) {
    if (M == 0) return FG_OK;
    GemmPlan pl = plan_gemm(M, N, K);
    pl.splits = 1;
    CUtensorMap tmX, tmW;
    fg_status s = make_tmap(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K, M, kChunk, pl.nt,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != FG_OK) return s;
    s = make_tmap(&tmW, W, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K, N, kChunk, kTileF,
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
    return run_gemm<false, true>(tmX, tmW, p, pl, st);
}

}  // namespace fg
