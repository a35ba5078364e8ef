// quant.cu -- group-wise 4-bit quantiser (weights at load time, K/V rows at
// append), its exact dequantiser, and the KV-cache row store.
//
// Quantisation ("FlexGen 完全拆解", section on weight and KV-cache
// compression; packing per "bjbfmj.com/news/40234" section 6.3): per group of
// 64 contiguous values, min/max, 4-bit unsigned codes, two codes per byte.
//
// Layout of the work: a group is 128 bytes of fp16, read as one 16-byte
// vector by each of 8 consecutive lanes, so a warp streams 4 groups (512
// contiguous bytes) per iteration.  Min/max meet through 3 xor-shuffles; each
// lane writes its 8 codes as one 32-bit word, and lane 0 of the group writes
// (min, scale) as one 8-byte store.  The kernel is HBM-bound at 2 + 0.625
// bytes per element.
#include <math_constants.h>

#include "fg_internal.cuh"

namespace {

using namespace fgd;

__device__ __forceinline__ void unpack8(const uint4& raw, float (&v)[8]) {
    const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// One lane quantises one whole group of 64 fp16 values staged in shared
// memory (a row of kQRow bytes: 128 of values, padding against bank
// conflicts): min and max in the IEEE total order over the 64, scale =
// (M - m) / 15 by IEEE division, then the 64 codes (code4), packed two per
// byte with the lower element in the low nibble: word i (written to
// codes_dst[i]) holds elements 8i .. 8i + 7.  The same arithmetic as
// quantize8, for one lane.
constexpr int kQRow = 144;
constexpr int kQWarps = 8;   // warps per block; each stages 32 groups

__device__ __forceinline__ void quantize64(const uint8_t* row, uint32_t* codes_dst, float2* meta_dst) {
    float v[8];
    // min and max by the hardware fminf / fmaxf; they can differ from the
    // IEEE total order only in the sign of a zero result, so a zero min or
    // max is recomputed in the total order
    float mn = CUDART_INF_F, mx = -CUDART_INF_F;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        unpack8(*reinterpret_cast<const uint4*>(row + 16 * i), v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            mn = fminf(mn, v[j]);
            mx = fmaxf(mx, v[j]);
        }
    }
    if (mn == 0.0f || mx == 0.0f) {
        unpack8(*reinterpret_cast<const uint4*>(row), v);
        mn = v[0];
        mx = v[0];
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {
            unpack8(*reinterpret_cast<const uint4*>(row + 16 * i), v);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                mn = tmin(mn, v[j]);
                mx = tmax(mx, v[j]);
            }
        }
    }
    const float scale = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
    const float inv = scale != 0.0f ? __frcp_rn(scale) : 0.0f;
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
        uint32_t packed = 0u;
        if (scale != 0.0f) {
            unpack8(*reinterpret_cast<const uint4*>(row + 16 * i), v);
            uint32_t ties = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                bool near_tie;
                packed |= code4_fast(__fsub_rn(v[j], mn), inv, &near_tie) << (4 * j);
                ties |= (near_tie ? 1u : 0u) << j;
            }
            // rare: decide the elements near a rounding tie by IEEE division
            for (; ties; ties &= ties - 1) {
                const int j = __ffs(ties) - 1;
                const float x = __half2float(reinterpret_cast<const __half*>(row + 16 * i)[j]);
                packed = (packed & ~(0xFu << (4 * j))) | (code4_exact(__fsub_rn(x, mn), scale) << (4 * j));
            }
        }
        codes_dst[i] = packed;
    }
    *meta_dst = make_float2(mn, scale);
}

// Contiguous groups: group g covers x[64 g .. 64 g + 63].  Each warp takes 32
// consecutive groups at a time: the 4 KB come in by coalesced 16-byte loads
// into the warp's staging rows, then lane l quantises group l and writes its
// 32 code bytes and (min, scale) -- consecutive lanes, consecutive addresses.
__global__ void __launch_bounds__(32 * kQWarps) quantize_g4_kernel(const uint4* __restrict__ x,
                                                                  int64_t ngroups,
                                                                  uint32_t* __restrict__ codes,
                                                                  float2* __restrict__ meta) {
    __shared__ __align__(16) uint8_t stage[kQWarps][32 * kQRow];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    uint8_t* st = stage[wib];
    const int64_t warp = static_cast<int64_t>(blockIdx.x) * kQWarps + wib;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kQWarps;
    for (int64_t base = warp * 32; base < ngroups; base += nwarps * 32) {
        const int ng = static_cast<int>(min(static_cast<int64_t>(32), ngroups - base));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = lane + 32 * k, gg = i >> 3, p = i & 7;
            if (gg < ng)
                *reinterpret_cast<uint4*>(st + gg * kQRow + 16 * p) = ld_stream(x + (base + gg) * 8 + p);
        }
        __syncwarp();
        if (lane < ng) quantize64(st + lane * kQRow, codes + (base + lane) * 8, meta + base + lane);
        __syncwarp();   // the staging rows are refilled next
    }
}

// Exact dequantisation: x^ = fp16(fma(code, scale, min)).
__global__ void __launch_bounds__(256) dequant_g4_kernel(const uint32_t* __restrict__ codes,
                                                         const float2* __restrict__ meta,
                                                         int64_t ngroups,
                                                         uint4* __restrict__ x) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    griddep_wait();
    griddep_launch();
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         t < ngroups * 8; t += nthreads) {
        const int64_t g = t >> 3;
        const uint32_t w = codes[t];
        const float2 m = meta[g];
        uint4 out;
        uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float a = __fmaf_rn(static_cast<float>((w >> (8 * i)) & 0xF), m.y, m.x);
            const float b = __fmaf_rn(static_cast<float>((w >> (8 * i + 4)) & 0xF), m.y, m.x);
            const __half2 h = __halves2half2(__float2half_rn(a), __float2half_rn(b));
            o[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        x[t] = out;
    }
}

// KV-cache row store: token t of sequence b is qkv row (b*T + t); its k and v
// parts (per head, groups of 64 along d) go to cache slot slot0 + t.  Groups
// are numbered (k/v, sequence, head, token, group in the row) with the group
// in the row fastest, then the token: consecutive groups fill consecutive
// cache rows of one (sequence, head).  Each warp takes 32 consecutive groups:
// lane l finds group l's source, the warp stages the 32 x 128 bytes by
// 16-byte loads (each group's address passed by shuffle), and lane l
// quantises group l (quantize64) and writes it -- the warp's code and
// (min, scale) stores are contiguous.
__global__ void __launch_bounds__(32 * kQWarps) kv_store_kernel(
    const __half* __restrict__ qkv, int64_t ld, int32_t B, int32_t T, int32_t H, int32_t d,
    int32_t cap, int32_t slot0, uint8_t* __restrict__ k_codes, uint8_t* __restrict__ v_codes,
    float* __restrict__ k_meta, float* __restrict__ v_meta) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    griddep_wait();
    griddep_launch();
    __shared__ __align__(16) uint8_t stage[kQWarps][32 * kQRow];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    uint8_t* st = stage[wib];
    const int gpr = d / 64;                                   // groups per head row
    const int64_t per_head = static_cast<int64_t>(T) * gpr;     // groups per (k/v, b, h)
    const int64_t ngroups = static_cast<int64_t>(2) * B * H * per_head;
    const int64_t h1 = static_cast<int64_t>(H) * d;
    const int64_t warp = static_cast<int64_t>(blockIdx.x) * kQWarps + wib;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kQWarps;
    for (int64_t base = warp * 32; base < ngroups; base += nwarps * 32) {
        const int ng = static_cast<int>(min(static_cast<int64_t>(32), ngroups - base));
        // this lane's group: source, destination row, k or v, group in the row
        const __half* src = qkv;
        int64_t row = 0;
        int is_v = 0, gi = 0;
        if (lane < ng) {
            const int64_t g = base + lane;
            const int64_t head = g / per_head;           // (k/v, b, h)
            const int64_t r2 = g % per_head;
            const int64_t t = r2 / gpr;
            gi = static_cast<int>(r2 % gpr);
            is_v = static_cast<int>(head / (static_cast<int64_t>(B) * H));
            const int64_t bh = head % (static_cast<int64_t>(B) * H);
            const int64_t h = bh % H;
            const int64_t tok = (bh / H) * T + t;
            src = qkv + tok * ld + (1 + is_v) * h1 + h * d + gi * 64;
            row = bh * cap + slot0 + t;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = lane + 32 * k, gg = i >> 3, p = i & 7;
            const __half* gs = reinterpret_cast<const __half*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src), gg));
            if (gg < ng)
                *reinterpret_cast<uint4*>(st + gg * kQRow + 16 * p) =
                    *reinterpret_cast<const uint4*>(gs + 8 * p);
        }
        __syncwarp();
        if (lane < ng)
            quantize64(st + lane * kQRow,
                       reinterpret_cast<uint32_t*>((is_v ? v_codes : k_codes) + row * (d / 2) + gi * 32),
                       reinterpret_cast<float2*>((is_v ? v_meta : k_meta) + (row * gpr + gi) * 2));
        __syncwarp();   // the staging rows are refilled next
    }
}

// Grid for a grid-stride kernel: one block per per_block work items, at most
// 8 blocks per SM.
int grid_for(int64_t work_items, int per_block) {
    int64_t blocks = fg::cdiv(work_items, per_block);
    const int64_t cap = static_cast<int64_t>(fg::num_sms()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

}  // namespace

namespace fg {

fg_status launch_quantize_g4(const __half* x, int64_t ngroups, uint8_t* codes, float* meta,
                             cudaStream_t st) {
    if (ngroups == 0) return FG_OK;
    const int grid = grid_for(ngroups, 32 * kQWarps);  // 32 groups per warp at a time
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, ngroups * (128.0 + 40.0));
    quantize_g4_kernel<<<grid, 32 * kQWarps, 0, st>>>(reinterpret_cast<const uint4*>(x), ngroups,
                                             reinterpret_cast<uint32_t*>(codes),
                                             reinterpret_cast<float2*>(meta));
    return cuda_error(cudaGetLastError(), "quantize_g4 launch");
}

fg_status launch_dequant_g4(const uint8_t* codes, const float* meta, int64_t ngroups,
                            __half* x, cudaStream_t st, int trace_cls) {
    if (ngroups == 0) return FG_OK;
    const int grid = grid_for(ngroups * 8, 256);
    TraceScope ts(trace_cls, st, 0.0, ngroups * (128.0 + 40.0));
    {
        const cudaError_t le_ = fg::launch_pdl(dequant_g4_kernel, dim3(grid), dim3(256), 0, st,
            reinterpret_cast<const uint32_t*>(codes),
                                            reinterpret_cast<const float2*>(meta), ngroups,
                                            reinterpret_cast<uint4*>(x));
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "dequant_g4_kernel launch");
    }
    return cuda_error(cudaGetLastError(), "dequant_g4 launch");
}

fg_status launch_kv_store(const __half* qkv, int64_t ld, int32_t B, int32_t T, int32_t H,
                          int32_t d, const fg_kv4* c, int32_t slot0, cudaStream_t st) {
    const int64_t ngroups = static_cast<int64_t>(B) * T * 2 * H * (d / 64);
    if (ngroups == 0) return FG_OK;
    const int grid = grid_for(ngroups, 32 * kQWarps);  // 32 groups per warp at a time
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, ngroups * (128.0 + 40.0));
    {
        const cudaError_t le_ = fg::launch_pdl(kv_store_kernel, dim3(grid), dim3(32 * kQWarps), 0, st,
            qkv, ld, B, T, H, d, c->cap, slot0, c->k_codes,
                                          c->v_codes, c->k_meta, c->v_meta);
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "kv_store_kernel launch");
    }
    return cuda_error(cudaGetLastError(), "kv_store launch");
}

}  // namespace fg
