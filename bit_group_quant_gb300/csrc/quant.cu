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

// Contiguous groups: group g covers x[64 g .. 64 g + 63].
__global__ void __launch_bounds__(256) quantize_g4_kernel(const uint4* __restrict__ x,
                                                          int64_t ngroups,
                                                          uint32_t* __restrict__ codes,
                                                          float2* __restrict__ meta) {
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3;       // group within the warp's 4
    const int lane8 = lane & 7;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t w = warp; w * 4 < ngroups; w += nwarps) {
        const int64_t g = w * 4 + sub;
        const bool valid = g < ngroups;
        float v[8];
        if (valid) {
            unpack8(ld_stream(x + g * 8 + lane8), v);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        float mn, scale;
        const uint32_t packed = quantize8(v, mn, scale);
        if (valid) {
            codes[g * 8 + lane8] = packed;
            if (lane8 == 0) meta[g] = make_float2(mn, scale);
        }
    }
}

// Exact dequantisation: x^ = fp16(fma(code, scale, min)).
__global__ void __launch_bounds__(256) dequant_g4_kernel(const uint32_t* __restrict__ codes,
                                                         const float2* __restrict__ meta,
                                                         int64_t ngroups,
                                                         uint4* __restrict__ x) {
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
// parts (per head, groups of 64 along d) go to cache slot slot0 + t.
// One group per 8 lanes, as in quantize_g4_kernel.  Groups are numbered
// (k/v, sequence, head, token, group in the row) with the group in the row
// fastest, then the token: consecutive groups go to consecutive cache rows of
// one (sequence, head), so a warp's and its neighbours' codes and (min,
// scale) stores are contiguous.
__global__ void __launch_bounds__(256) kv_store_kernel(const __half* __restrict__ qkv, int64_t ld,
                                                       int32_t B, int32_t T, int32_t H,
                                                       int32_t d, int32_t cap, int32_t slot0,
                                                       uint8_t* __restrict__ k_codes,
                                                       uint8_t* __restrict__ v_codes,
                                                       float* __restrict__ k_meta,
                                                       float* __restrict__ v_meta) {
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3;
    const int lane8 = lane & 7;
    const int gpr = d / 64;                                   // groups per head row
    const int64_t per_head = static_cast<int64_t>(T) * gpr;     // groups per (k/v, b, h)
    const int64_t ngroups = static_cast<int64_t>(2) * B * H * per_head;
    const int64_t h1 = static_cast<int64_t>(H) * d;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t w = warp; w * 4 < ngroups; w += nwarps) {
        const int64_t g = w * 4 + sub;
        const bool valid = g < ngroups;
        int64_t tok = 0, t = 0, bh = 0;
        int is_v = 0, h = 0, gi = 0;
        float v[8];
        if (valid) {
            const int64_t head = g / per_head;           // (k/v, b, h)
            const int64_t r2 = g % per_head;
            t = r2 / gpr;
            gi = static_cast<int>(r2 % gpr);
            is_v = static_cast<int>(head / (static_cast<int64_t>(B) * H));
            bh = head % (static_cast<int64_t>(B) * H);
            h = static_cast<int>(bh % H);
            tok = (bh / H) * T + t;
            const __half* src = qkv + tok * ld + (1 + is_v) * h1 + static_cast<int64_t>(h) * d +
                                gi * 64 + lane8 * 8;
            unpack8(*reinterpret_cast<const uint4*>(src), v);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        float mn, scale;
        const uint32_t packed = quantize8(v, mn, scale);
        if (valid) {
            const int64_t row = bh * cap + slot0 + t;
            uint8_t* cdst = (is_v ? v_codes : k_codes) + row * (d / 2) + gi * 32;
            reinterpret_cast<uint32_t*>(cdst)[lane8] = packed;
            if (lane8 == 0) {
                float* mdst = (is_v ? v_meta : k_meta) + (row * gpr + gi) * 2;
                *reinterpret_cast<float2*>(mdst) = make_float2(mn, scale);
            }
        }
    }
}

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
    const int grid = grid_for(ngroups, 32);  // 32 groups per 256-thread block
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, ngroups * (128.0 + 40.0));
    quantize_g4_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(x), ngroups,
                                             reinterpret_cast<uint32_t*>(codes),
                                             reinterpret_cast<float2*>(meta));
    return cuda_error(cudaGetLastError(), "quantize_g4 launch");
}

fg_status launch_dequant_g4(const uint8_t* codes, const float* meta, int64_t ngroups,
                            __half* x, cudaStream_t st) {
    if (ngroups == 0) return FG_OK;
    const int grid = grid_for(ngroups * 8, 256);
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, ngroups * (128.0 + 40.0));
    dequant_g4_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint32_t*>(codes),
                                            reinterpret_cast<const float2*>(meta), ngroups,
                                            reinterpret_cast<uint4*>(x));
    return cuda_error(cudaGetLastError(), "dequant_g4 launch");
}

fg_status launch_kv_store(const __half* qkv, int64_t ld, int32_t B, int32_t T, int32_t H,
                          int32_t d, const fg_kv4* c, int32_t slot0, cudaStream_t st) {
    const int64_t ngroups = static_cast<int64_t>(B) * T * 2 * H * (d / 64);
    if (ngroups == 0) return FG_OK;
    const int grid = grid_for(ngroups, 32);
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, ngroups * (128.0 + 40.0));
    kv_store_kernel<<<grid, 256, 0, st>>>(qkv, ld, B, T, H, d, c->cap, slot0, c->k_codes,
                                          c->v_codes, c->k_meta, c->v_meta);
    return cuda_error(cudaGetLastError(), "kv_store launch");
}

}  // namespace fg
