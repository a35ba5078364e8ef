// attn.cu -- decode attention over the 4-bit KV cache (with the new token's
// K/V append fused in) and causal prefill attention.
//
// Dataflow ("FlexGen 完全拆解", section on the inference dataflow): the
// prefill computes Q, K, V for all prompt tokens; each decode step appends
// the new k, v row to the cache and attends the single query over the s+t
// cached rows.  Stored 4-bit tensors are dequantised to FP16 before use
// (section on compression), so every cached row -- the new one included --
// is read back through dequantisation.
#include <math_constants.h>

#include "fg_internal.cuh"

namespace {

using namespace fgd;

constexpr int kDecThreads = 128;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exact dequantised value, as a float: fp16(fma(code, scale, min)).
__device__ __forceinline__ float deq(uint32_t code, float2 m) {
    return __half2float(__float2half_rn(__fmaf_rn(static_cast<float>(code), m.y, m.x)));
}

// One CTA per (head, sequence).  Shared memory: scores[L] then the partial
// output table [R][D].
template <int D>
__global__ void __launch_bounds__(kDecThreads) decode_attn_kernel(
    const __half* __restrict__ qkv, int64_t ld, int32_t H, int32_t cap, int32_t pos,
    int32_t fuse_append, uint8_t* k_codes, uint8_t* v_codes, float* k_meta, float* v_meta,
    __half* __restrict__ out) {
    constexpr int GPR = D / 64;          // groups per head row
    constexpr int TPR = D / 8;           // threads per V row (8 dims each)
    constexpr int R = kDecThreads / TPR; // V rows in flight per pass
    extern __shared__ float dsm[];
    __shared__ float qf[D];
    __shared__ float red[kDecThreads / 32];

    const int h = blockIdx.x, b = blockIdx.y;
    const int L = pos + 1;
    const int64_t h1 = static_cast<int64_t>(H) * D;
    const int64_t row0 = (static_cast<int64_t>(b) * H + h) * cap;  // cache row of slot 0
    float* sc = dsm;
    float* part = dsm + ((L + 3) & ~3);

    if (fuse_append && threadIdx.x < 32) {
        const int lane = threadIdx.x, grp = lane >> 3, lane8 = lane & 7;
        const bool valid = grp < 2 * GPR;
        const int is_v = grp / GPR, gi = grp % GPR;
        float v[8];
        if (valid) {
            const uint4 raw = *reinterpret_cast<const uint4*>(
                qkv + b * ld + (1 + is_v) * h1 + static_cast<int64_t>(h) * D + gi * 64 + lane8 * 8);
            const __half2* hh = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(hh[i]);
                v[2 * i] = f.x;
                v[2 * i + 1] = f.y;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        float mn, scale;
        const uint32_t packed = quantize8(v, mn, scale);
        if (valid) {
            const int64_t row = row0 + pos;
            uint8_t* cdst = (is_v ? v_codes : k_codes) + row * (D / 2) + gi * 32;
            reinterpret_cast<uint32_t*>(cdst)[lane8] = packed;
            if (lane8 == 0) {
                float* mdst = (is_v ? v_meta : k_meta) + (row * GPR + gi) * 2;
                *reinterpret_cast<float2*>(mdst) = make_float2(mn, scale);
            }
        }
    }
    for (int t = threadIdx.x; t < D; t += kDecThreads)
        qf[t] = __half2float(qkv[b * ld + static_cast<int64_t>(h) * D + t]);
    __syncthreads();

    const float scale = __fdiv_rn(1.0f, __fsqrt_rn(static_cast<float>(D)));
    // Scores: one cache row per thread, dot product in ascending dimension.
    float lmax = -CUDART_INF_F;
    for (int j = threadIdx.x; j < L; j += kDecThreads) {
        const uint4* kc = reinterpret_cast<const uint4*>(k_codes + (row0 + j) * (D / 2));
        const float2* km = reinterpret_cast<const float2*>(k_meta + (row0 + j) * GPR * 2);
        float dot = 0.0f;
#pragma unroll
        for (int g = 0; g < GPR; ++g) {
            const float2 m = km[g];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint4 raw = kc[g * 2 + u];
                const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int dim = g * 64 + u * 32 + wi * 8 + e;
                        dot = __fadd_rn(dot, __fmul_rn(qf[dim], deq((w4[wi] >> (4 * e)) & 0xF, m)));
                    }
                }
            }
        }
        const float s = __fmul_rn(dot, scale);
        sc[j] = s;
        lmax = fmaxf(lmax, s);
    }
    lmax = warp_max(lmax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lmax;
    __syncthreads();
    float mx = red[0];
#pragma unroll
    for (int i = 1; i < kDecThreads / 32; ++i) mx = fmaxf(mx, red[i]);
    __syncthreads();
    float lsum = 0.0f;
    for (int j = threadIdx.x; j < L; j += kDecThreads) {
        const float p = expf(sc[j] - mx);
        sc[j] = p;
        lsum += p;
    }
    lsum = warp_sum(lsum);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lsum;
    __syncthreads();
    float l = 0.0f;
#pragma unroll
    for (int i = 0; i < kDecThreads / 32; ++i) l += red[i];

    // Weighted V sum: TPR threads per row, 8 dims each; R rows per pass.
    const int r = threadIdx.x / TPR, c8 = threadIdx.x % TPR;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    for (int j = r; j < L; j += R) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(v_codes + (row0 + j) * (D / 2) + c8 * 4);
        const float2 m = reinterpret_cast<const float2*>(v_meta + (row0 + j) * GPR * 2)[c8 / 8];
        const float p = sc[j];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], __fmul_rn(p, deq((w >> (4 * e)) & 0xF, m)));
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) part[r * D + c8 * 8 + e] = acc[e];
    __syncthreads();
    for (int t = threadIdx.x; t < D; t += kDecThreads) {
        float o = 0.0f;
#pragma unroll
        for (int rr = 0; rr < R; ++rr) o += part[rr * D + t];
        out[b * h1 + static_cast<int64_t>(h) * D + t] = __float2half_rn(__fdiv_rn(o, l));
    }
}

// Causal prefill attention over fp16 Q/K/V.  One CTA per (32-query tile,
// head, sequence); 4 threads per query, each owning D/4 interleaved dims
// (dim = 4*e + part) so the 4 reads of a key row hit 4 different banks.
constexpr int kPreQ = 32;
constexpr int kPreK = 32;

template <int D>
__global__ void __launch_bounds__(128) prefill_attn_kernel(const __half* __restrict__ qkv,
                                                           int32_t s, int32_t H,
                                                           __half* __restrict__ out) {
    constexpr int DP = D / 4;
    __shared__ float Ks[kPreK][D];
    __shared__ float Vs[kPreK][D];
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int64_t h1 = static_cast<int64_t>(H) * D, ld = 3 * h1;
    const int part = threadIdx.x & 3;
    const int i = qt * kPreQ + (threadIdx.x >> 2);
    const unsigned gmask = 0xFu << (threadIdx.x & 28);
    const __half* base = qkv + static_cast<int64_t>(b) * s * ld + static_cast<int64_t>(h) * D;
    const float scale = __fdiv_rn(1.0f, __fsqrt_rn(static_cast<float>(D)));

    float q[DP], acc[DP];
    float m = -CUDART_INF_F, l = 0.0f;
#pragma unroll
    for (int e = 0; e < DP; ++e) {
        q[e] = (i < s) ? __half2float(base[static_cast<int64_t>(i) * ld + 4 * e + part]) : 0.0f;
        acc[e] = 0.0f;
    }
    const int last_q = min(s - 1, qt * kPreQ + kPreQ - 1);
    for (int k0 = 0; k0 <= last_q; k0 += kPreK) {
        __syncthreads();
        for (int t = threadIdx.x; t < kPreK * D / 8; t += blockDim.x) {
            const int jj = t / (D / 8), c = (t % (D / 8)) * 8;
            const int j = k0 + jj;
            float kv[8], vv[8];
            if (j < s) {
                const uint4 kr = *reinterpret_cast<const uint4*>(base + static_cast<int64_t>(j) * ld + h1 + c);
                const uint4 vr = *reinterpret_cast<const uint4*>(base + static_cast<int64_t>(j) * ld + 2 * h1 + c);
                const __half2* kh = reinterpret_cast<const __half2*>(&kr);
                const __half2* vh = reinterpret_cast<const __half2*>(&vr);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 kf = __half22float2(kh[u]);
                    const float2 vf = __half22float2(vh[u]);
                    kv[2 * u] = kf.x;
                    kv[2 * u + 1] = kf.y;
                    vv[2 * u] = vf.x;
                    vv[2 * u + 1] = vf.y;
                }
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) kv[u] = vv[u] = 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                Ks[jj][c + u] = kv[u];
                Vs[jj][c + u] = vv[u];
            }
        }
        __syncthreads();
        if (i < s) {
            float sc[kPreK];
            float tmax = -CUDART_INF_F;
#pragma unroll
            for (int jj = 0; jj < kPreK; ++jj) {
                float dot = 0.0f;
#pragma unroll
                for (int e = 0; e < DP; ++e) dot += q[e] * Ks[jj][4 * e + part];
                dot += __shfl_xor_sync(gmask, dot, 1);
                dot += __shfl_xor_sync(gmask, dot, 2);
                const bool ok = (k0 + jj) <= i;
                sc[jj] = ok ? dot * scale : -CUDART_INF_F;
                tmax = fmaxf(tmax, sc[jj]);
            }
            const float mnew = fmaxf(m, tmax);
            const float corr = expf(m - mnew);
            l *= corr;
#pragma unroll
            for (int e = 0; e < DP; ++e) acc[e] *= corr;
#pragma unroll
            for (int jj = 0; jj < kPreK; ++jj) {
                const float p = expf(sc[jj] - mnew);
                l += p;
#pragma unroll
                for (int e = 0; e < DP; ++e) acc[e] += p * Vs[jj][4 * e + part];
            }
            m = mnew;
        }
    }
    if (i < s) {
        __half* o = out + (static_cast<int64_t>(b) * s + i) * h1 + static_cast<int64_t>(h) * D;
        const float inv = 1.0f / l;
#pragma unroll
        for (int e = 0; e < DP; ++e) o[4 * e + part] = __float2half_rn(acc[e] * inv);
    }
}

template <int D>
fg_status launch_decode_t(const __half* qkv, int64_t ld, const fg_kv4* c, int32_t pos,
                          int32_t fuse_append, __half* out, cudaStream_t st) {
    const int L = pos + 1;
    const size_t smem = sizeof(float) * (((L + 3) & ~3) + kDecThreads * 8);
    auto kern = decode_attn_kernel<D>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return fg::cuda_error(e, "decode_attn smem attribute");
    }
    dim3 grid(c->H, c->B);
    // algorithmic traffic: L packed K and V rows (codes + fp32 meta) per (b, h),
    // the new k, v written back, q/k/v read and the output written
    const double row = D / 2 + (D / 64) * 8.0;
    const double bh = static_cast<double>(c->B) * c->H;
    fg::TraceScope ts(FG_TRACE_ATTN_DECODE, st, 4.0 * bh * L * D,
                      bh * (2.0 * L * row + (fuse_append ? 2.0 * row : 0.0) + 3.0 * D * 2 + D * 2));
    kern<<<grid, kDecThreads, smem, st>>>(qkv, ld, c->H, c->cap, pos, fuse_append, c->k_codes,
                                          c->v_codes, c->k_meta, c->v_meta, out);
    return fg::cuda_error(cudaGetLastError(), "decode_attn launch");
}

}  // namespace

namespace fg {

fg_status launch_decode_attn(const __half* qkv, int64_t ld, const fg_kv4* c, int32_t pos,
                             int32_t fuse_append, __half* out, cudaStream_t st) {
    if (c->B == 0) return FG_OK;
    if (c->d == 64) return launch_decode_t<64>(qkv, ld, c, pos, fuse_append, out, st);
    return launch_decode_t<128>(qkv, ld, c, pos, fuse_append, out, st);
}

fg_status launch_prefill_attn(const __half* qkv, int32_t B, int32_t s, int32_t H, int32_t d,
                              __half* out, cudaStream_t st) {
    if (B == 0 || s == 0) return FG_OK;
    dim3 grid(static_cast<unsigned>(cdiv(s, kPreQ)), H, B);
    const double bh = static_cast<double>(B) * H;
    TraceScope ts(FG_TRACE_ATTN_PREFILL, st, 2.0 * bh * s * (s + 1.0) * d,
                  bh * s * d * 2.0 * 4.0);
    if (d == 64)
        prefill_attn_kernel<64><<<grid, 128, 0, st>>>(qkv, s, H, out);
    else
        prefill_attn_kernel<128><<<grid, 128, 0, st>>>(qkv, s, H, out);
    return cuda_error(cudaGetLastError(), "prefill_attn launch");
}

}  // namespace fg
