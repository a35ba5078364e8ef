// small.cu -- LayerNorm, token + position embedding and the greedy argmax
// (the OPT layer's pre-LN normalisations, the model input and the choice of
// the next token).  All are bandwidth-trivial next to the projections.
#include <math_constants.h>

#include "fg_internal.cuh"

namespace {

constexpr int kLnThreads = 256;
constexpr int kLnMaxVec = 8;   // up to 8 x 8 x 256 = 16384 columns held in registers

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int i = 0; i < kLnThreads / 32; ++i) t += red[i];
    return t;
}

// y = (x - mean) / sqrt(var + eps) * gamma + beta; mean, biased variance fp32.
// One block per row; the row stays in registers as packed fp16 (4 registers
// per 8 values, converted in each pass) so that enough rows are in flight
// per SM to cover the load latency.
__global__ void __launch_bounds__(kLnThreads) layernorm_kernel(const __half* __restrict__ x,
                                                               int64_t cols, int64_t x_ld,
                                                               const __half* __restrict__ g,
                                                               const __half* __restrict__ b,
                                                               float eps, __half* __restrict__ y) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    fgd::griddep_wait();
    fgd::griddep_launch();
    __shared__ float red[kLnThreads / 32];
    const int64_t row = blockIdx.x;
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * x_ld);
    const int nvec = static_cast<int>(cols / 8);
    uint4 raw[kLnMaxVec];
#pragma unroll
    for (int i = 0; i < kLnMaxVec; ++i) {
        const int c = threadIdx.x + i * kLnThreads;
        raw[i] = c < nvec ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kLnMaxVec; ++i) {
        if (threadIdx.x + i * kLnThreads < nvec) {
            const __half2* h = reinterpret_cast<const __half2*>(&raw[i]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __half22float2(h[j]);
                s += f.x + f.y;
            }
        }
    }
    const float mean = __fdiv_rn(block_sum(s, red), static_cast<float>(cols));
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < kLnMaxVec; ++i) {
        if (threadIdx.x + i * kLnThreads < nvec) {
            const __half2* h = reinterpret_cast<const __half2*>(&raw[i]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __half22float2(h[j]);
                const float d0 = __fsub_rn(f.x, mean);
                q = __fadd_rn(q, __fmul_rn(d0, d0));
                const float d1 = __fsub_rn(f.y, mean);
                q = __fadd_rn(q, __fmul_rn(d1, d1));
            }
        }
    }
    const float var = __fdiv_rn(block_sum(q, red), static_cast<float>(cols));
    const float denom = __fsqrt_rn(__fadd_rn(var, eps));
    uint4* yr = reinterpret_cast<uint4*>(y + row * cols);
    const uint4* gr = reinterpret_cast<const uint4*>(g);
    const uint4* br = reinterpret_cast<const uint4*>(b);
#pragma unroll
    for (int i = 0; i < kLnMaxVec; ++i) {
        const int c = threadIdx.x + i * kLnThreads;
        if (c < nvec) {
            const uint4 graw = gr[c], braw = br[c];
            const __half2* xh = reinterpret_cast<const __half2*>(&raw[i]);
            const __half2* gh = reinterpret_cast<const __half2*>(&graw);
            const __half2* bh = reinterpret_cast<const __half2*>(&braw);
            uint4 out;
            __half2* oh = reinterpret_cast<__half2*>(&out);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 xf = __half22float2(xh[j]);
                const float2 gf = __half22float2(gh[j]);
                const float2 bf = __half22float2(bh[j]);
                const float a0 = __fadd_rn(__fmul_rn(__fdiv_rn(__fsub_rn(xf.x, mean), denom), gf.x), bf.x);
                const float a1 = __fadd_rn(__fmul_rn(__fdiv_rn(__fsub_rn(xf.y, mean), denom), gf.y), bf.y);
                oh[j] = __halves2half2(__float2half_rn(a0), __float2half_rn(a1));
            }
            yr[c] = out;
        }
    }
}

// y[r] = e_tok[ids[r]] + e_pos[p]  (fp32 add, one rounding), with
// p = max(pos0 + r % T - pad[r / T], 0): the position counted from the
// sequence's first real slot under left padding (pad NULL: no padding).
__global__ void __launch_bounds__(256) embed_kernel(const int32_t* __restrict__ ids, int64_t ntok,
                                                    int32_t T, int32_t pos0,
                                                    const int32_t* __restrict__ pad,
                                                    const __half* __restrict__ e_tok,
                                                    const __half* __restrict__ e_pos, int32_t h1,
                                                    __half* __restrict__ y) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    fgd::griddep_wait();
    fgd::griddep_launch();
    const int64_t nvec = static_cast<int64_t>(h1) / 8;
    const int64_t total = ntok * nvec;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / nvec, c = i % nvec;
        const int64_t id = ids[r];
        const int64_t p0 = pad ? max(pad[r / T], 0) : 0;
        const int64_t p = max(pos0 + r % T - p0, static_cast<int64_t>(0));
        const uint4 a = reinterpret_cast<const uint4*>(e_tok + id * h1)[c];
        const uint4 bb = reinterpret_cast<const uint4*>(e_pos + p * h1)[c];
        const __half2* ah = reinterpret_cast<const __half2*>(&a);
        const __half2* bh = reinterpret_cast<const __half2*>(&bb);
        uint4 out;
        __half2* oh = reinterpret_cast<__half2*>(&out);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 af = __half22float2(ah[j]);
            const float2 bf = __half22float2(bh[j]);
            oh[j] = __halves2half2(__float2half_rn(__fadd_rn(af.x, bf.x)),
                                   __float2half_rn(__fadd_rn(af.y, bf.y)));
        }
        reinterpret_cast<uint4*>(y + r * h1)[c] = out;
    }
}

// Greedy choice per row of fp32 logits: the index of the largest value, the
// lowest such index among equal values (so the result does not depend on
// the reduction order).  One CTA per row.
constexpr int kArgThreads = 512;

struct ValIdx {
    float v;
    int32_t i;
};
__device__ __forceinline__ ValIdx better(ValIdx a, ValIdx b) {
    return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

__global__ void __launch_bounds__(kArgThreads) argmax_kernel(const float* __restrict__ logits,
                                                             int64_t V, int32_t* __restrict__ out) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    fgd::griddep_wait();
    fgd::griddep_launch();
    __shared__ ValIdx red[kArgThreads / 32];
    const float* row = logits + static_cast<int64_t>(blockIdx.x) * V;
    ValIdx best{-CUDART_INF_F, 0x7fffffff};
    // 4 independent loads in flight per thread; indices rise within a thread
    int64_t j = threadIdx.x;
    for (; j + 3 * kArgThreads < V; j += 4 * kArgThreads) {
        const float a = row[j], b = row[j + kArgThreads], c = row[j + 2 * kArgThreads],
                    d = row[j + 3 * kArgThreads];
        best = better(best, ValIdx{a, static_cast<int32_t>(j)});
        best = better(best, ValIdx{b, static_cast<int32_t>(j + kArgThreads)});
        best = better(best, ValIdx{c, static_cast<int32_t>(j + 2 * kArgThreads)});
        best = better(best, ValIdx{d, static_cast<int32_t>(j + 3 * kArgThreads)});
    }
    for (; j < V; j += kArgThreads) best = better(best, ValIdx{row[j], static_cast<int32_t>(j)});
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const ValIdx other{__shfl_xor_sync(0xffffffffu, best.v, o),
                           __shfl_xor_sync(0xffffffffu, best.i, o)};
        best = better(best, other);
    }
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        ValIdx r = red[0];
#pragma unroll
        for (int i = 1; i < kArgThreads / 32; ++i) r = better(r, red[i]);
        // a row of -inf only (never for finite logits) still yields index 0
        out[blockIdx.x] = r.i == 0x7fffffff ? 0 : r.i;
    }
}

}  // namespace

namespace fg {

fg_status launch_layernorm(const __half* x, int64_t rows, int64_t cols, int64_t x_ld,
                           const __half* g, const __half* b, float eps, __half* y,
                           cudaStream_t st) {
    if (rows == 0) return FG_OK;
    if (cols > static_cast<int64_t>(kLnMaxVec) * 8 * kLnThreads)
        return set_error(FG_ERR_UNSUPPORTED, "layernorm: cols %lld > %d", (long long)cols,
                         kLnMaxVec * 8 * kLnThreads);
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, rows * cols * 4.0);
    {
        const cudaError_t le_ = fg::launch_pdl(layernorm_kernel, dim3(static_cast<unsigned>(rows)), dim3(kLnThreads), 0, st,
            x, cols, x_ld, g, b, eps, y);
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "layernorm_kernel launch");
    }
    return cuda_error(cudaGetLastError(), "layernorm launch");
}

fg_status launch_embed(const int32_t* ids, int64_t ntok, int32_t T, int32_t pos0,
                       const int32_t* pad, const __half* e_tok, const __half* e_pos, int32_t h1,
                       __half* y, cudaStream_t st) {
    if (ntok == 0) return FG_OK;
    int64_t blocks = cdiv(ntok * (h1 / 8), 256);
    if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, ntok * h1 * 6.0);
    {
        const cudaError_t le_ = fg::launch_pdl(embed_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
            ids, ntok, T, pos0, pad, e_tok, e_pos, h1, y);
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "embed_kernel launch");
    }
    return cuda_error(cudaGetLastError(), "embed launch");
}

fg_status launch_argmax(const float* logits, int64_t B, int64_t V, int32_t* out, cudaStream_t st) {
    if (B == 0) return FG_OK;
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, B * V * 4.0 + B * 4.0);
    {
        const cudaError_t le_ = fg::launch_pdl(argmax_kernel, dim3(static_cast<unsigned>(B)), dim3(kArgThreads), 0, st,
            logits, V, out);
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "argmax_kernel launch");
    }
    return cuda_error(cudaGetLastError(), "argmax launch");
}

}  // namespace fg
