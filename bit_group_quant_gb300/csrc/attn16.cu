// attn16.cu -- the uncompressed (fp16) KV cache: prefill store and decode
// attention with the new row's append fused in.
//
// This is the setting the pages compare the 4-bit cache against ("FlexGen 完全
// 拆解", results for input length 512: FlexGen with and without 4-bit
// compression): the same decoder, the K/V rows kept as the QKV projection
// made them.  The decode attention is a stream over 2 * L rows of d fp16 per
// (sequence, head), 2 * 256 B per key at d = 128 -- four times the 4-bit
// cache's bytes -- with a dot product and an axpy per row: HBM-bound, so the
// rows go through shared memory by bulk copies and the arithmetic is plain
// fp32 FMA.

#include <math_constants.h>

#include <algorithm>

#include "fg_internal.cuh"

namespace {

using namespace fgd;

// ---------------------------------------------------------------------------
// Store: token t of sequence b (qkv row b*T + t) -> slot slot0 + t, k and v
// of every head copied as 16-byte vectors.
// ---------------------------------------------------------------------------
__global__ void kv_store_f16_kernel(const __half* __restrict__ qkv, int64_t ld, int32_t T,
                                    int32_t H, int32_t d, int32_t cap, int32_t slot0,
                                    __half* __restrict__ k, __half* __restrict__ v,
                                    int64_t nvec) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    griddep_wait();
    griddep_launch();
    // vector i: row r = i / (2 h1 / 8), then k/v and the 8 values within
    const int64_t h1 = static_cast<int64_t>(H) * d;
    const int64_t per_row = 2 * h1 / 8;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nvec;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / per_row, w = i % per_row;
        const int is_v = w >= h1 / 8;
        const int64_t e = (w - (is_v ? h1 / 8 : 0)) * 8;   // element within k (or v)
        const int64_t b = r / T, t = r % T;
        const int64_t hh = e / d, di = e % d;
        const uint4 val = *reinterpret_cast<const uint4*>(qkv + r * ld + (1 + is_v) * h1 + e);
        __half* dst = (is_v ? v : k) + (((b * H + hh) * cap) + slot0 + t) * d + di;
        *reinterpret_cast<uint4*>(dst) = val;
    }
}

// ---------------------------------------------------------------------------
// Decode attention over the fp16 cache.  One CTA (4 warps) per (head,
// sequence).  For the L attended rows the K region and then the V region
// (each contiguous) are fetched in chunks of kCK rows by 1-D bulk copies into
// a ring of kNB buffers; thread 0 refills a buffer after the block barrier
// that ends its use, and every wait is bounded.  Pass 1: lanes take 16-byte
// pieces of a row (D / 8 lanes per row), a dot product with q in fp32 and a
// shuffle reduction give each score; then the exact maximum and
// p_j = exp(s_j - max).  Pass 2: each lane accumulates p_j v_j over its 8
// dimensions; the warps' partial sums meet in shared memory.
// ---------------------------------------------------------------------------
constexpr int kThreads = 128;
constexpr int kNW = kThreads / 32;
constexpr int kCK = 64;   // rows per chunk
constexpr int kNB = 3;    // chunk buffers

__device__ __forceinline__ void h8_to_f(const uint4& raw, float (&f)[8]) {
    const __half2* hh = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 x = __half22float2(hh[i]);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads) decode_attn_f16_kernel(
    const __half* __restrict__ qkv, int64_t ld, int32_t H, int32_t cap, int32_t pos,
    const int32_t* __restrict__ pad, int32_t fuse_append, __half* kc, __half* vc,
    __half* __restrict__ out, int* status, unsigned long long wait_ns) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    griddep_wait();
    griddep_launch();
    constexpr int LPR = D / 8;          // lanes per row
    constexpr int RPI = 32 / LPR;       // rows per warp per step
    constexpr int RB = D * 2;           // bytes per row
    constexpr int CB = kCK * RB;        // bytes per chunk
    extern __shared__ __align__(128) uint8_t dyn[];
    __shared__ __align__(8) uint64_t full_bar[kNB];
    __shared__ float red[kNW];
    __shared__ float part[kNW][RPI][D];
    __shared__ int fail_sh;

    const int h = blockIdx.x, b = blockIdx.y;
    // attended slots p0..pos (a padding count outside [0, pos] is clamped)
    const int p0 = pad ? min(max(pad[b], 0), pos) : 0;
    const int L = pos + 1 - p0;
    const int nK = (L + kCK - 1) / kCK;
    const int nseq = 2 * nK;   // K chunks, then V chunks
    const int64_t h1 = static_cast<int64_t>(H) * D;
    const int64_t rowb = (static_cast<int64_t>(b) * H + h) * cap;   // cache row of slot 0
    const int64_t row0 = rowb + p0;                                  // first attended row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LPR, piece = lane % LPR;   // row within the step, 16-B piece
    const uint32_t ring = smem_u32(dyn);
    float* sc = reinterpret_cast<float*>(dyn + kNB * CB);

    if (fuse_append && warp == 0) {
        // the new k and v rows, D / 8 vectors each, into slot pos
        for (int i = lane; i < 2 * (D / 8); i += 32) {
            const int is_v = i >= D / 8, c = i - (is_v ? D / 8 : 0);
            const uint4 val = *reinterpret_cast<const uint4*>(
                qkv + b * ld + (1 + is_v) * h1 + static_cast<int64_t>(h) * D + c * 8);
            *reinterpret_cast<uint4*>((is_v ? vc : kc) + (rowb + pos) * D + c * 8) = val;
        }
        // the appended rows are read back below by bulk copies (async proxy)
        fence_proxy_async_global();
    }
    float q[8];
    h8_to_f(*reinterpret_cast<const uint4*>(qkv + b * ld + static_cast<int64_t>(h) * D + piece * 8), q);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNB; ++i) mbar_init(smem_u32(&full_bar[i]), 1);
        fence_mbar_init();
        fail_sh = 0;
    }
    __syncthreads();

    auto chunk_n = [&](int c) { return min(kCK, L - c * kCK); };
    auto issue = [&](int seq) {
        const bool is_v = seq >= nK;
        const int c = is_v ? seq - nK : seq;
        const int n = chunk_n(c);
        const int slot = seq % kNB;
        const uint32_t bar = smem_u32(&full_bar[slot]);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * RB));
        bulk_load(ring + slot * CB, (is_v ? vc : kc) + (row0 + c * kCK) * D, n * RB, bar);
    };
    int issued_hi = -1;   // thread 0: highest chunk seq issued so far
    if (threadIdx.x == 0)
        for (int i = 0; i < kNB && i < nseq; ++i) issue(issued_hi = i);
    // bounded wait for chunk seq, made uniform over the warp (pass 1
    // shuffles across the warp); a warp that gives up raises fail_sh, read
    // by every thread after the barrier that ends the chunk
    auto wait_chunk = [&](int seq) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full_bar[seq % kNB]),
                                                          (seq / kNB) & 1, nullptr, wait_ns));
        if (!ok && lane == 0) fail_sh = 1;
        return ok;
    };
    bool failed = false;
    const float attn_scale = __fdiv_rn(1.0f, __fsqrt_rn(static_cast<float>(D)));

    // ---------------- pass 1: scores
    float lmax = -CUDART_INF_F;
    for (int c = 0; c < nK; ++c) {
        const bool ok = wait_chunk(c);
        const uint8_t* buf = dyn + (c % kNB) * CB;
        const int n = ok ? chunk_n(c) : 0;
        for (int rb = warp * RPI; rb < n; rb += kNW * RPI) {   // warp-uniform
            const int r = rb + sub;
            float dot = 0.0f;
            if (r < n) {
                float kv[8];
                h8_to_f(*reinterpret_cast<const uint4*>(buf + r * RB + piece * 16), kv);
#pragma unroll
                for (int i = 0; i < 8; ++i) dot = fmaf(q[i], kv[i], dot);
            }
#pragma unroll
            for (int o = 1; o < LPR; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            if (r < n && piece == 0) {
                const float s = dot * attn_scale;
                sc[c * kCK + r] = s;
                lmax = fmaxf(lmax, s);
            }
        }
        __syncthreads();   // buffer c % kNB is free; fail_sh visible
        if (fail_sh) {
            failed = true;
            break;
        }
        if (threadIdx.x == 0 && c + kNB < nseq) issue(issued_hi = c + kNB);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    if (lane == 0) red[warp] = lmax;
    __syncthreads();
    float mx = red[0];
#pragma unroll
    for (int i = 1; i < kNW; ++i) mx = fmaxf(mx, red[i]);
    __syncthreads();
    float lsum = 0.0f;
    if (!failed) {
        for (int j = threadIdx.x; j < L; j += kThreads) {
            const float p = expf(sc[j] - mx);
            sc[j] = p;
            lsum += p;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    if (lane == 0) red[warp] = lsum;
    __syncthreads();
    float l = 0.0f;
#pragma unroll
    for (int i = 0; i < kNW; ++i) l += red[i];

    // ---------------- pass 2: sum_j p_j v_j over this lane's 8 dimensions
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int c = 0; c < nK && !failed; ++c) {
        const int seq = nK + c;
        const bool ok = wait_chunk(seq);
        const uint8_t* buf = dyn + (seq % kNB) * CB;
        const int n = ok ? chunk_n(c) : 0;
        for (int r = warp * RPI + sub; r < n; r += kNW * RPI) {
            const float p = sc[c * kCK + r];
            float vv[8];
            h8_to_f(*reinterpret_cast<const uint4*>(buf + r * RB + piece * 16), vv);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vv[i], acc[i]);
        }
        __syncthreads();   // buffer free; fail_sh visible
        if (fail_sh) {
            failed = true;
            break;
        }
        if (threadIdx.x == 0 && seq + kNB < nseq) issue(issued_hi = seq + kNB);
    }
    if (failed) {
        // no copy may land after the block leaves: wait (bounded) for every
        // buffer's last issued chunk, then report
        if (threadIdx.x == 0) {
            for (int i = 0; i < kNB && i <= issued_hi; ++i) {
                const int last = i + ((issued_hi - i) / kNB) * kNB;   // last chunk issued to buffer i
                mbar_wait(smem_u32(&full_bar[i]), (last / kNB) & 1, nullptr, wait_ns);
            }
            report(status, fg::kDevTimeout);
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) part[warp][sub][piece * 8 + i] = acc[i];
    __syncthreads();
    for (int i = threadIdx.x; i < D; i += kThreads) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kNW; ++w)
#pragma unroll
            for (int r = 0; r < RPI; ++r) s += part[w][r][i];
        out[b * h1 + static_cast<int64_t>(h) * D + i] = __float2half_rn(s / l);
    }
}

}  // namespace

namespace fg {

fg_status launch_kv_store_f16(const __half* qkv, int64_t ld, int32_t T, const fg_kv16* c,
                              int32_t slot0, cudaStream_t st) {
    const int64_t nvec = static_cast<int64_t>(c->B) * T * 2 * c->H * c->d / 8;
    if (nvec == 0) return FG_OK;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>(cdiv(nvec, threads), 64LL * num_sms());
    TraceScope ts(FG_TRACE_OTHER, st, 0.0, 2.0 * nvec * 16);
    {
        const cudaError_t le_ = fg::launch_pdl(kv_store_f16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st,
            qkv, ld, T, c->H, c->d, c->cap, slot0, reinterpret_cast<__half*>(c->k), reinterpret_cast<__half*>(c->v), nvec);
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "kv_store_f16_kernel launch");
    }
    return cuda_error(cudaGetLastError(), "kv_store_f16 launch");
}

template <int D>
static fg_status launch_decode_f16_t(const __half* qkv, int64_t ld, const fg_kv16* c, int32_t pos,
                                     const int32_t* pad, int32_t fuse_append, __half* out,
                                     cudaStream_t st) {
    const int L = pos + 1;
    const size_t smem = static_cast<size_t>(kNB) * kCK * D * 2 + sizeof(float) * ((L + 3) & ~3);
    if (smem > 220 * 1024)
        return set_error(FG_ERR_UNSUPPORTED, "decode_attn_f16: context %d needs %zu B of shared memory",
                         L, smem);
    auto kern = decode_attn_f16_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_error(e, "decode_attn_f16 smem attribute");
    dim3 grid(c->H, c->B);
    // algorithmic traffic: L fp16 K and V rows per (b, h), the new rows
    // written, q/k/v read, the output written
    const double bh = static_cast<double>(c->B) * c->H;
    TraceScope ts(FG_TRACE_ATTN_DECODE, st, 4.0 * bh * L * D,
                  bh * (2.0 * L * D * 2 + (fuse_append ? 2.0 * D * 2 : 0.0) + 3.0 * D * 2 + D * 2));
    {
        const cudaError_t le_ = fg::launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st,
            qkv, ld, c->H, c->cap, pos, pad, fuse_append,
                                       reinterpret_cast<__half*>(c->k),
                                       reinterpret_cast<__half*>(c->v), out, device_status_ptr(),
                                       wait_limit_ns());
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "kern launch");
    }
    return cuda_error(cudaGetLastError(), "decode_attn_f16 launch");
}

fg_status launch_decode_attn_f16(const __half* qkv, int64_t ld, const fg_kv16* c, int32_t pos,
                                 const int32_t* pad, int32_t fuse_append, __half* out,
                                 cudaStream_t st) {
    if (c->B == 0) return FG_OK;
    if (c->d == 64) return launch_decode_f16_t<64>(qkv, ld, c, pos, pad, fuse_append, out, st);
    return launch_decode_f16_t<128>(qkv, ld, c, pos, pad, fuse_append, out, st);
}

}  // namespace fg
