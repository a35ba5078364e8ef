// attn_tc.cu -- causal prefill attention on the 5th-generation tensor cores.
//
// For every (sequence, head) of the block: out[i] = sum_{j <= i} softmax_j(
// q_i . k_j / sqrt(d)) v_j over the s prompt tokens, from the fp16 q, k, v
// the QKV projection produced ("FlexGen 完全拆解", section
// 从 Transformer 推理的数据流重新定义卸载: the prefill computes Q, K, V of the
// whole prompt and attends causally).
//
// Persistent: two CTAs per SM walk the (128-query block, head, sequence)
// items, the query blocks of each (sequence, head) together and heaviest
// first; a CTA loads the next item's Q while its current item's last P V
// runs.  Per key block of 128:
//   S = Q K^T   tcgen05.mma (M 128 queries, N 128 keys, K = d), Q and K
//               K-major in shared memory (TMA, 128-byte swizzle), S in TMEM;
//   softmax     four warps, one query row per thread (its TMEM lane): the
//               row maximum, p = 2^(s*log2(e)/sqrt(d) - m), the row sum in
//               fp32, p rounded to fp16 and written back into TMEM over S;
//   O += P V    tcgen05.mma with P as the TMEM A operand (M 128, K 128 keys)
//               and V MN-major in shared memory (N = d), O in TMEM.
// The reference maximum m is raised only when a row's block maximum exceeds
// it by more than 2^8 (then O and the row sum are rescaled in TMEM); every
// p stays below 2^8 in fp16 and O and the sum are always relative to the
// same m, so the result is the exact softmax up to the fp16 rounding of the
// p that enter P V (the row sum takes them unrounded, in fp32).
// A left-padded sequence is computed as its real part alone: query and key
// blocks start at its first real slot, so each real row is bit-identical to
// the same prompt run unpadded; the block zeroes its padding rows.
//
// Warp roles (256 threads): warp 0 = TMA producer (Q once; K and V per key
// block, one buffer each); warp 1 = TMEM allocator and the single MMA
// issuer; warps 4-7 = softmax and output (warp w: TMEM lanes 32(w%4)..).
// Every wait is bounded; an expired wait records a timeout in the device
// status word and the CTA drains what it issued and returns.
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "fg_internal.cuh"

namespace {

using namespace fgd;

constexpr int kBQ = 128;                  // queries per CTA (MMA M)
constexpr int kBK = 128;                  // keys per block
constexpr int kThreadsT = 256;
constexpr uint32_t kBoxBytes = 128 * 128; // one TMA box: 128 rows x 64 fp16
constexpr float kRescaleLog2 = 8.0f;      // raise the reference max when exceeded by 2^8
constexpr int kNumBarsT = 10;
// At most two CTAs per SM (each holds 256 TMEM columns): the shared memory
// request is at least this much whatever d is.
constexpr size_t kMinSmemT = 100 * 1024;

template <int D>
constexpr size_t attn_tc_smem() {
    const size_t need = 1024 + 3 * static_cast<size_t>(D / 64) * kBoxBytes + 8 * kNumBarsT + 16;
    return need > kMinSmemT ? need : kMinSmemT;
}

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle:
// 128-byte rows hold 64 consecutive MN elements (one row per k), 8 rows form
// a 1024-byte swizzle atom, consecutive 8-k groups are 1024 bytes apart, and
// the next 64 MN elements start `lbo` bytes further.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(lbo >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}
// Instruction descriptor: fp16 A (K-major) and B (MN-major), fp32 D, M x N.
__device__ __forceinline__ uint32_t idesc_f16_f32_bmn(int M, int N) {
    return (1u << 4) | (1u << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// 32 lanes x 32 bit, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
        "14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// 32 lanes x 32 bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreadsT, 2)
    prefill_attn_tc_kernel(const __grid_constant__ CUtensorMap tm, int32_t s_all, int32_t H,
                           int32_t B, const int32_t* __restrict__ pad, __half* __restrict__ out_all,
                           int* status, unsigned long long wait_ns) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    griddep_wait();
    griddep_launch();
    constexpr int NB = D / 64;                     // 64-dim boxes per tile
    constexpr uint32_t kTile = NB * kBoxBytes;     // bytes of Q, K or V
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sQ = base, sK = base + kTile, sV = base + 2 * kTile;
    const uint32_t bars = base + 3 * kTile;
    const uint32_t q_full = bars, q_empty = bars + 8, k_full = bars + 16, k_empty = bars + 24,
                   v_full = bars + 32, v_empty = bars + 40, s_full = bars + 48,
                   p_full = bars + 56, pv_done = bars + 64, drain = bars + 72;
    uint8_t* const gen = smem_raw - raw;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gen + bars + 8 * kNumBarsT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int64_t h1 = static_cast<int64_t>(H) * D;
    const int nqb = (s_all + kBQ - 1) / kBQ;
    const int nitems = nqb * H * B;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t lim = wait_ns;
    // Work item j -> (query block, head, sequence): the query blocks of one
    // (sequence, head) are consecutive items, heaviest first, so the CTAs
    // that take them at about the same time share that head's K and V
    // through L2 (the grid size is odd, so with a power-of-two block count
    // each CTA's items cycle through every block weight).  The real part of
    // sequence b (s_all - p0 slots from its first real slot p0) and its key
    // blocks.  Every role walks the same items.
    struct Item {
        int qb, h, b, p0, s, q0, nkb, row0;
    };
    auto item_at = [&](int j) {
        Item it;
        const int bh = j / nqb;
        it.qb = nqb - 1 - (j - bh * nqb);
        it.b = bh / H;
        it.h = bh - it.b * H;
        // first real slot (a padding count outside [0, s_all) is clamped)
        it.p0 = pad ? min(max(pad[it.b], 0), s_all - 1) : 0;
        it.s = s_all - it.p0;
        it.q0 = it.qb * kBQ;
        it.nkb = it.qb + 1;                  // key blocks 0..qb (keys past a query masked)
        it.row0 = it.b * s_all + it.p0;      // tensor-map row of the real part's first slot
        return it;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBarsT; ++i)       // p_full: the four softmax warps
            mbar_init(bars + 8u * i, bars + 8u * i == p_full ? 4u : 1u);
        *abort_flag = (status != nullptr && *reinterpret_cast<volatile int*>(status) != 0);
        fence_mbar_init();
        prefetch_tmap(&tm);
    }
    __syncthreads();
    if (*abort_flag) return;           // an earlier wait expired: skip (uniform)
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + 128;    // S (and P over it) and O columns
    auto fail = [&]() {
        *abort_flag = 1;
        report(status, fg::kDevTimeout);
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: per item Q, then K and V of each
            // key block (one buffer each; parities count blocks over items)
            int g = 0, t = 0, kl = -1, vl = -1;
            bool stop = false;
            for (int j = blockIdx.x; j < nitems && !stop; j += gridDim.x) {
                const Item it = item_at(j);
                if (it.q0 >= it.s) continue;
                const int colQ = it.h * D, colK = static_cast<int>(h1) + it.h * D,
                          colV = 2 * static_cast<int>(h1) + it.h * D;
                if (!mbar_wait(q_empty, (t & 1) ^ 1u, abort_flag, lim)) {
                    fail();
                    break;
                }
                mbar_arrive_expect_tx(q_full, kTile);
                for (int x = 0; x < NB; ++x)
                    tma_load_2d(sQ + x * kBoxBytes, &tm, colQ + 64 * x, it.row0 + it.q0, q_full);
                ++t;
                for (int i = 0; i < it.nkb; ++i, ++g) {
                    if (!mbar_wait(k_empty, (g & 1) ^ 1u, abort_flag, lim)) {
                        fail();
                        stop = true;
                        break;
                    }
                    mbar_arrive_expect_tx(k_full, kTile);
                    for (int x = 0; x < NB; ++x)
                        tma_load_2d(sK + x * kBoxBytes, &tm, colK + 64 * x, it.row0 + i * kBK, k_full);
                    kl = g;
                    if (!mbar_wait(v_empty, (g & 1) ^ 1u, abort_flag, lim)) {
                        fail();
                        stop = true;
                        break;
                    }
                    mbar_arrive_expect_tx(v_full, kTile);
                    for (int x = 0; x < NB; ++x)
                        tma_load_2d(sV + x * kBoxBytes, &tm, colV + 64 * x, it.row0 + i * kBK, v_full);
                    vl = g;
                }
            }
            // no copy may land after the CTA leaves: the phase of the last
            // load issued into each buffer
            if (t > 0) mbar_wait(q_full, (t - 1) & 1, nullptr, lim);
            if (kl >= 0) mbar_wait(k_full, kl & 1, nullptr, lim);
            if (vl >= 0) mbar_wait(v_full, vl & 1, nullptr, lim);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (the whole warp loops, lane 0 issues)
        const uint32_t idS = idesc_f16_f32(kBQ, kBK);
        const uint32_t idO = idesc_f16_f32_bmn(kBQ, D);
        bool ok = true;
        int g = 0, t = 0;
        for (int j = blockIdx.x; j < nitems && ok; j += gridDim.x) {
            const Item it = item_at(j);
            if (it.q0 >= it.s) continue;
            ok = __all_sync(0xffffffffu, mbar_wait(q_full, t & 1, abort_flag, lim));
            ++t;
            for (int i = 0; i < it.nkb && ok; ++i, ++g) {
                const uint32_t ph = g & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(k_full, ph, abort_flag, lim));
                // S overwrites the P that the previous P V reads: wait for it
                if (ok && g > 0) ok = __all_sync(0xffffffffu, mbar_wait(pv_done, ph ^ 1u, abort_flag, lim));
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                        mma_f16(tS, sw128_desc(sQ + off), sw128_desc(sK + off), idS, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(k_empty);
                    if (i == it.nkb - 1) mma_commit(q_empty);   // the item's last use of Q
                    mma_commit(s_full);
                }
                __syncwarp();
                ok = __all_sync(0xffffffffu, mbar_wait(p_full, ph, abort_flag, lim));
                if (ok) ok = __all_sync(0xffffffffu, mbar_wait(v_full, ph, abort_flag, lim));
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_f16_ta(tO, tS + 8 * kk, sw128_desc_mn(sV + kk * 2048, kBoxBytes), idO,
                                   (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(v_empty);
                    mma_commit(pv_done);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) fail();
        // every MMA issued completes before TMEM is freed
        if (lane == 0) {
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, lim);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------- softmax and output: thread = query row r of the block
        const int qq = warp & 3;
        const int r = qq * 32 + lane;
        const uint32_t tl = static_cast<uint32_t>(qq * 32) << 16;
        const float sl2 = __fdiv_rn(1.0f, __fsqrt_rn(static_cast<float>(D))) * 1.4426950408889634f;
        bool ok = true;
        int g = 0;
        for (int j = blockIdx.x; j < nitems && ok; j += gridDim.x) {
            const Item it = item_at(j);
            auto out_row = [&](int slot) {
                return out_all + (static_cast<int64_t>(it.b) * s_all + slot) * h1 +
                       static_cast<int64_t>(it.h) * D;
            };
            // padding rows among this block's slots: zeros
            for (int i = r; i < kBQ * (D / 8); i += 128) {
                const int slot = it.qb * kBQ + i / (D / 8);
                if (slot < it.p0)
                    *reinterpret_cast<uint4*>(out_row(slot) + (i % (D / 8)) * 8) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
            if (it.q0 >= it.s) continue;
            const int qi = it.q0 + r;                 // query index in the real part
            float m_ref = -CUDART_INF_F, l = 0.0f;
            for (int i = 0; i < it.nkb; ++i, ++g) {
                if (!__all_sync(0xffffffffu, mbar_wait(s_full, g & 1, abort_flag, lim))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const bool diag = i == it.qb;
                // keys of this block past the query are masked (diagonal block
                // only): columns >= lim_c, set to -inf before use
                const int lim_c = diag ? qi - it.q0 + 1 : kBK;
                // pass 1: the row maximum, two 32-column chunks per TMEM wait,
                // reduced as trees
                float mxa = -CUDART_INF_F, mxb = -CUDART_INF_F;
#pragma unroll 1
                for (int c = 0; c < 4; c += 2) {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tS + tl + 32 * c, v0);
                    tmem_ld32(tS + tl + 32 * c + 32, v1);
                    tmem_wait_ld();
                    float t[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int c0 = 32 * c + jj, c1 = c0 + 16, c2 = c0 + 32, c3 = c0 + 48;
                        const float x0 = c0 < lim_c ? __uint_as_float(v0[jj]) : -CUDART_INF_F;
                        const float x1 = c1 < lim_c ? __uint_as_float(v0[jj + 16]) : -CUDART_INF_F;
                        const float x2 = c2 < lim_c ? __uint_as_float(v1[jj]) : -CUDART_INF_F;
                        const float x3 = c3 < lim_c ? __uint_as_float(v1[jj + 16]) : -CUDART_INF_F;
                        t[jj] = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
                    }
#pragma unroll
                    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
                        for (int jj = 0; jj < w; ++jj) t[jj] = fmaxf(t[jj], t[jj + w]);
                    if (c == 0) mxa = t[0]; else mxb = t[0];
                }
                const float mb = fmaxf(mxa, mxb) * sl2;
                // raise the reference maximum when this block's exceeds it by
                // more than 2^8 (the first block always sets it); O and the
                // row sum are rescaled in TMEM (warp-wide, as TMEM access is)
                const bool raise = mb > m_ref + kRescaleLog2;
                const float m_new = raise ? mb : m_ref;
                if (__any_sync(0xffffffffu, raise) && i > 0) {
                    const float alpha = raise ? ex2(m_ref - m_new) : 1.0f;
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tO + tl + 32 * c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            v[jj] = __float_as_uint(__uint_as_float(v[jj]) * alpha);
                        tmem_st32(tO + tl + 32 * c, v);
                    }
                    l *= alpha;
                }
                m_ref = m_new;
                // pass 2: p = 2^(s sl2 - m) (masked: 2^-inf = 0), written as
                // fp16 pairs over the S columns already read (P of keys 32c..
                // goes to columns 16c..16c+15); the row sum in fp32 over four
                // partial sums
                float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                const float nm = -m_ref;
#pragma unroll 1
                for (int c = 0; c < 4; c += 2) {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tS + tl + 32 * c, v0);
                    tmem_ld32(tS + tl + 32 * c + 32, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const uint32_t(&v)[32] = h2 ? v1 : v0;
                        const int cb = 32 * (c + h2);
                        uint32_t pk[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const float xa = cb + 2 * jj < lim_c ? __uint_as_float(v[2 * jj]) : -CUDART_INF_F;
                            const float xb = cb + 2 * jj + 1 < lim_c ? __uint_as_float(v[2 * jj + 1]) : -CUDART_INF_F;
                            const float pa = ex2(fmaf(xa, sl2, nm));
                            const float pb = ex2(fmaf(xb, sl2, nm));
                            ls[jj & 3] += pa + pb;
                            const __half2 hp = __floats2half2_rn(pa, pb);
                            pk[jj] = *reinterpret_cast<const uint32_t*>(&hp);
                        }
                        tmem_st16(tS + tl + 16 * (c + h2), pk);
                    }
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
            }
            if (!ok) break;
            // output: O / l once the item's last P V has completed
            if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (g - 1) & 1, abort_flag, lim))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv = 1.0f / l;
            __half* orow = out_row(it.p0 + qi);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tO + tl + 32 * c, v);
                tmem_wait_ld();
                if (qi < it.s) {
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 8) {
                        __half2 hh[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            hh[u] = __floats2half2_rn(__uint_as_float(v[jj + 2 * u]) * inv,
                                                      __uint_as_float(v[jj + 2 * u + 1]) * inv);
                        *reinterpret_cast<uint4*>(orow + 32 * c + jj) = *reinterpret_cast<uint4*>(hh);
                    }
                }
            }
            // this thread's O reads are complete before the next item's first
            // P V (ordered through the p_full arrive of that item's block)
            tc_fence_before();
        }
        if (!ok && lane == 0) fail();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

template <int D>
fg_status launch_tc(const CUtensorMap& tm, int32_t B, int32_t s, int32_t H, const int32_t* pad,
                    __half* out, cudaStream_t st) {
    auto kern = prefill_attn_tc_kernel<D>;
    const size_t smem = attn_tc_smem<D>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return fg::cuda_error(e, "prefill_attn_tc smem attribute");
    // persistent: two CTAs per SM (less one, so the count is odd) over all
    // (query block, head, sequence) items
    const int64_t items = fg::cdiv(s, kBQ) * H * static_cast<int64_t>(B);
    int64_t grid = 2 * static_cast<int64_t>(fg::num_sms()) - 1;
    if (grid > items) grid = items;
    {
        const cudaError_t le_ = fg::launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreadsT), smem, st,
            tm, s, H, B, pad, out, fg::device_status_ptr(), fg::wait_limit_ns());
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "kern launch");
    }
    return fg::cuda_error(cudaGetLastError(), "prefill_attn_tc launch");
}

}  // namespace

namespace fg {

bool prefill_attn_tc_supported(int32_t d) { return d == 64 || d == 128; }

fg_status launch_prefill_attn_tc(const __half* qkv, int32_t B, int32_t s, int32_t H, int32_t d,
                                 const int32_t* pad, __half* out, cudaStream_t st) {
    if (B == 0 || s == 0) return FG_OK;
    const int64_t h1 = static_cast<int64_t>(H) * d;
    // q | k | v rows of all sequences: [B * s][3 h1] fp16, boxes of 128 rows x 64 columns
    CUtensorMap tm;
    fg_status r = make_tmap(&tm, qkv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, 3 * h1,
                            static_cast<uint64_t>(B) * s, 64, kBQ, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != FG_OK) return r;
    const double bh = static_cast<double>(B) * H;
    TraceScope ts(FG_TRACE_ATTN_PREFILL, st, 2.0 * bh * s * (s + 1.0) * d, bh * s * d * 2.0 * 4.0);
    return d == 64 ? launch_tc<64>(tm, B, s, H, pad, out, st) : launch_tc<128>(tm, B, s, H, pad, out, st);
}

}  // namespace fg
