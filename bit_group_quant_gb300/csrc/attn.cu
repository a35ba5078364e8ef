// attn.cu -- decode attention over the 4-bit KV cache (with the new token's
// K/V append fused in), its top-K sparse form (a scores pass of the same
// kernels, then one warp per (sequence, head) selecting the kept rows and
// gathering their V), and causal prefill attention.
//
// Dataflow ("FlexGen 完全拆解", section on the inference dataflow): the
// prefill computes Q, K, V for all prompt tokens; each decode step appends
// the new k, v row to the cache and attends the single query over the s+t
// cached rows.  Stored 4-bit tensors are dequantised to FP16 before use
// (section on compression), so every cached row -- the new one included --
// is read back through dequantisation.
//
// Left padding (prompts of different lengths in one block): sequence b's
// tokens occupy slots pad[b].. of its rows; every query attends only keys at
// slots >= pad[b], and prefill queries in padding slots output zeros.  With
// pad NULL every sequence starts at slot 0.
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

// ---------------------------------------------------------------------------
// Decode attention over the 4-bit cache.
//
// For a cached row with codes c, group min m and scale s (per 64 dims):
//   q . k^  = sum_g [ m_g * Q_g + s_g * sum_{i in g} q_i c_i ],  Q_g = sum_{i in g} q_i
//   sum_j p_j v^_j[i] = sum_j p_j m_{j,g} + sum_j (p_j s_{j,g}) c_{j,i}
// so (min, scale) apply once per key and group, and the code dot products run
// on the tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate) with the
// codes masked in place as fp16 subnormals c * 2^-24 (16 c * 2^-24 for odd
// nibble pairs, compensated by q / 16 in the other operand or by 1/16 at the
// end): one AND per pair of codes, and sum x c = 2^24 times the MMA sum, with
// no offset term whose cancellation the tensor cores' accumulation would
// blur.
//
// One CTA (4 warps) per (head, sequence); warps take 16-key tiles in turn.
// Pass 1: scores of all L keys into shared memory.  Then the exact maximum
// and p_j = exp(score_j - max).  Pass 2: the V sums.  K and V are each read
// once from HBM (16-byte / 32-byte coalesced lane loads).
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// half2 codes of nibble pair (p, p+4) of word w in the staged kernel's
// encoding: masked in place as fp16 subnormals, c * 2^-24 for even p and
// 16 c * 2^-24 for odd p (p = 2, 3 read from w >> 8) -- one AND per pair
// plus one shift per word.  No offset term: the tensor cores sum the
// products q * c * 2^-24 without a large common part to cancel.
__device__ __forceinline__ uint32_t enc_pair(uint32_t w, uint32_t w8, int p) {
    const uint32_t src = p < 2 ? w : w8;
    return src & ((p & 1) ? 0x00F000F0u : 0x000F000Fu);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t ldg32(const uint8_t* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}

// ---------------------------------------------------------------------------
// Top-K sparse decode attention ("FlexGen 完全拆解", section on the paper's
// further approximations): the scores of every cached key are computed, and
// only the V rows of the keep_pct percent highest scores are loaded.  The
// softmax keeps its full maximum and normaliser over all attended rows; rows
// not kept add nothing.  ceil(L * keep_pct / 100) rows are kept, equal
// scores lowest slot first.
// ---------------------------------------------------------------------------

__device__ __forceinline__ int topk_count(int L, int keep_pct) {
    return static_cast<int>((static_cast<int64_t>(L) * keep_pct + 99) / 100);
}

// Order-preserving unsigned key of an fp32 score: a larger score has a larger
// key, and -0 and +0 (canonicalised by the addition) share one key.
__device__ __forceinline__ uint32_t score_key(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Candidate keys a warp ranks exactly (the scores of the cut bin).
constexpr int kTkCand = 128;

// Bin of a score in 256 equal bins over [mn, mx] (inv = 256 / (mx - mn)):
// each step is monotone in s, so a higher bin holds only higher scores.
__device__ __forceinline__ uint32_t tk_bin(float s, float mn, float inv) {
    return static_cast<uint32_t>(min(max(static_cast<int>((s - mn) * inv), 0), 255));
}

// Warp-wide: the highest digit d of the 256-bin histogram hc with
// #(keys above d) < need <= #(d and above); every lane gets d and
// #(above d).  Lane l reads bins 255 - 8l down to 248 - 8l.
__device__ __forceinline__ void tk_scan(const uint32_t* hc, uint32_t need, int lane,
                                        uint32_t& digit, uint32_t& above) {
    uint32_t c[8], cnt = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        c[i] = hc[255 - 8 * lane - i];
        cnt += c[i];
    }
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - cnt;
    const bool mine = excl < need && need <= incl;   // exactly one lane
    uint32_t d = 0u, a = 0u, acc = excl;
    if (mine) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (acc + c[i] >= need) {
                d = 255 - 8 * lane - i;
                a = acc;
                break;
            }
            acc += c[i];
        }
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    digit = __shfl_sync(0xffffffffu, d, src);
    above = __shfl_sync(0xffffffffu, a, src);
}

// Asynchronous 16- and 8-byte global -> shared copies (cp.async), completed
// together by cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void tk_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void tk_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

constexpr int kTkChunk = 32;   // kept rows per buffer of the gather (two buffers)

// Shared space of topk_gather_kernel (one warp per block): the scores, two
// buffers of kTkChunk kept rows (codes then (min, scale)), the histogram,
// candidate keys and slots, the chosen candidates, the surely kept slots and
// the merged kept list.
template <int D>
__host__ __device__ constexpr int tk_row_bytes() {
    return D == 128 ? 80 : 48;   // d/2 code bytes + d/64 (min, scale) pairs, 16-byte multiple
}
template <int D>
__host__ __device__ constexpr int tk_smem_bytes(int Lp, int kp) {
    return 4 * Lp + 2 * kTkChunk * tk_row_bytes<D>() + 256 * 4 + 3 * kTkCand * 4 + 2 * 4 * kp;
}

// One warp: the ksel highest of the L scores sc[0..L) (shared; equal
// scores: lower index first) as ascending indices sel[0..ksel).  mx / mn:
// the scores' maximum and minimum.  Usual path: a histogram over 256 equal
// bins of [mn, mx] gives the cut bin; every index in a higher bin is kept
// (list a, ascending) and the cut bin's scores (at most kTkCand, in index
// order) are ranked exactly, the chosen ones forming list b; the two lists
// are merged by rank.  Otherwise (a crowded bin, or all scores equal) a radix
// selection finds the cut key in four 8-bit digit passes and one pass in
// index order keeps every key above it and the first `need` equal to it.
__device__ void warp_topk_select(const float* sc, int L, int ksel, float mx, float mn, int* sel,
                                 uint32_t* hist, uint32_t* ckey, int* cidx, int* lb, int* la,
                                 int lane) {
    const uint32_t lt = (1u << lane) - 1u;
    if (ksel >= L) {
        for (int j = lane; j < L; j += 32) sel[j] = j;
        __syncwarp();
        return;
    }
    const float inv = 256.0f / (mx - mn);
    if (mx > mn && inv < CUDART_INF_F) {
        for (int i = lane; i < 256; i += 32) hist[i] = 0u;
        __syncwarp();
        for (int j = lane; j < L; j += 32) atomicAdd(&hist[tk_bin(sc[j], mn, inv)], 1u);
        __syncwarp();
        uint32_t bstar, above;
        tk_scan(hist, static_cast<uint32_t>(ksel), lane, bstar, above);
        const int need_b = ksel - static_cast<int>(above);   // kept from the cut bin, >= 1
        // the surely kept (list a) and the cut bin's candidates, in index order
        int na = 0, nc = 0;
        for (int c0 = 0; c0 < L; c0 += 32) {
            const int j = c0 + lane;
            const float sj = j < L ? sc[j] : 0.0f;
            const uint32_t bin = j < L ? tk_bin(sj, mn, inv) : 0u;
            const bool sure = j < L && bin > bstar, cut = j < L && bin == bstar;
            const unsigned bs = __ballot_sync(0xffffffffu, sure), bc = __ballot_sync(0xffffffffu, cut);
            if (sure) la[na + __popc(bs & lt)] = j;
            const int at = nc + __popc(bc & lt);
            if (cut && at < kTkCand) {
                ckey[at] = score_key(sj);
                cidx[at] = j;
            }
            na += __popc(bs);
            nc += __popc(bc);
        }
        __syncwarp();
        if (nc <= kTkCand) {
            // the need_b-th highest candidate key T, then the chosen ones in
            // index order: keys above T, and the first (need_b - #above) equal
            uint32_t t_key = 0u, t_gt = 0u;
            bool has = false;
            for (int i = lane; i < nc; i += 32) {
                const uint32_t ki = ckey[i];
                uint32_t gt = 0u, ge = 0u;
                for (int m = 0; m < nc; ++m) {
                    const uint32_t km = ckey[m];
                    gt += km > ki;
                    ge += km >= ki;
                }
                if (gt < static_cast<uint32_t>(need_b) && static_cast<uint32_t>(need_b) <= ge) {
                    t_key = ki;
                    t_gt = gt;
                    has = true;
                }
            }
            const int src = __ffs(__ballot_sync(0xffffffffu, has)) - 1;
            const uint32_t T = __shfl_sync(0xffffffffu, t_key, src);
            const int need_t = need_b - static_cast<int>(__shfl_sync(0xffffffffu, t_gt, src));
            int nb = 0, eq_seen = 0;
            for (int c0 = 0; c0 < nc; c0 += 32) {
                const int i = c0 + lane;
                const uint32_t k = i < nc ? ckey[i] : 0u;
                const bool eq = i < nc && k == T;
                const unsigned beq = __ballot_sync(0xffffffffu, eq);
                const bool take = (i < nc && k > T) || (eq && eq_seen + __popc(beq & lt) < need_t);
                const unsigned bt = __ballot_sync(0xffffffffu, take);
                if (take) lb[nb + __popc(bt & lt)] = cidx[i];
                nb += __popc(bt);
                eq_seen += __popc(beq);
            }
            __syncwarp();
            // merge the ascending lists a (na) and b (nb = need_b) by rank
            auto rank = [](const int* list, int n, int x) {   // #elements < x
                int lo = 0, hi = n;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (list[mid] < x) lo = mid + 1; else hi = mid;
                }
                return lo;
            };
            for (int i = lane; i < na; i += 32) sel[i + rank(lb, nb, la[i])] = la[i];
            for (int i = lane; i < nb; i += 32) sel[i + rank(la, na, lb[i])] = lb[i];
            __syncwarp();
            return;
        }
    }
    // radix selection on the keys
    uint32_t prefix = 0u, pmask = 0u, need = static_cast<uint32_t>(ksel);
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = lane; i < 256; i += 32) hist[i] = 0u;
        __syncwarp();
        for (int j = lane; j < L; j += 32) {
            const uint32_t k = score_key(sc[j]);
            if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
        }
        __syncwarp();
        uint32_t dig, above;
        tk_scan(hist, need, lane, dig, above);
        __syncwarp();   // hist is cleared next
        prefix |= dig << shift;
        pmask |= 0xFFu << shift;
        need -= above;
    }
    int at = 0, eq_seen = 0;
    for (int c0 = 0; c0 < L; c0 += 32) {
        const int j = c0 + lane;
        const uint32_t k = j < L ? score_key(sc[j]) : 0u;
        const bool eq = j < L && k == prefix;
        const unsigned beq = __ballot_sync(0xffffffffu, eq);
        const bool take = (j < L && k > prefix) ||
                          (eq && static_cast<uint32_t>(eq_seen + __popc(beq & lt)) < need);
        const unsigned bt = __ballot_sync(0xffffffffu, take);
        if (take) sel[at + __popc(bt & lt)] = j;
        at += __popc(bt);
        eq_seen += __popc(beq);
    }
    __syncwarp();
}

// Top-K select-and-gather: one warp (the whole block) per (sequence, head)
// u = blockIdx.x, over the scores and (max, min, normaliser) the scores pass
// of the decode kernel wrote (sc_in [B*H][sc_ld], st_in [B*H][4]).  The
// scores come into shared memory in one round of asynchronous copies; the
// warp picks the kept slots (warp_topk_select); the kept rows' codes and
// (min, scale) stream through two buffers of kTkChunk rows (the next chunk's
// copies in flight while one is summed); out = sum_j p_j v^_j / normaliser
// over them, p_j = exp(s_j - max), v^ = m + c s (unrounded, as the dense
// kernels use it), lane l owning D/32 dimensions.  The V rows of the kept
// slots are the only V bytes read.
template <int D>
__global__ void __launch_bounds__(32) topk_gather_kernel(
    const float* __restrict__ sc_in, const float* __restrict__ st_in, int32_t sc_ld, int32_t H,
    int32_t cap, int32_t pos, const int32_t* __restrict__ pad, int32_t keep_pct, int32_t kmax,
    const uint8_t* __restrict__ v_codes, const float* __restrict__ v_meta,
    __half* __restrict__ out, int32_t* __restrict__ sel_out) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    griddep_wait();
    griddep_launch();
    constexpr int G = D / 64, RB = D / 2, RS = tk_row_bytes<D>(), DPL = D / 32;
    extern __shared__ __align__(128) uint8_t dyn[];
    const int lane = threadIdx.x;
    const int64_t u = blockIdx.x;
    const int b = static_cast<int>(u / H), h = static_cast<int>(u % H);
    const int p0 = pad ? min(max(pad[b], 0), pos) : 0;
    const int L = pos + 1 - p0;
    const int ksel = topk_count(L, keep_pct);
    const int Lp = (pos + 4) & ~3, kp = (kmax + 3) & ~3;
    float* sc = reinterpret_cast<float*>(dyn);
    uint8_t* rows = dyn + 4 * Lp;
    uint32_t* hist = reinterpret_cast<uint32_t*>(rows + 2 * kTkChunk * RS);
    uint32_t* ckey = hist + 256;
    int* cidx = reinterpret_cast<int*>(ckey + kTkCand);
    int* lb = cidx + kTkCand;
    int* la = lb + kTkCand;
    int* sel = la + kp;
    // the scores (sc_ld >= 4 * ceil(L / 4): whole 16-byte pieces stay in the row)
    const float* g = sc_in + u * sc_ld;
    for (int i = lane; 4 * i < L; i += 32) cp_async16(sc + 4 * i, g + 4 * i);
    const float mx = st_in[u * 4], mn = st_in[u * 4 + 1], l = st_in[u * 4 + 2];
    cp_async_wait_all();
    __syncwarp();
    warp_topk_select(sc, L, ksel, mx, mn, sel, hist, ckey, cidx, lb, la, lane);
    if (sel_out)
        for (int r = lane; r < kmax; r += 32) sel_out[u * kmax + r] = r < ksel ? p0 + sel[r] : -1;
    // the kept rows' weights, into list a's space (no longer needed)
    float* w = reinterpret_cast<float*>(la);
    for (int r = lane; r < ksel; r += 32) w[r] = expf(sc[sel[r]] - mx);
    // the kept rows, kTkChunk at a time: RB / 16 code pieces and the
    // (min, scale) pairs per row
    const int64_t row0 = u * cap + p0;
    constexpr int CPR = RB / 16 + 1;
    const int nch = (ksel + kTkChunk - 1) / kTkChunk;
    auto issue = [&](int ci) {
        const int r0 = ci * kTkChunk, n = min(kTkChunk, ksel - r0);
        uint8_t* buf = rows + (ci & 1) * kTkChunk * RS;
        for (int i = lane; i < n * CPR; i += 32) {
            const int r = i / CPR, c = i % CPR;
            const int64_t row = row0 + sel[r0 + r];
            uint8_t* dst = buf + r * RS;
            if (c < RB / 16)
                cp_async16(dst + 16 * c, v_codes + row * RB + 16 * c);
            else if (G == 2)
                cp_async16(dst + RB, v_meta + row * 4);
            else
                cp_async8(dst + RB, v_meta + row * 2);
        }
        tk_commit();
    };
    const int grp = (lane * DPL) / 64;
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.0f;
    issue(0);
    for (int ci = 0; ci < nch; ++ci) {
        if (ci + 1 < nch) {
            issue(ci + 1);      // its buffer was last read by chunk ci - 1
            tk_wait<1>();
        } else {
            tk_wait<0>();
        }
        __syncwarp();
        const uint8_t* buf = rows + (ci & 1) * kTkChunk * RS;
        const int r0 = ci * kTkChunk, n = min(kTkChunk, ksel - r0);
#pragma unroll 4
        for (int r = 0; r < n; ++r) {
            const uint8_t* rr = buf + r * RS;
            const float2 m = *reinterpret_cast<const float2*>(rr + RB + 8 * grp);
            const uint32_t cw = DPL == 4 ? *reinterpret_cast<const uint16_t*>(rr + 2 * lane) : rr[lane];
            const float wr = w[r0 + r];
#pragma unroll
            for (int i = 0; i < DPL; ++i)
                acc[i] = fmaf(wr, fmaf(static_cast<float>((cw >> (4 * i)) & 15u), m.y, m.x), acc[i]);
        }
        __syncwarp();           // this buffer is refilled by chunk ci + 2
    }
    __half* o = out + u * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; i += 2)
        *reinterpret_cast<__half2*>(o + i) = __floats2half2_rn(acc[i] / l, acc[i + 1] / l);
}

// Pass 2 (the V sums) over the nv attended keys read straight from global
// memory: key u is cache row row0 + u with weight p = sc[u].  MMA e (nibble e
// of every code word) has rows = dims (row g: word g, row g+8: word 8+g) and
// k = 16 keys paired in registers; B column n = g holds p * s_g (fp16) for
// group g.
template <int D>
__device__ __forceinline__ void v_pass_global(const float* sc, int nv,
                                              const uint8_t* v_codes, const float* v_meta,
                                              int64_t row0, int warp, int g, int t,
                                              float (&accv)[8][4], float& s_pm) {
    constexpr int G = D / 64, RB = D / 2, NWARP = kDecThreads / 32;
    const bool gown = g < G;
    const int ntile = (nv + 15) >> 4;
    for (int kt = warp; kt < ntile; kt += NWARP) {
        const int j0 = kt * 16;
        const int keys[4] = {j0 + 2 * t, j0 + 2 * t + 1, j0 + 2 * t + 8, j0 + 2 * t + 9};
        int slot[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int uu = min(keys[u], nv - 1);
            slot[u] = uu;
        }
        uint32_t bw[2] = {0u, 0u};
        {
            float pp[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool ok = keys[u] < nv;
                const float p = ok ? sc[slot[u]] : 0.0f;
                float pv = 0.0f;
                if (gown && ok) {
                    const float2 m = *reinterpret_cast<const float2*>(
                        v_meta + ((row0 + slot[u]) * G + g) * 2);
                    pv = p * m.y;
                    s_pm += p * m.x;
                }
                pp[u] = pv;
            }
            bw[0] = pack_h2(pp[0], pp[1]);
            bw[1] = pack_h2(pp[2], pp[3]);
        }
        // code words: word g (dims 8g..8g+7) and, for D = 128, word 8+g
        uint32_t w0[4], w1[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint8_t* r = v_codes + (row0 + slot[u]) * RB;
            w0[u] = ldg32(r + 4 * g);
            w1[u] = (D == 128) ? ldg32(r + 32 + 4 * g) : 0u;
        }
        // (key pair, word) -> PRMT so each 16-bit half holds one key's nibbles
        const uint32_t lo0 = __byte_perm(w0[0], w0[1], 0x5410), hi0 = __byte_perm(w0[0], w0[1], 0x7632);
        const uint32_t lo2 = __byte_perm(w0[2], w0[3], 0x5410), hi2 = __byte_perm(w0[2], w0[3], 0x7632);
        const uint32_t lo1 = __byte_perm(w1[0], w1[1], 0x5410), hi1 = __byte_perm(w1[0], w1[1], 0x7632);
        const uint32_t lo3 = __byte_perm(w1[2], w1[3], 0x5410), hi3 = __byte_perm(w1[2], w1[3], 0x7632);
        const uint32_t lo0s = lo0 >> 8, hi0s = hi0 >> 8, lo1s = lo1 >> 8, hi1s = hi1 >> 8;
        const uint32_t lo2s = lo2 >> 8, hi2s = hi2 >> 8, lo3s = lo3 >> 8, hi3s = hi3 >> 8;
        __syncwarp();   // mma.sync is .aligned: reconverge after the per-key loads above
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int p = e & 3;   // MMA e: codes k_e c 2^-24, k_e = 16 for odd e
            const uint32_t a0 = e < 4 ? enc_pair(lo0, lo0s, p) : enc_pair(hi0, hi0s, p);
            const uint32_t a2 = e < 4 ? enc_pair(lo2, lo2s, p) : enc_pair(hi2, hi2s, p);
            const uint32_t a1 = (D == 128) ? (e < 4 ? enc_pair(lo1, lo1s, p) : enc_pair(hi1, hi1s, p)) : 0u;
            const uint32_t a3 = (D == 128) ? (e < 4 ? enc_pair(lo3, lo3s, p) : enc_pair(hi3, hi3s, p)) : 0u;
            mma16816(accv[e], a0, a1, a2, a3, bw[0], bw[1]);
        }
    }
}

// SCORES: the scores pass of top-K attention -- no V pass; the L scores go
// to sc_out[(b*H + h) * sc_ld ..] and (max, min, normaliser) to
// st_out[(b*H + h) * 4 ..] for topk_gather_kernel.  Dynamic shared memory
// holds the L scores.
template <int D, bool SCORES>
__global__ void __launch_bounds__(kDecThreads) decode_attn_kernel(
    const __half* __restrict__ qkv, int64_t ld, int32_t H, int32_t cap, int32_t pos,
    const int32_t* __restrict__ pad, int32_t fuse_append, uint8_t* k_codes, uint8_t* v_codes,
    float* k_meta, float* v_meta, __half* __restrict__ out, float* __restrict__ sc_out,
    float* __restrict__ st_out, int32_t sc_ld) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    griddep_wait();
    griddep_launch();
    constexpr int G = D / 64;            // groups per head row
    constexpr int RB = D / 2;            // code bytes per row
    constexpr int WPT = D / 32;          // code words per lane per row in pass 1
    constexpr int NX = 2 * WPT;          // pass-1 MMAs per 16 keys
    constexpr int NWARP = kDecThreads / 32;
    extern __shared__ float dsm[];
    __shared__ float qsum[G];
    __shared__ float red[NWARP];
    __shared__ float red_min[NWARP];
    __shared__ float part[NWARP][D];
    __shared__ float part_s[NWARP][2][2];   // per warp, per group: sum p m, sum p'

    const int h = blockIdx.x, b = blockIdx.y;
    // attended slots p0..pos (a padding count outside [0, pos] is clamped)
    const int p0 = pad ? min(max(pad[b], 0), pos) : 0;
    const int L = pos + 1 - p0;
    const int64_t h1 = static_cast<int64_t>(H) * D;
    const int64_t rowb = (static_cast<int64_t>(b) * H + h) * cap;  // cache row of slot 0
    const int64_t row0 = rowb + p0;                                 // first attended row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    float* sc = dsm;

    if (fuse_append && warp == 0) {
        const int grp = lane >> 3, lane8 = lane & 7;
        const bool valid = grp < 2 * G;
        const int is_v = grp / G, gi = grp % G;
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
            const int64_t row = rowb + pos;
            uint8_t* cdst = (is_v ? v_codes : k_codes) + row * RB + gi * 32;
            reinterpret_cast<uint32_t*>(cdst)[lane8] = packed;
            if (lane8 == 0) {
                float* mdst = (is_v ? v_meta : k_meta) + (row * G + gi) * 2;
                *reinterpret_cast<float2*>(mdst) = make_float2(mn, scale);
            }
        }
    }
    const __half* qrow = qkv + b * ld + static_cast<int64_t>(h) * D;
    if (warp == 1) {   // per-group sums of q (fp32)
        float s0 = 0.0f, s1 = 0.0f;
        for (int i = lane; i < D; i += 32) {
            const float qv = __half2float(qrow[i]);
            if (i < 64) s0 += qv; else s1 += qv;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, o);
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        if (lane == 0) {
            qsum[0] = s0;
            if (G > 1) qsum[G - 1] = s1;
        }
    }
    // q as the B operand of the pass-1 MMAs: lane (g, t) owns code words
    // WPT*t .. WPT*t + WPT-1 of a row (dims 8 WPT t ..); MMA x uses word x/2,
    // nibble pairs (2h, 2h+4) and (2h+1, 2h+5) with h = x % 2.  Column n = g of
    // B holds q restricted to group g (columns >= G are zero), so the MMA sums
    // each group separately.
    uint32_t qb[NX][2];
    {
        const int my_grp = (WPT * t * 8) / 64;
        const bool use = g < G && g == my_grp;
#pragma unroll
        for (int x = 0; x < NX; ++x) {
            const int base = 8 * (WPT * t + (x >> 1)) + 2 * (x & 1);
            const float q0 = use ? __half2float(qrow[base]) : 0.0f;
            const float q4 = use ? __half2float(qrow[base + 4]) : 0.0f;
            const float q1 = use ? __half2float(qrow[base + 1]) : 0.0f;
            const float q5 = use ? __half2float(qrow[base + 5]) : 0.0f;
            qb[x][0] = pack_h2(q0, q4);
            qb[x][1] = pack_h2(q1 * 0.0625f, q5 * 0.0625f);   // exact: pairs e+1 carry 16 c
        }
    }
    __syncthreads();

    const float attn_scale = __fdiv_rn(1.0f, __fsqrt_rn(static_cast<float>(D)));
    const float Q0 = qsum[0], Q1 = qsum[G - 1];
    const int ntile = (L + 15) >> 4;

    // ---------------- pass 1: scores
    float lmax = -CUDART_INF_F, lmin = CUDART_INF_F;   // lmin: SCORES only
    for (int kt = warp; kt < ntile; kt += NWARP) {
        const int ja = min(kt * 16 + g, L - 1), jb = min(kt * 16 + g + 8, L - 1);
        const uint8_t* ra = k_codes + (row0 + ja) * RB + t * (WPT * 4);
        const uint8_t* rb = k_codes + (row0 + jb) * RB + t * (WPT * 4);
        uint32_t wa[WPT], wb[WPT];
        if (WPT == 4) {
            const uint4 va = *reinterpret_cast<const uint4*>(ra);
            const uint4 vb = *reinterpret_cast<const uint4*>(rb);
            wa[0] = va.x; wa[1] = va.y; wa[WPT > 2 ? 2 : 0] = va.z; wa[WPT > 3 ? 3 : 0] = va.w;
            wb[0] = vb.x; wb[1] = vb.y; wb[WPT > 2 ? 2 : 0] = vb.z; wb[WPT > 3 ? 3 : 0] = vb.w;
        } else {
            const uint2 va = *reinterpret_cast<const uint2*>(ra);
            const uint2 vb = *reinterpret_cast<const uint2*>(rb);
            wa[0] = va.x; wa[1] = va.y;
            wb[0] = vb.x; wb[1] = vb.y;
        }
        uint32_t wa8[WPT], wb8[WPT];
#pragma unroll
        for (int i = 0; i < WPT; ++i) {
            wa8[i] = wa[i] >> 8;
            wb8[i] = wb[i] >> 8;
        }
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        __syncwarp();   // mma.sync is .aligned: reconverge after last round's lane-0 work
#pragma unroll
        for (int x = 0; x < NX; ++x) {
            const int e = 2 * (x & 1);
            const int wi = x >> 1;
            mma16816(acc, enc_pair(wa[wi], wa8[wi], e), enc_pair(wb[wi], wb8[wi], e),
                     enc_pair(wa[wi], wa8[wi], e + 1), enc_pair(wb[wi], wb8[wi], e + 1),
                     qb[x][0], qb[x][1]);
        }
        if (t == 0) {
            // acc: (key g, group 0), (key g, group 1), (key g+8, group 0), (key g+8, group 1)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int j = kt * 16 + g + 8 * half;
                if (j < L) {
                    const float* km = k_meta + (row0 + j) * G * 2;
                    float dot;
                    // sum q c = 2^24 acc per group
                    if (G == 2) {
                        const float4 m = *reinterpret_cast<const float4*>(km);
                        dot = m.x * Q0 + 16777216.0f * m.y * acc[2 * half] +
                              m.z * Q1 + 16777216.0f * m.w * acc[2 * half + 1];
                    } else {
                        const float2 m = *reinterpret_cast<const float2*>(km);
                        dot = m.x * Q0 + 16777216.0f * m.y * acc[2 * half];
                    }
                    const float s = dot * attn_scale;
                    sc[j] = s;
                    lmax = fmaxf(lmax, s);
                    if (SCORES) lmin = fminf(lmin, s);
                }
            }
        }
    }
    lmax = warp_max(lmax);
    if (lane == 0) red[warp] = lmax;
    if (SCORES) {
        lmin = -warp_max(-lmin);
        if (lane == 0) red_min[warp] = lmin;
    }
    __syncthreads();
    float mx = red[0], mn = SCORES ? red_min[0] : 0.0f;
#pragma unroll
    for (int i = 1; i < NWARP; ++i) {
        mx = fmaxf(mx, red[i]);
        if (SCORES) mn = fminf(mn, red_min[i]);
    }
    __syncthreads();
    float lsum = 0.0f;
    for (int j = threadIdx.x; j < L; j += kDecThreads) {
        const float p = expf(sc[j] - mx);
        if (!SCORES) sc[j] = p;   // the scores pass keeps the scores
        lsum += p;
    }
    lsum = warp_sum(lsum);
    if (lane == 0) red[warp] = lsum;
    __syncthreads();
    float l = 0.0f;
#pragma unroll
    for (int i = 0; i < NWARP; ++i) l += red[i];
    if constexpr (SCORES) {
        const int64_t bh = static_cast<int64_t>(b) * H + h;
        for (int j = threadIdx.x; j < L; j += kDecThreads) sc_out[bh * sc_ld + j] = sc[j];
        if (threadIdx.x == 0) {
            st_out[bh * 4] = mx;
            st_out[bh * 4 + 1] = mn;
            st_out[bh * 4 + 2] = l;
        }
        return;
    }

    // ---------------- pass 2: V
    float accv[8][4];
#pragma unroll
    for (int e = 0; e < 8; ++e) accv[e][0] = accv[e][1] = accv[e][2] = accv[e][3] = 0.0f;
    float s_pm = 0.0f;   // this lane's keys: sum p * min (group g)
    const bool gown = g < G;
    v_pass_global<D>(sc, L, v_codes, v_meta, row0, warp, g, t, accv, s_pm);
    // group sums of this warp: reduce over the 4 lanes (g, t) of each group
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) s_pm += __shfl_xor_sync(0xffffffffu, s_pm, o);
    if (t == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            part[warp][8 * g + e] = accv[e][0];                 // group 0 dims x p'(group 0)
            if (D == 128) part[warp][64 + 8 * g + e] = accv[e][3];  // group 1 dims x p'(group 1)
        }
        if (gown) part_s[warp][g][0] = s_pm;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < D; i += kDecThreads) {
        const int grp = i >> 6;
        float dsum = 0.0f, pm = 0.0f;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) {
            dsum += part[w][i];
            pm += part_s[w][grp][0];
        }
        // dim i comes from MMA e = i % 8: sum (p s) c = 2^24 / k_e acc, k_e = 16 for odd e
        const float kinv = (i & 1) ? 1048576.0f : 16777216.0f;
        const float o = (pm + kinv * dsum) / l;
        out[b * h1 + static_cast<int64_t>(h) * D + i] = __float2half_rn(o);
    }
}

// Decode attention for d = 128 with the cache streamed through shared memory.
// The same per-group algebra as decode_attn_kernel, but the codes enter the
// MMAs as fp16 subnormals c * 2^-24 (one AND per pair of codes, no offset to
// cancel), so sum q c = 2^24 acc and sum (p s) c = 2^24 acc / k.  For one
// (head, sequence) the L cached rows of K codes, K (min, scale), V codes and
// V (min, scale) are four contiguous regions, fetched in chunks of kCK rows by
// 1-D bulk asynchronous copies (the async proxy) into a ring of kNB chunk
// buffers -- K chunks first, then V chunks, so V streams in while the K pass
// computes.  Thread 0 refills a buffer after the block barrier that ends its
// use; every wait on a chunk is bounded.
// 128-key chunks, 2 buffers (23 KB per block) and <= 64 registers give 8
// blocks per SM: with the 2 block barriers per chunk, many resident blocks
// keep more bytes in flight than deeper rings would (measured on GB300:
// 4.1-4.7 TB/s at contexts 513-2049, against 3.5-4.2 with 4 x 128 keys).
constexpr int kCK = 128;           // keys per staged chunk
constexpr int kNB = 2;             // chunk buffers
constexpr int kMinBlocks = 8;      // resident blocks per SM (register cap)
constexpr int kCKMax = kCK + 16;   // the last chunk absorbs a remainder of up to 16 keys
constexpr int kRB128 = 64;         // code bytes per row (d = 128)
constexpr int kMB128 = 16;         // (min, scale) bytes per row (2 groups)
constexpr int kChunkBytes = kCKMax * (kRB128 + kMB128);   // codes, then meta

// SCORES: the scores pass of top-K attention.  Only the K chunks are
// staged; after pass 1 the scores go to sc_out[(b*H + h) * sc_ld ..] and
// (max, min, normaliser) to st_out[(b*H + h) * 4 ..] for topk_gather_kernel,
// and there is no V pass.

template <bool SCORES>
__global__ void __launch_bounds__(kDecThreads, kMinBlocks) decode_attn_staged_kernel(
    const __half* __restrict__ qkv, int64_t ld, int32_t H, int32_t cap, int32_t pos,
    const int32_t* __restrict__ pad, int32_t fuse_append, uint8_t* k_codes, uint8_t* v_codes,
    float* k_meta, float* v_meta, __half* __restrict__ out, int* status,
    unsigned long long wait_ns, float* __restrict__ sc_out, float* __restrict__ st_out,
    int32_t sc_ld) {
    // the inputs come from earlier kernels of the stream (this launch may
    // start before they finish): wait for them, then let the next kernel be
    // scheduled
    griddep_wait();
    griddep_launch();
    constexpr int D = 128, G = 2, RB = kRB128, WPT = D / 32, NX = 2 * WPT;
    constexpr int NWARP = kDecThreads / 32;
    extern __shared__ __align__(128) uint8_t dyn[];
    __shared__ __align__(8) uint64_t full_bar[kNB];
    __shared__ float qsum[G];
    __shared__ float red[NWARP];
    __shared__ float red_min[NWARP];
    __shared__ float part[NWARP][D];
    __shared__ float part_s[NWARP][2][2];
    __shared__ int fail_sh;

    const int h = blockIdx.x, b = blockIdx.y;
    // attended slots p0..pos (a padding count outside [0, pos] is clamped)
    const int p0 = pad ? min(max(pad[b], 0), pos) : 0;
    const int L = pos + 1 - p0;
    // chunks of kCK keys; a remainder of <= 16 keys joins the last full chunk
    int nK = (L + kCK - 1) / kCK;
    if (nK > 1 && L - (nK - 1) * kCK <= 16) --nK;
    const int nseq = SCORES ? nK : 2 * nK;   // K chunks, then (dense) V chunks
    auto chunk_n = [&](int c) { return c == nK - 1 ? L - c * kCK : kCK; };
    const int64_t h1 = static_cast<int64_t>(H) * D;
    const int64_t rowb = (static_cast<int64_t>(b) * H + h) * cap;  // cache row of slot 0
    const int64_t row0 = rowb + p0;                                 // first attended row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const uint32_t ring = smem_u32(dyn);
    float* sc = reinterpret_cast<float*>(dyn + kNB * kChunkBytes);

    if (fuse_append && warp == 0) {
        const int grp = lane >> 3, lane8 = lane & 7;
        const bool valid = grp < 2 * G;
        const int is_v = grp / G, gi = grp % G;
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
            const int64_t row = rowb + pos;
            uint8_t* cdst = (is_v ? v_codes : k_codes) + row * RB + gi * 32;
            reinterpret_cast<uint32_t*>(cdst)[lane8] = packed;
            if (lane8 == 0) {
                float* mdst = (is_v ? v_meta : k_meta) + (row * G + gi) * 2;
                *reinterpret_cast<float2*>(mdst) = make_float2(mn, scale);
            }
        }
        // the appended row is read back below by bulk copies (async proxy)
        fence_proxy_async_global();
    }
    const __half* qrow = qkv + b * ld + static_cast<int64_t>(h) * D;
    if (warp == 1) {   // per-group sums of q (fp32)
        float s0 = 0.0f, s1 = 0.0f;
        for (int i = lane; i < D; i += 32) {
            const float qv = __half2float(qrow[i]);
            if (i < 64) s0 += qv; else s1 += qv;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, o);
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        if (lane == 0) {
            qsum[0] = s0;
            qsum[1] = s1;
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNB; ++i) mbar_init(smem_u32(&full_bar[i]), 1);
        fence_mbar_init();
        fail_sh = 0;
    }
    // q as the B operand of the pass-1 MMAs (see decode_attn_kernel)
    uint32_t qb[NX][2];
    {
        const int my_grp = (WPT * t * 8) / 64;
        const bool use = g < G && g == my_grp;
#pragma unroll
        for (int x = 0; x < NX; ++x) {
            const int base = 8 * (WPT * t + (x >> 1)) + 2 * (x & 1);
            const float q0 = use ? __half2float(qrow[base]) : 0.0f;
            const float q4 = use ? __half2float(qrow[base + 4]) : 0.0f;
            const float q1 = use ? __half2float(qrow[base + 1]) : 0.0f;
            const float q5 = use ? __half2float(qrow[base + 5]) : 0.0f;
            qb[x][0] = pack_h2(q0, q4);
            qb[x][1] = pack_h2(q1 * 0.0625f, q5 * 0.0625f);   // exact: pairs e+1 carry 16 c
        }
    }
    __syncthreads();

    // chunk seq: K chunks 0..nK-1, then V chunks; buffer seq % kNB, phase seq / kNB
    auto issue = [&](int seq) {
        const bool is_v = seq >= nK;
        const int c = is_v ? seq - nK : seq;
        const int r0 = c * kCK, n = chunk_n(c);
        const int slot = seq % kNB;
        const uint32_t dst = ring + slot * kChunkBytes;
        const uint32_t bar = smem_u32(&full_bar[slot]);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * (RB + kMB128)));
        bulk_load(dst, (is_v ? v_codes : k_codes) + (row0 + r0) * RB, n * RB, bar);
        bulk_load(dst + kCKMax * RB, (is_v ? v_meta : k_meta) + (row0 + r0) * G * 2, n * kMB128, bar);
    };
    int issued_hi = -1;   // thread 0: highest chunk seq issued so far
    if (threadIdx.x == 0)
        for (int i = 0; i < kNB && i < nseq; ++i) issue(issued_hi = i);
    // Bounded wait for chunk seq, made uniform over the warp (the MMAs are
    // warp-synchronous); a warp that gives up raises fail_sh, which every
    // thread reads after the block barrier that ends the chunk.  One block
    // barrier per chunk: it also frees the buffer for the next copy.
    auto wait_chunk = [&](int seq) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full_bar[seq % kNB]),
                                                          (seq / kNB) & 1, nullptr, wait_ns));
        if (!ok && lane == 0) fail_sh = 1;
        return ok;
    };
    bool failed = false;

    const float attn_scale = __fdiv_rn(1.0f, __fsqrt_rn(static_cast<float>(D)));
    const float Q0 = qsum[0], Q1 = qsum[1];

    // ---------------- pass 1: scores
    float lmax = -CUDART_INF_F, lmin = CUDART_INF_F;   // lmin: SCORES only
    for (int c = 0; c < nK; ++c) {
        const bool ok = wait_chunk(c);
        const uint8_t* buf = dyn + (c % kNB) * kChunkBytes;
        const int r0 = c * kCK, n = chunk_n(c);
        const int ntile = ok ? (n + 15) >> 4 : 0;
        for (int kt = warp; kt < ntile; kt += NWARP) {
            const int ja = min(kt * 16 + g, n - 1), jb = min(kt * 16 + g + 8, n - 1);
            const uint4 va = *reinterpret_cast<const uint4*>(buf + ja * RB + t * 16);
            const uint4 vb = *reinterpret_cast<const uint4*>(buf + jb * RB + t * 16);
            const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
            const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
            uint32_t wa8[4], wb8[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                wa8[i] = wa[i] >> 8;
                wb8[i] = wb[i] >> 8;
            }
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            __syncwarp();
#pragma unroll
            for (int x = 0; x < NX; ++x) {
                const int e = 2 * (x & 1);
                const int wi = x >> 1;
                mma16816(acc, enc_pair(wa[wi], wa8[wi], e), enc_pair(wb[wi], wb8[wi], e),
                         enc_pair(wa[wi], wa8[wi], e + 1), enc_pair(wb[wi], wb8[wi], e + 1),
                         qb[x][0], qb[x][1]);
            }
            if (t == 0) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int jl = kt * 16 + g + 8 * half;
                    if (jl < n) {
                        const float4 m = *reinterpret_cast<const float4*>(buf + kCKMax * RB + jl * kMB128);
                        // sum q c = 2^24 acc per group
                        const float dot = m.x * Q0 + 16777216.0f * m.y * acc[2 * half] +
                                          m.z * Q1 + 16777216.0f * m.w * acc[2 * half + 1];
                        const float s = dot * attn_scale;
                        sc[r0 + jl] = s;
                        lmax = fmaxf(lmax, s);
                        if (SCORES) lmin = fminf(lmin, s);
                    }
                }
            }
        }
        __syncthreads();   // buffer c % kNB is free; fail_sh visible
        if (fail_sh) {
            failed = true;
            break;
        }
        if (threadIdx.x == 0 && c + kNB < nseq) issue(issued_hi = c + kNB);
    }
    lmax = warp_max(lmax);
    if (lane == 0) red[warp] = lmax;
    if (SCORES) {
        lmin = -warp_max(-lmin);
        if (lane == 0) red_min[warp] = lmin;
    }
    __syncthreads();
    float mx = red[0], mn = SCORES ? red_min[0] : 0.0f;
#pragma unroll
    for (int i = 1; i < NWARP; ++i) {
        mx = fmaxf(mx, red[i]);
        if (SCORES) mn = fminf(mn, red_min[i]);
    }
    __syncthreads();
    float lsum = 0.0f;
    if (!failed) {
        for (int j = threadIdx.x; j < L; j += kDecThreads) {
            const float p = expf(sc[j] - mx);
            if (!SCORES) sc[j] = p;   // the scores pass keeps the scores
            lsum += p;
        }
    }
    lsum = warp_sum(lsum);
    if (lane == 0) red[warp] = lsum;
    __syncthreads();
    float l = 0.0f;
#pragma unroll
    for (int i = 0; i < NWARP; ++i) l += red[i];
    if (SCORES && !failed) {   // block-uniform; no chunk is in flight after a clean pass 1
        const int64_t bh = static_cast<int64_t>(b) * H + h;
        for (int j = threadIdx.x; j < L; j += kDecThreads) sc_out[bh * sc_ld + j] = sc[j];
        if (threadIdx.x == 0) {
            st_out[bh * 4] = mx;
            st_out[bh * 4 + 1] = mn;
            st_out[bh * 4 + 2] = l;
        }
        return;
    }

    // ---------------- pass 2: V (see decode_attn_kernel for the MMA layout)
    float accv[8][4];
#pragma unroll
    for (int e = 0; e < 8; ++e) accv[e][0] = accv[e][1] = accv[e][2] = accv[e][3] = 0.0f;
    float s_pm = 0.0f;   // this lane's keys: sum p * min (group g)
    const bool gown = g < G;
    for (int c = 0; c < nK && !failed && !SCORES; ++c) {
        const int seq = nK + c;
        const bool ok = wait_chunk(seq);
        const uint8_t* buf = dyn + (seq % kNB) * kChunkBytes;
        const int r0 = c * kCK, n = chunk_n(c);
        const int ntile = ok ? (n + 15) >> 4 : 0;
        for (int kt = warp; kt < ntile; kt += NWARP) {
            const int j0 = kt * 16;
            // The 16 keys of the tile in any order the P fragment shares: lane t
            // takes keys j0 + t + 4u.  Rows of 64 code bytes put keys two apart
            // in the same bank; keys one apart differ by 16 banks, so the four
            // lanes of a fragment row read at most 2-way conflicting banks (the
            // pairs 2t, 2t + 1, 2t + 8, 2t + 9 were 4-way).
            int keys[4] = {j0 + t, j0 + 4 + t, j0 + 8 + t, j0 + 12 + t};
            uint32_t bw[2];
            {
                float pp[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const bool ok = keys[u] < n;
                    const float p = ok ? sc[r0 + keys[u]] : 0.0f;
                    float pv = 0.0f;
                    if (gown && ok) {
                        const float2 m = *reinterpret_cast<const float2*>(buf + kCKMax * RB + keys[u] * kMB128 + g * 8);
                        pv = p * m.y;
                        s_pm += p * m.x;
                    }
                    pp[u] = pv;
                }
                bw[0] = pack_h2(pp[0], pp[1]);
                bw[1] = pack_h2(pp[2], pp[3]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) keys[u] = min(keys[u], n - 1);
            uint32_t w0[4], w1[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint8_t* r = buf + keys[u] * RB;
                w0[u] = *reinterpret_cast<const uint32_t*>(r + 4 * g);
                w1[u] = *reinterpret_cast<const uint32_t*>(r + 32 + 4 * g);
            }
            const uint32_t lo0 = __byte_perm(w0[0], w0[1], 0x5410), hi0 = __byte_perm(w0[0], w0[1], 0x7632);
            const uint32_t lo2 = __byte_perm(w0[2], w0[3], 0x5410), hi2 = __byte_perm(w0[2], w0[3], 0x7632);
            const uint32_t lo1 = __byte_perm(w1[0], w1[1], 0x5410), hi1 = __byte_perm(w1[0], w1[1], 0x7632);
            const uint32_t lo3 = __byte_perm(w1[2], w1[3], 0x5410), hi3 = __byte_perm(w1[2], w1[3], 0x7632);
            __syncwarp();
            const uint32_t lo0s = lo0 >> 8, hi0s = hi0 >> 8, lo1s = lo1 >> 8, hi1s = hi1 >> 8;
            const uint32_t lo2s = lo2 >> 8, hi2s = hi2 >> 8, lo3s = lo3 >> 8, hi3s = hi3 >> 8;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int p = e & 3;   // MMA e: codes 1 + k_e c 2^-10, k_e = 16 for odd e
                const uint32_t a0 = e < 4 ? enc_pair(lo0, lo0s, p) : enc_pair(hi0, hi0s, p);
                const uint32_t a2 = e < 4 ? enc_pair(lo2, lo2s, p) : enc_pair(hi2, hi2s, p);
                const uint32_t a1 = e < 4 ? enc_pair(lo1, lo1s, p) : enc_pair(hi1, hi1s, p);
                const uint32_t a3 = e < 4 ? enc_pair(lo3, lo3s, p) : enc_pair(hi3, hi3s, p);
                mma16816(accv[e], a0, a1, a2, a3, bw[0], bw[1]);
            }
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
    for (int o = 1; o < 4; o <<= 1) s_pm += __shfl_xor_sync(0xffffffffu, s_pm, o);
    if (t == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            part[warp][8 * g + e] = accv[e][0];
            part[warp][64 + 8 * g + e] = accv[e][3];
        }
        if (gown) part_s[warp][g][0] = s_pm;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < D; i += kDecThreads) {
        const int grp = i >> 6;
        float dsum = 0.0f, pm = 0.0f;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) {
            dsum += part[w][i];
            pm += part_s[w][grp][0];
        }
        // dim i comes from MMA e = i % 8: sum (p s) c = 2^24 / k_e acc, k_e = 16 for odd e
        const float kinv = (i & 1) ? 1048576.0f : 16777216.0f;
        const float o = (pm + kinv * dsum) / l;
        out[b * h1 + static_cast<int64_t>(h) * D + i] = __float2half_rn(o);
    }
}


// Dynamic shared memory a block may use (227 KB less the kernels' static arrays).
constexpr size_t kMaxDynSmem = 220 * 1024;

// Rows kept by top-K attention over L rows (host copy of topk_count).
int topk_count_host(int L, int keep_pct) {
    return static_cast<int>((static_cast<int64_t>(L) * keep_pct + 99) / 100);
}

// Algorithmic bytes of one decode-attention launch: per (b, h) the L packed
// K rows and the V rows summed (all L, or the kept ones), codes + fp32 meta;
// the new k, v written back; q/k/v read and the output written.
double decode_attn_bytes(int D, double bh, int L, int nv, bool fuse_append) {
    const double row = D / 2 + (D / 64) * 8.0;
    return bh * ((static_cast<double>(L) + nv) * row + (fuse_append ? 2.0 * row : 0.0) + 3.0 * D * 2 + D * 2);
}

// Scores workspace of top-K attention: sc [B*H][ld] fp32 (ld = the largest
// L rounded up to 4), then st [B*H][4] fp32 (max, min, normaliser).
struct TopkWs {
    float* sc;
    float* st;
    int sc_ld;
    size_t bytes;
};
TopkWs topk_ws_layout(int32_t B, int32_t H, int32_t pos, void* base) {
    TopkWs w{};
    w.sc_ld = (pos + 4) & ~3;
    const size_t a = (static_cast<size_t>(B) * H * w.sc_ld * 4 + 255) & ~static_cast<size_t>(255);
    w.bytes = a + ((static_cast<size_t>(B) * H * 16 + 255) & ~static_cast<size_t>(255));
    w.sc = static_cast<float*>(base);
    w.st = base ? reinterpret_cast<float*>(static_cast<char*>(base) + a) : nullptr;
    return w;
}

template <int D, bool SCORES>
fg_status launch_decode_t(const __half* qkv, int64_t ld, const fg_kv4* c, int32_t pos,
                          const int32_t* pad, int32_t fuse_append, __half* out, const TopkWs& w,
                          cudaStream_t st) {
    const int L = pos + 1;
    const size_t smem = sizeof(float) * ((L + 3) & ~3);
    if (smem > kMaxDynSmem)
        return fg::set_error(FG_ERR_UNSUPPORTED, "decode_attn: context %d needs %zu B of shared memory",
                             L, smem);
    auto kern = decode_attn_kernel<D, SCORES>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return fg::cuda_error(e, "decode_attn smem attribute");
    }
    dim3 grid(c->H, c->B);
    const double bh = static_cast<double>(c->B) * c->H;
    fg::TraceScope ts(FG_TRACE_ATTN_DECODE, st, (SCORES ? 2.0 : 4.0) * bh * L * D,
                      decode_attn_bytes(D, bh, L, SCORES ? 0 : L, fuse_append != 0));
    {
        const cudaError_t le_ = fg::launch_pdl(kern, dim3(grid), dim3(kDecThreads), smem, st,
            qkv, ld, c->H, c->cap, pos, pad, fuse_append,
                                          c->k_codes, c->v_codes, c->k_meta, c->v_meta, out,
                                          w.sc, w.st, w.sc_ld);
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "kern launch");
    }
    return fg::cuda_error(cudaGetLastError(), "decode_attn launch");
}

template <bool SCORES>
fg_status launch_decode_staged(const __half* qkv, int64_t ld, const fg_kv4* c, int32_t pos,
                               const int32_t* pad, int32_t fuse_append, __half* out,
                               const TopkWs& w, cudaStream_t st) {
    constexpr int D = 128;
    const int L = pos + 1;
    const size_t smem = static_cast<size_t>(kNB) * kChunkBytes + sizeof(float) * ((L + 3) & ~3);
    if (smem > kMaxDynSmem)
        return fg::set_error(FG_ERR_UNSUPPORTED, "decode_attn: context %d needs %zu B of shared memory",
                             L, smem);
    auto kern = decode_attn_staged_kernel<SCORES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return fg::cuda_error(e, "decode_attn smem attribute");
    dim3 grid(c->H, c->B);
    const double bh = static_cast<double>(c->B) * c->H;
    fg::TraceScope ts(FG_TRACE_ATTN_DECODE, st, (SCORES ? 2.0 : 4.0) * bh * L * D,
                      decode_attn_bytes(D, bh, L, SCORES ? 0 : L, fuse_append != 0));
    {
        const cudaError_t le_ = fg::launch_pdl(kern, dim3(grid), dim3(kDecThreads), smem, st,
            qkv, ld, c->H, c->cap, pos, pad, fuse_append,
                                          c->k_codes, c->v_codes, c->k_meta, c->v_meta, out,
                                          fg::device_status_ptr(), fg::wait_limit_ns(), w.sc, w.st,
                                          w.sc_ld);
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "kern launch");
    }
    return fg::cuda_error(cudaGetLastError(), "decode_attn launch");
}

template <int D>
fg_status launch_topk_gather(const fg_kv4* c, int32_t pos, const int32_t* pad, int32_t keep_pct,
                             int32_t kmax, int32_t* sel_out, __half* out, const TopkWs& w,
                             cudaStream_t st) {
    const int Lp = (pos + 4) & ~3, kp = (kmax + 3) & ~3;
    const size_t smem = static_cast<size_t>(tk_smem_bytes<D>(Lp, kp));
    if (smem > kMaxDynSmem)
        return fg::set_error(FG_ERR_UNSUPPORTED,
                             "decode_attn_topk: context %d at keep %d%% needs %zu B of shared memory",
                             pos + 1, keep_pct, smem);
    auto kern = topk_gather_kernel<D>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return fg::cuda_error(e, "topk_gather smem attribute");
    }
    const int64_t units = static_cast<int64_t>(c->B) * c->H;
    const double row = D / 2 + (D / 64) * 8.0;
    fg::TraceScope ts(FG_TRACE_ATTN_DECODE, st, 2.0 * units * kmax * D,
                      static_cast<double>(units) * (kmax * row + D * 2.0));
    {
        const cudaError_t le_ = fg::launch_pdl(kern, dim3(static_cast<unsigned>(units)), dim3(32), smem, st,
            w.sc, w.st, w.sc_ld, c->H, c->cap, pos, pad, keep_pct, kmax, c->v_codes, c->v_meta, out, sel_out);
        if (le_ != cudaSuccess) return fg::cuda_error(le_, "kern launch");
    }
    return fg::cuda_error(cudaGetLastError(), "topk_gather launch");
}

}  // namespace

namespace fg {

fg_status launch_decode_attn(const __half* qkv, int64_t ld, const fg_kv4* c, int32_t pos,
                             const int32_t* pad, int32_t fuse_append, __half* out,
                             cudaStream_t st) {
    if (c->B == 0) return FG_OK;
    const TopkWs none{};
    if (c->d == 64) return launch_decode_t<64, false>(qkv, ld, c, pos, pad, fuse_append, out, none, st);
    return launch_decode_staged<false>(qkv, ld, c, pos, pad, fuse_append, out, none, st);
}

size_t decode_topk_ws_bytes(int32_t B, int32_t H, int32_t pos) {
    return topk_ws_layout(B, H, pos, nullptr).bytes;
}

int32_t decode_topk_kmax(int32_t pos, int32_t keep_pct) {
    return topk_count_host(pos + 1, keep_pct);
}

fg_status launch_decode_attn_topk(const __half* qkv, int64_t ld, const fg_kv4* c, int32_t pos,
                                  const int32_t* pad, int32_t fuse_append, int32_t keep_pct,
                                  int32_t* sel_out, void* ws, size_t ws_bytes, __half* out,
                                  cudaStream_t st) {
    if (c->B == 0) return FG_OK;
    const TopkWs w = topk_ws_layout(c->B, c->H, pos, ws);
    if (ws == nullptr || ws_bytes < w.bytes)
        return set_error(FG_ERR_WORKSPACE, "decode_attn_topk: workspace %zu < %zu bytes", ws_bytes,
                         w.bytes);
    const int32_t kmax = decode_topk_kmax(pos, keep_pct);
    fg_status s = c->d == 64 ? launch_decode_t<64, true>(qkv, ld, c, pos, pad, fuse_append, out, w, st)
                             : launch_decode_staged<true>(qkv, ld, c, pos, pad, fuse_append, out, w, st);
    if (s != FG_OK) return s;
    return c->d == 64 ? launch_topk_gather<64>(c, pos, pad, keep_pct, kmax, sel_out, out, w, st)
                      : launch_topk_gather<128>(c, pos, pad, keep_pct, kmax, sel_out, out, w, st);
}

fg_status launch_prefill_attn(const __half* qkv, int32_t B, int32_t s, int32_t H, int32_t d,
                              const int32_t* pad, __half* out, cudaStream_t st) {
    if (B == 0 || s == 0) return FG_OK;
    if (!prefill_attn_tc_supported(d))
        return set_error(FG_ERR_UNSUPPORTED, "prefill_attn: head dim %d not in {64, 128}", d);
    return launch_prefill_attn_tc(qkv, B, s, H, d, pad, out, st);
}

}  // namespace fg
