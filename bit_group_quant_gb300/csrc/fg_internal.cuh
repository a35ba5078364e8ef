// fg_internal.cuh -- shared device helpers (inline PTX for mbarrier, TMA and
// tcgen05) and host-side declarations used across libfg's translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fg.h"

namespace fg {

constexpr int kGroup = 64;                 // quantisation group (elements)
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s per bounded wait
constexpr int kNumSMsHint = 152;

// Device status codes written by kernels (first error wins).
constexpr int kDevTimeout = 1;

// ---------------------------------------------------------------- host side

fg_status set_error(fg_status s, const char* fmt, ...);
fg_status cuda_error(cudaError_t e, const char* what);
int* device_status_ptr();                  // per current device, never NULL on success
uint64_t wait_limit_ns();
int take_drop_arrive();                    // test knob: consumed by the next GEMM launch
int num_sms();

// Tracing (fg_trace_begin / fg_trace_end): counts every launch of the class
// and, when the class is timed, brackets the launch with a CUDA event pair.
class TraceScope {
  public:
    TraceScope(int cls_bit, cudaStream_t st, double flops, double bytes);
    ~TraceScope();
    TraceScope(const TraceScope&) = delete;
    TraceScope& operator=(const TraceScope&) = delete;

  private:
    int rec_ = -1;
    cudaStream_t st_;
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Launchers implemented in the kernel translation units.  All validate
// nothing: the exported entry points validate first.
fg_status launch_quantize_g4(const __half* x, int64_t ngroups, uint8_t* codes, float* meta,
                             cudaStream_t st);
fg_status launch_dequant_g4(const uint8_t* codes, const float* meta, int64_t ngroups,
                            __half* x, cudaStream_t st, int trace_cls = FG_TRACE_OTHER);
fg_status launch_kv_store(const __half* qkv, int64_t ld, int32_t B, int32_t T, int32_t H,
                          int32_t d, const fg_kv4* c, int32_t slot0, cudaStream_t st);
fg_status launch_layernorm(const __half* x, int64_t rows, int64_t cols, int64_t x_ld,
                           const __half* g, const __half* b, float eps, __half* y,
                           cudaStream_t st);
fg_status launch_embed(const int32_t* ids, int64_t ntok, int32_t T, int32_t pos0,
                       const int32_t* pad, const __half* e_tok, const __half* e_pos, int32_t h1,
                       __half* y, cudaStream_t st);
fg_status launch_argmax(const float* logits, int64_t B, int64_t V, int32_t* out, cudaStream_t st);
fg_status launch_decode_attn(const __half* qkv, int64_t ld, const fg_kv4* c, int32_t pos,
                             const int32_t* pad, int32_t fuse_append, __half* out,
                             cudaStream_t st);
// Top-K sparse attention keeping ceil(L * keep_pct / 100) rows (1 <= keep_pct
// <= 100): a scores pass then a select-and-gather pass, through a workspace
// of decode_topk_ws_bytes(B, H, pos); the kept slots are written to sel_out
// [B][H][decode_topk_kmax] if given.
fg_status launch_decode_attn_topk(const __half* qkv, int64_t ld, const fg_kv4* c, int32_t pos,
                                  const int32_t* pad, int32_t fuse_append, int32_t keep_pct,
                                  int32_t* sel_out, void* ws, size_t ws_bytes, __half* out,
                                  cudaStream_t st);
size_t decode_topk_ws_bytes(int32_t B, int32_t H, int32_t pos);
int32_t decode_topk_kmax(int32_t pos, int32_t keep_pct);
// The uncompressed (fp16) cache: store of T rows per sequence at slot0, and
// decode attention with the append fused.
fg_status launch_kv_store_f16(const __half* qkv, int64_t ld, int32_t T, const fg_kv16* c,
                              int32_t slot0, cudaStream_t st);
fg_status launch_decode_attn_f16(const __half* qkv, int64_t ld, const fg_kv16* c, int32_t pos,
                                 const int32_t* pad, int32_t fuse_append, __half* out,
                                 cudaStream_t st);
fg_status launch_prefill_attn(const __half* qkv, int32_t B, int32_t s, int32_t H, int32_t d,
                              const int32_t* pad, __half* out, cudaStream_t st);
// attn_tc.cu: the same causal prefill attention on tcgen05 (d 64 or 128).
bool prefill_attn_tc_supported(int32_t d);
fg_status launch_prefill_attn_tc(const __half* qkv, int32_t B, int32_t s, int32_t H, int32_t d,
                                 const int32_t* pad, __half* out, cudaStream_t st);

struct GemmPlan {
    int nt;          // activation rows per tile (MMA N), multiple of 16, <= 256
    int tok_tiles;
    int feat_tiles;  // ceil(N / 128)
    int splits;      // K splits (grid.z); > 1 only when plan_rows fit one token tile
    int kc_per_split;  // K chunks (of 64) per split, a multiple of 4
    size_t ws_bytes; // fp32 partial sums (and, for the TMEM kernel, its flags), or the fp16 weights
    size_t ws_min;   // what the launch cannot do without (the fp16 weights are optional)
    // the TMEM-operand kernel for one token tile of at most 160 rows
    // (gemm_dec.cu): clusters of dec_c CTAs share each activation stage;
    // dec_units = (feature tiles / dec_c) * (K / 256) units dealt out evenly
    // over dec_Q clusters
    // prefill-sized blocks: the weights are dequantised once into fp16 at the
    // start of the workspace and the fp16 pipeline multiplies them
    int f16w;
    int dec;
    int dec_c, dec_Q, dec_nbox;
    long long dec_units;
    size_t dec_part_bytes;   // partial sums; the flags follow
};
// The summation order of every output -- hence its value -- depends on (N, K),
// the SM count and which kernel plan_rows selects (at most 160 rows with K a
// multiple of 256: the TMEM kernel; at most 256: one token tile with K split
// across CTAs; more: whole tiles), never on M itself: launches that must give
// identical rows (the batches of one block and the whole block) pass the same
// plan_rows.  plan_rows < M means plan_rows = M.  dequant = false plans the
// fp16-weight GEMM (no TMEM kernel).
GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int64_t plan_rows = 0, bool dequant = true);
fg_status launch_gemm_g4(const __half* X, int64_t M, const fg_q4* W, const __half* bias,
                         const __half* residual, int act, __half* Y, void* ws, size_t ws_bytes,
                         cudaStream_t st, int64_t plan_rows = 0);
// gemm_dec.cu: fills the TMEM-kernel fields of pl and returns true when that
// kernel takes (M, N, K, plan_rows); launches it.
bool plan_gemm_dec(int64_t M, int64_t N, int64_t K, int64_t plan_rows, GemmPlan& pl);
fg_status launch_gemm_dec(const __half* X, int64_t M, const fg_q4* W, const __half* bias,
                          const __half* residual, int act, __half* Y, void* ws, size_t ws_bytes,
                          cudaStream_t st, const GemmPlan& pl);
// Programmatic dependent launch.  Every kernel of a layer step is launched
// with programmatic stream serialization: it may be scheduled while the
// kernel before it in the stream is still running, so its set-up (barriers,
// TMEM, tensor-map prefetch) and its reads of data no earlier kernel writes
// (the 4-bit weights) overlap that kernel's tail.  Each kernel signals
// griddep_launch() early and calls griddep_wait() before its first access to
// memory that an earlier kernel writes or reads.  The next kernel is
// scheduled only after every CTA of this one has started, so a grid whose
// CTAs wait on one another (all co-resident) is never starved by it.
// (Launched without the attribute, or after a non-kernel stream operation,
// the wait returns at once and the signal has no effect.)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}
// Adds the programmatic-serialization attribute to a launch configuration
// that already carries `n` attributes in `attr` (room for one more).
inline void add_pdl_attr(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int n) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = n + 1;
}

// 2-D row-major tensor map [rows][cols] of `esize`-byte elements, box {bx, by}.
fg_status make_tmap(CUtensorMap* tm, const void* ptr, CUtensorMapDataType dt, int esize,
                    uint64_t cols, uint64_t rows, uint32_t bx, uint32_t by,
                    CUtensorMapSwizzle swz);
// gemm_pf.cu: Y = act(X W16^T + bias) + residual with fp16 weights W16 [N][K]
// on CTA pairs (the prefill regime, weights dequantised once beforehand).
fg_status launch_gemm_pf(const __half* X, int64_t M, const __half* W16, int64_t N, int64_t K,
                         const __half* bias, const __half* residual, int act, __half* Y,
                         cudaStream_t st);
fg_status launch_gemm_f16_f32out(const __half* X, int64_t M, const __half* W, int64_t N,
                                 int64_t K, float* Y, cudaStream_t st);

}  // namespace fg

// ---------------------------------------------------------------- device side
namespace fgd {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch (see fg::launch_pdl): wait until every
// earlier kernel of the stream has completed and its memory is visible;
// allow the next kernel to be scheduled.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void report(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  Returns
// false if the time limit passes or, when `abort` is not null, another role
// of the CTA raised *abort.  Drains of work already in flight pass a null
// `abort` so that they end only on completion or on the time limit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0) {
            if (abort != nullptr && *abort) return false;
            if (globaltimer() - t0 > limit_ns) return false;
        }
    }
}

// Same, for long waits of warps that have nothing else to do: backs off with
// __nanosleep so the spinning leaves issue slots to the other warps of its
// sub-partition.  Never stops early on an abort flag (used for drains).
__device__ __forceinline__ bool mbar_wait_sleepy(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        __nanosleep(200);
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

// ---- TMA (bulk tensor copies, no multicast)
__device__ __forceinline__ void prefetch_tmap(const void* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tm, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tm), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// 1-D bulk copy global -> this CTA's shared memory (both addresses 16-byte
// aligned, size a multiple of 16), completing `bytes` of transaction count on
// the mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// Orders this thread's earlier generic global writes before later async-proxy
// (TMA / bulk copy) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Multicast variant: the box lands at the same shared-memory offset in every
// CTA of the cluster named in `mask`, completing bytes on each one's mbarrier
// at the same offset.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const void* tm, int x, int y,
                                               uint32_t bar, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tm), "r"(x), "r"(y), "r"(bar), "h"(mask)
        : "memory");
}

// ---- thread-block clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tcgen05 (5th-generation tensor cores, accumulators in TMEM)
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, fp16 inputs, fp32 accumulate: A is 128
// lanes (rows) x 8 columns (16 fp16 k values, two per 32-bit column) of TMEM.
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on an mbarrier when all previously issued tcgen05 ops of this
// thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// Arrive once on the mbarrier at the same offset in every CTA of `mask`
// when all previously issued tcgen05 ops of this thread have completed.
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
// 32 lanes x 32 bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
        "14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// 32 lanes x 32 bit, 8 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 lanes x 32 bit, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- CTA pairs (cta_group::2): one MMA over two SMs of a 2-CTA cluster.
// M = 256 rows, the even CTA's 128 rows and the odd CTA's 128 rows of A at
// the same shared-memory offset; N split in halves, columns 0..N/2-1 from the
// even CTA's B and N/2..N-1 from the odd CTA's; each CTA's TMEM receives its
// own 128 rows of D.  Issued by the even CTA only.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T over the pair, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at the same offset in every CTA of `mask` when
// all pair MMAs previously issued by this thread have completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier that may sit in the peer CTA of the pair (bar: shared::cluster
// address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tm, int x, int y,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tm), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// Arrive (release, cluster scope) on an mbarrier of another CTA of the
// cluster (bar: shared::cluster address from mapa_shared).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait (acquire, cluster scope) for a barrier that other CTAs of the
// cluster arrive on; same contract as mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort, uint64_t limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 31u) == 0) {
            if (abort != nullptr && *abort) return false;
            if (globaltimer() - t0 > limit_ns) return false;
        }
    }
}

// ---- flags between CTAs of one grid (global memory, gpu scope)
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes (64 fp16), 8-row atoms of 1024 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);      // start address
    d |= static_cast<uint64_t>(16u >> 4) << 16;                 // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;               // stride byte offset: 8 rows
    d |= static_cast<uint64_t>(1) << 46;                        // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                        // 128-byte swizzle
    return d;
}
// Instruction descriptor: fp16 A and B (K-major), fp32 D, shape M x N.
__device__ __forceinline__ uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// ---- dequantisation of stored 4-bit codes
// 8 codes (one 32-bit word, element 0 in the lowest nibble) -> the 8 fp16
// values fp16(fma(c, s, m)): one fp32 fused multiply-add, then round to
// nearest even -- the dequantisation of the definition, bit for bit.
//
// A code is masked into an fp16 word as the subnormal c * 2^-24 (nibbles 1
// and 3 of each byte pair are taken in place, as 16c * 2^-24), converted to
// fp32 exactly, and multiplied by S = s * 2^24 (S16 = s * 2^20): the product
// is exactly c * s, so the fma rounds c*s + m once, as the definition does.
// (Scaling s by a power of two is exact: fp16 inputs bound s below 2^14.)
__device__ __forceinline__ uint4 dequant8(uint32_t w, float S, float S16, float m) {
    const uint32_t w8 = w >> 8;
    const uint32_t t0 = w & 0x000F000Fu, t1 = w & 0x00F000F0u;     // (c0, c4), (16c1, 16c5)
    const uint32_t t2 = w8 & 0x000F000Fu, t3 = w8 & 0x00F000F0u;   // (c2, c6), (16c3, 16c7)
    const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&t0));
    const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&t1));
    const float2 a2 = __half22float2(*reinterpret_cast<const __half2*>(&t2));
    const float2 a3 = __half22float2(*reinterpret_cast<const __half2*>(&t3));
    __half2 h[4];
    h[0] = __floats2half2_rn(__fmaf_rn(a0.x, S, m), __fmaf_rn(a1.x, S16, m));   // (e0, e1)
    h[1] = __floats2half2_rn(__fmaf_rn(a2.x, S, m), __fmaf_rn(a3.x, S16, m));   // (e2, e3)
    h[2] = __floats2half2_rn(__fmaf_rn(a0.y, S, m), __fmaf_rn(a1.y, S16, m));   // (e4, e5)
    h[3] = __floats2half2_rn(__fmaf_rn(a2.y, S, m), __fmaf_rn(a3.y, S16, m));   // (e6, e7)
    return *reinterpret_cast<uint4*>(h);
}

// The same eight values with the FMAs of codes that share a multiplier
// paired into packed fp32x2 FMAs (each half one single-rounding FMA, so the
// result is bit-identical to dequant8): 21 instructions per word instead of
// 25, for the kernels where the dequantisation bounds the throughput.
__device__ __forceinline__ uint4 dequant8_x2(uint32_t w, float S, float S16, float m) {
    const uint32_t w8 = w >> 8;
    const uint32_t t0 = w & 0x000F000Fu, t1 = w & 0x00F000F0u;     // (c0, c4), (16c1, 16c5)
    const uint32_t t2 = w8 & 0x000F000Fu, t3 = w8 & 0x00F000F0u;   // (c2, c6), (16c3, 16c7)
    const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&t0));
    const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&t1));
    const float2 a2 = __half22float2(*reinterpret_cast<const __half2*>(&t2));
    const float2 a3 = __half22float2(*reinterpret_cast<const __half2*>(&t3));
    const float2 SS = make_float2(S, S), S16S16 = make_float2(S16, S16), MM = make_float2(m, m);
    const float2 r0 = __ffma2_rn(a0, SS, MM);        // (e0, e4)
    const float2 r1 = __ffma2_rn(a1, S16S16, MM);    // (e1, e5)
    const float2 r2 = __ffma2_rn(a2, SS, MM);        // (e2, e6)
    const float2 r3 = __ffma2_rn(a3, S16S16, MM);    // (e3, e7)
    __half2 h[4];
    h[0] = __floats2half2_rn(r0.x, r1.x);   // (e0, e1)
    h[1] = __floats2half2_rn(r2.x, r3.x);   // (e2, e3)
    h[2] = __floats2half2_rn(r0.y, r1.y);   // (e4, e5)
    h[3] = __floats2half2_rn(r2.y, r3.y);   // (e6, e7)
    return *reinterpret_cast<uint4*>(h);
}

// ---- IEEE total order helpers (finite values): -0 below +0.
__device__ __forceinline__ bool total_less(float a, float b) {
    return a < b || (a == b && (__float_as_uint(a) >> 31) > (__float_as_uint(b) >> 31));
}
__device__ __forceinline__ float tmin(float a, float b) { return total_less(b, a) ? b : a; }
__device__ __forceinline__ float tmax(float a, float b) { return total_less(a, b) ? b : a; }

// The 4-bit code of num = x - min (>= 0): clamp(rint(num / scale), 0, 15)
// with the IEEE quotient; inv = the IEEE reciprocal of scale.  The fast
// quotient num * inv lies within 3 ulp of the IEEE one; where it lies that
// close to a rounding tie, the IEEE division itself is taken.  Rounding to an
// integer by adding 1.5 * 2^23: for 0 <= t <= 15 the sum's unit in the last
// place is 1, so round-to-nearest-even of the sum is rint(t) and its low
// mantissa bits hold the integer; clamping to [0, 15] first gives
// clamp(rint(t)) as the bounds are integers.
constexpr float kCodeMagic = 12582912.0f;
// The fast code; *near_tie set when the fast quotient lies too close to a
// rounding tie to decide it (then code4_exact decides).
__device__ __forceinline__ uint32_t code4_fast(float num, float inv, bool* near_tie) {
    const float t = fminf(fmaxf(__fmul_rn(num, inv), 0.0f), 15.0f);
    const float m = __fadd_rn(t, kCodeMagic);
    *near_tie = fabsf(fabsf(__fsub_rn(t, __fsub_rn(m, kCodeMagic))) - 0.5f) < 1.0f / 65536.0f;
    return __float_as_uint(m) & 0xFu;
}
__device__ __forceinline__ uint32_t code4_exact(float num, float scale) {
    const float t = fminf(fmaxf(__fdiv_rn(num, scale), 0.0f), 15.0f);
    return __float_as_uint(__fadd_rn(t, kCodeMagic)) & 0xFu;
}
__device__ __forceinline__ uint32_t code4(float num, float inv, float scale) {
    bool near_tie;
    const uint32_t c = code4_fast(num, inv, &near_tie);
    return near_tie ? code4_exact(num, scale) : c;
}

// Quantise one group of 64 values held by 8 consecutive lanes (8 values per
// lane, lane8 = lane & 7 holds elements 8*lane8 .. 8*lane8+7).  Returns the
// 8 codes packed into one word (element 8*lane8 in the lowest nibble) and
// writes (min, scale) of the group.  Matches the definition bit for bit:
// fp32 min/max in the IEEE total order, scale = (M - m) / 15 (IEEE divide),
// code = clamp(rint((x - m) / scale), 0, 15), all zero when scale == 0.
__device__ __forceinline__ uint32_t quantize8(const float (&v)[8], float& mn_out,
                                              float& scale_out) {
    float mn = v[0], mx = v[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) {
        mn = tmin(mn, v[i]);
        mx = tmax(mx, v[i]);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        mn = tmin(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = tmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const float scale = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
    uint32_t packed = 0;
    if (scale != 0.0f) {
        const float inv = __frcp_rn(scale);
#pragma unroll
        for (int i = 0; i < 8; ++i) packed |= code4(__fsub_rn(v[i], mn), inv, scale) << (4 * i);
    }
    mn_out = mn;
    scale_out = scale;
    return packed;
}

}  // namespace fgd
