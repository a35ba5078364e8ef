// noalloc.cu -- fg_dequant_gemm_g4_noalloc: the 4-bit dequant-GEMM for
// callers that must not allocate device memory.
//
// fg_dequant_gemm_g4 takes its K-split scratch (fp32 partial sums) from a
// workspace the caller allocates.  Some callers cannot do that: a plugin
// running inside a host program that owns the whole device-memory budget
// through its own pool and forbids other allocations, or a latency-critical
// loop where cudaMalloc / cudaFree would synchronise the device.  This entry
// point gives them the same computation with the scratch held in a fixed
// file-scope device array instead; it calls no allocating routine.
#include <mutex>

#include "fg_internal.cuh"

namespace {

// Fixed scratch for the K-split partial sums: 16 MiB on every GPU that loads
// the library, held until the process exits.
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDev];   // device address of g_noalloc_scratch, per device

// In host code g_noalloc_scratch names a host-side stand-in, not device
// memory, so the device address is looked up once per device (with that
// device current) and cached.
fg_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fg::cuda_error(e, "dequant_gemm_g4_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDev)
        return fg::set_error(FG_ERR_UNSUPPORTED, "dequant_gemm_g4_noalloc: device %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return fg::cuda_error(e, "dequant_gemm_g4_noalloc: cudaGetSymbolAddress");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return FG_OK;
}

}  // namespace

extern "C" {

fg_status fg_dequant_gemm_g4_noalloc(const fg_f16* X, int64_t M, const fg_q4* W,
                                     const fg_f16* bias, const fg_f16* residual, int32_t act,
                                     fg_f16* Y, fg_stream stream) {
    if (W == nullptr) return fg::set_error(FG_ERR_NULL, "dequant_gemm_g4_noalloc: null fg_q4");
    // Only the scratch a shape cannot do without: the K-split partial sums
    // (and the decode kernel's fixup flags).  Prefill-sized blocks, which
    // would put an fp16 copy of the weights into a large enough workspace,
    // are offered exactly `need` bytes, so they always take the fused path
    // and the array never holds a weight copy.
    const size_t need = (M > 0 && W->rows > 0 && W->cols > 0) ? fg::plan_gemm(M, W->rows, W->cols).ws_min : 0;
    if (need > kNoAllocScratchBytes)
        return fg::set_error(FG_ERR_WORKSPACE,
                             "dequant_gemm_g4_noalloc: this shape needs %zu bytes of K-split "
                             "scratch, the built-in scratch holds %zu; use fg_dequant_gemm_g4 "
                             "with a caller workspace",
                             need, kNoAllocScratchBytes);
    void* scratch = nullptr;
    fg_status s = scratch_address(&scratch);
    if (s != FG_OK) return s;
    // Nothing in the scratch has to start at zero.  Every partial sum read is
    // written earlier in the same call.  The decode kernel's fixup flags (after
    // its partial sums) hold a per-launch tag, set once a part is written and
    // cleared once it is consumed; the tag also changes after fg_check reports
    // a timeout, so flags a failed call left set never match a later call.
    return fg_dequant_gemm_g4(X, M, W, bias, residual, act, Y, need > 0 ? scratch : nullptr,
                              need, stream);
}

}  // extern "C"
