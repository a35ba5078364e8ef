// api.cu -- libfg's exported C ABI: host-side validation, the per-device
// status word, and the decoder layer step that sequences the kernels under
// the block schedule.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "fg_internal.cuh"

namespace {

thread_local char g_err[512];

// FG device status word, one per device: [0] the first error code a kernel
// reported (0: none), [1] how many times fg_check has cleared an error.  The
// second word lets kernels that tag cross-CTA flags with a per-launch value
// (the decode GEMM's fixup) change that value after a failed launch, so a
// replay of the same launch (a CUDA graph) never accepts a flag the failed
// launch left behind.
__device__ int g_dev_status[2];

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
int g_sms[kMaxDevices];
std::mutex g_dev_mu;

std::atomic<long long> g_wait_ns{0};
std::atomic<int> g_drop_arrive{0};

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
    return d;
}

inline cudaStream_t S(fg_stream s) { return reinterpret_cast<cudaStream_t>(s); }
inline const __half* H(const fg_f16* p) { return reinterpret_cast<const __half*>(p); }
inline __half* Hm(fg_f16* p) { return reinterpret_cast<__half*>(p); }

#define FG_REQUIRE(cond, status, ...)                 \
    do {                                              \
        if (!(cond)) return fg::set_error(status, __VA_ARGS__); \
    } while (0)

fg_status check_q4(const fg_q4* q, const char* what) {
    FG_REQUIRE(q != nullptr, FG_ERR_NULL, "%s: null fg_q4", what);
    FG_REQUIRE(q->codes != nullptr && q->meta != nullptr, FG_ERR_NULL, "%s: null codes/meta", what);
    FG_REQUIRE(q->rows >= 0 && q->cols > 0 && q->cols % 64 == 0, FG_ERR_SHAPE,
               "%s: cols %lld must be a positive multiple of 64", what, (long long)q->cols);
    FG_REQUIRE(fg::aligned16(q->codes) && fg::aligned16(q->meta), FG_ERR_ALIGN,
               "%s: codes/meta must be 16-byte aligned", what);
    return FG_OK;
}

fg_status check_kv(const fg_kv4* c, const char* what) {
    FG_REQUIRE(c != nullptr, FG_ERR_NULL, "%s: null cache", what);
    FG_REQUIRE(c->k_codes && c->v_codes && c->k_meta && c->v_meta, FG_ERR_NULL,
               "%s: null cache buffer", what);
    FG_REQUIRE(c->d == 64 || c->d == 128, FG_ERR_UNSUPPORTED, "%s: head dim %d not in {64,128}",
               what, c->d);
    FG_REQUIRE(c->B >= 0 && c->H > 0 && c->cap > 0, FG_ERR_SHAPE, "%s: bad B/H/cap", what);
    FG_REQUIRE(fg::aligned16(c->k_codes) && fg::aligned16(c->v_codes) &&
                   fg::aligned16(c->k_meta) && fg::aligned16(c->v_meta),
               FG_ERR_ALIGN, "%s: cache buffers must be 16-byte aligned", what);
    return FG_OK;
}

fg_kv4 sub_cache(const fg_kv4* c, int32_t b0, int32_t nb) {
    fg_kv4 s = *c;
    const int64_t rows = static_cast<int64_t>(b0) * c->H * c->cap;
    s.k_codes = c->k_codes + rows * (c->d / 2);
    s.v_codes = c->v_codes + rows * (c->d / 2);
    s.k_meta = c->k_meta + rows * (c->d / 64) * 2;
    s.v_meta = c->v_meta + rows * (c->d / 64) * 2;
    s.B = nb;
    return s;
}

fg_status check_kv16(const fg_kv16* c, const char* what) {
    FG_REQUIRE(c != nullptr, FG_ERR_NULL, "%s: null cache", what);
    FG_REQUIRE(c->k && c->v, FG_ERR_NULL, "%s: null cache buffer", what);
    FG_REQUIRE(c->d == 64 || c->d == 128, FG_ERR_UNSUPPORTED, "%s: head dim %d not in {64,128}",
               what, c->d);
    FG_REQUIRE(c->B >= 0 && c->H > 0 && c->cap > 0, FG_ERR_SHAPE, "%s: bad B/H/cap", what);
    FG_REQUIRE(fg::aligned16(c->k) && fg::aligned16(c->v), FG_ERR_ALIGN,
               "%s: cache buffers must be 16-byte aligned", what);
    return FG_OK;
}

fg_kv16 sub_cache(const fg_kv16* c, int32_t b0, int32_t nb) {
    fg_kv16 s = *c;
    const int64_t el = static_cast<int64_t>(b0) * c->H * c->cap * c->d;
    s.k = c->k + el;
    s.v = c->v + el;
    s.B = nb;
    return s;
}

// The cache-specific steps of a layer: the prefill's store of the prompt's
// K/V rows and the decode step's attention (append fused).
fg_status kv_prefill_store(const __half* qkv, int64_t ld, int32_t nb, int32_t T, int32_t Hh,
                           int32_t d, const fg_kv4* c, cudaStream_t st) {
    return fg::launch_kv_store(qkv, ld, nb, T, Hh, d, c, 0, st);
}
fg_status kv_prefill_store(const __half* qkv, int64_t ld, int32_t, int32_t T, int32_t, int32_t,
                           const fg_kv16* c, cudaStream_t st) {
    return fg::launch_kv_store_f16(qkv, ld, T, c, 0, st);
}
fg_status kv_decode_attn(const __half* qkv, int64_t ld, const fg_kv4* c, int32_t pos,
                         const int32_t* pad, int32_t topk_pct, void* tk, size_t tk_bytes,
                         __half* out, cudaStream_t st) {
    if (topk_pct > 0 && topk_pct < 100)
        return fg::launch_decode_attn_topk(qkv, ld, c, pos, pad, 1, topk_pct, nullptr, tk, tk_bytes,
                                           out, st);
    return fg::launch_decode_attn(qkv, ld, c, pos, pad, 1, out, st);
}
fg_status kv_decode_attn(const __half* qkv, int64_t ld, const fg_kv16* c, int32_t pos,
                         const int32_t* pad, int32_t, void*, size_t, __half* out, cudaStream_t st) {
    return fg::launch_decode_attn_f16(qkv, ld, c, pos, pad, 1, out, st);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct LayerWs {
    __half *a, *qkv, *attn, *h, *u;
    void* gemm;
    size_t gemm_bytes;
    void* topk;          // top-K attention's scores (decode with 0 < topk_pct < 100)
    size_t topk_bytes;
    size_t total;
};

// Top-K scratch of one decode attention launch of nb sequences at context
// pos + 1 (0 unless 0 < topk_pct < 100).
size_t topk_scratch(int32_t phase, int32_t topk_pct, int64_t nb, int32_t H, int32_t pos) {
    if (phase != FG_PHASE_DECODE || topk_pct <= 0 || topk_pct >= 100) return 0;
    return fg::decode_topk_ws_bytes(static_cast<int32_t>(nb), H, pos);
}

LayerWs layer_ws_layout(const fg_layer* w, int64_t rows, int64_t rows_per_launch, char* base,
                        size_t topk_bytes) {
    LayerWs L{};
    const int64_t h1 = w->h1, h2 = w->h2;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char* p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    L.a = reinterpret_cast<__half*>(take(sizeof(__half) * rows * h1));
    L.qkv = reinterpret_cast<__half*>(take(sizeof(__half) * rows * 3 * h1));
    L.attn = reinterpret_cast<__half*>(take(sizeof(__half) * rows * h1));
    L.h = reinterpret_cast<__half*>(take(sizeof(__half) * rows * h1));
    L.u = reinterpret_cast<__half*>(take(sizeof(__half) * rows * h2));
    size_t g = 0;
    const int64_t NK[4][2] = {{3 * h1, h1}, {h1, h1}, {h2, h1}, {h1, h2}};
    for (auto& nk : NK) {
        const fg::GemmPlan pl = fg::plan_gemm(rows_per_launch, nk[0], nk[1], rows);
        if (pl.ws_bytes > g) g = pl.ws_bytes;
    }
    L.gemm_bytes = g;
    L.gemm = take(g);
    L.topk_bytes = topk_bytes;
    L.topk = take(topk_bytes);
    L.total = off;
    return L;
}

fg_status check_layer(const fg_layer* w) {
    FG_REQUIRE(w != nullptr, FG_ERR_NULL, "layer: null fg_layer");
    fg_status s;
    if ((s = check_q4(&w->qkv, "layer.qkv")) != FG_OK) return s;
    if ((s = check_q4(&w->out, "layer.out")) != FG_OK) return s;
    if ((s = check_q4(&w->fc1, "layer.fc1")) != FG_OK) return s;
    if ((s = check_q4(&w->fc2, "layer.fc2")) != FG_OK) return s;
    FG_REQUIRE(w->b_qkv && w->b_out && w->b_fc1 && w->b_fc2 && w->ln1_g && w->ln1_b && w->ln2_g &&
                   w->ln2_b,
               FG_ERR_NULL, "layer: null bias or LayerNorm parameter");
    FG_REQUIRE(w->H > 0 && w->h1 > 0 && w->h1 % w->H == 0, FG_ERR_SHAPE, "layer: h1 %% H != 0");
    const int d = w->h1 / w->H;
    FG_REQUIRE(d == 64 || d == 128, FG_ERR_UNSUPPORTED, "layer: head dim %d not in {64,128}", d);
    FG_REQUIRE(w->h2 % 64 == 0 && w->h1 % 64 == 0, FG_ERR_SHAPE, "layer: h1, h2 must be multiples of 64");
    FG_REQUIRE(w->qkv.rows == 3 * w->h1 && w->qkv.cols == w->h1 && w->out.rows == w->h1 &&
                   w->out.cols == w->h1 && w->fc1.rows == w->h2 && w->fc1.cols == w->h1 &&
                   w->fc2.rows == w->h1 && w->fc2.cols == w->h2,
               FG_ERR_SHAPE, "layer: projection shapes do not match h1=%d h2=%d", w->h1, w->h2);
    return FG_OK;
}

}  // namespace

namespace fg {

fg_status set_error(fg_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

fg_status cuda_error(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return FG_OK;
    return set_error(FG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int* device_status_ptr() {
    const int d = current_device();
    if (d < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_status_ptr[d]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dev_status) != cudaSuccess) return nullptr;
        g_status_ptr[d] = static_cast<int*>(p);
    }
    return g_status_ptr[d];
}

int num_sms() {
    const int d = current_device();
    if (d < 0) return kNumSMsHint;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_sms[d]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0)
            n = kNumSMsHint;
        g_sms[d] = n;
    }
    return g_sms[d];
}

uint64_t wait_limit_ns() {
    const long long w = g_wait_ns.load();
    return w > 0 ? static_cast<uint64_t>(w) : kDefaultWaitNs;
}

int take_drop_arrive() { return g_drop_arrive.exchange(0); }

// ---------------------------------------------------------------- tracing

namespace {

struct TraceRec {
    int cls;
    cudaEvent_t a, b;
};

struct Tracer {
    std::mutex mu;
    bool on = false;
    int timed_mask = 0;
    fg_trace_stats st{};
    std::vector<TraceRec> recs;
    std::vector<cudaEvent_t> pool;
    size_t used = 0;

    cudaEvent_t next_event() {
        if (used == pool.size()) {
            cudaEvent_t e = nullptr;
            if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
            pool.push_back(e);
        }
        return pool[used++];
    }
};

Tracer& tracer() {
    static Tracer* t = new Tracer();   // never destroyed: events may outlive static dtors
    return *t;
}

int class_index(int bit) {
    int i = 0;
    while (bit > 1) {
        bit >>= 1;
        ++i;
    }
    return i;
}

}  // namespace

TraceScope::TraceScope(int cls_bit, cudaStream_t st, double flops, double bytes) : st_(st) {
    Tracer& t = tracer();
    std::lock_guard<std::mutex> lk(t.mu);
    if (!t.on) return;
    const int ci = class_index(cls_bit);
    t.st.launches[ci] += 1;
    t.st.flops[ci] += flops;
    t.st.bytes[ci] += bytes;
    if (!(t.timed_mask & cls_bit)) return;
    TraceRec r{ci, t.next_event(), t.next_event()};
    if (!r.a || !r.b) return;
    cudaEventRecord(r.a, st);
    rec_ = static_cast<int>(t.recs.size());
    t.recs.push_back(r);
}

TraceScope::~TraceScope() {
    if (rec_ < 0) return;
    Tracer& t = tracer();
    std::lock_guard<std::mutex> lk(t.mu);
    if (rec_ < static_cast<int>(t.recs.size())) cudaEventRecord(t.recs[rec_].b, st_);
}

}  // namespace fg

// One decoder layer over either cache kind (Cache = fg_kv4 or fg_kv16); the
// cache is validated by the caller.
template <class Cache>
fg_status layer_step_impl(const fg_layer* w, const Cache* cache, const fg_f16* x_in, fg_f16* x_out,
                          int32_t phase, int32_t T, int32_t pos, const int32_t* pad, fg_policy p,
                          void* workspace, size_t ws_bytes, fg_stream stream) {
    fg_status s = check_layer(w);
    if (s != FG_OK) return s;
    FG_REQUIRE(x_in && x_out, FG_ERR_NULL, "layer_step: null x_in or x_out");
    FG_REQUIRE(x_in != x_out, FG_ERR_SHAPE, "layer_step: x_in and x_out may not alias");
    FG_REQUIRE((reinterpret_cast<uintptr_t>(pad) & 3u) == 0, FG_ERR_ALIGN,
               "layer_step: pad must be 4-byte aligned");
    FG_REQUIRE(fg::aligned16(x_in) && fg::aligned16(x_out), FG_ERR_ALIGN,
               "layer_step: x_in and x_out must be 16-byte aligned");
    FG_REQUIRE(p.gbs > 0 && p.k > 0 && p.order >= 0 && p.order <= 2, FG_ERR_SHAPE,
               "layer_step: bad policy");
    FG_REQUIRE(p.topk_pct >= 0 && p.topk_pct <= 100, FG_ERR_SHAPE,
               "layer_step: topk_pct %d outside [0, 100]", p.topk_pct);
    const int32_t bls = p.gbs * p.k;
    FG_REQUIRE(cache->B == bls, FG_ERR_SHAPE, "layer_step: cache holds %d sequences, bls = %d",
               cache->B, bls);
    const int d = w->h1 / w->H;
    FG_REQUIRE(cache->H == w->H && cache->d == d, FG_ERR_SHAPE, "layer_step: cache H/d mismatch");
    FG_REQUIRE(phase == FG_PHASE_PREFILL || phase == FG_PHASE_DECODE, FG_ERR_SHAPE,
               "layer_step: bad phase");
    if (phase == FG_PHASE_PREFILL) {
        FG_REQUIRE(T >= 1 && T <= cache->cap, FG_ERR_SHAPE, "layer_step: prefill T %d outside [1, cap]", T);
    } else {
        FG_REQUIRE(T == 1, FG_ERR_SHAPE, "layer_step: decode needs T == 1");
        FG_REQUIRE(pos >= 0 && pos < cache->cap, FG_ERR_SHAPE, "layer_step: pos %d outside [0, %d)",
                   pos, cache->cap);
    }
    const int64_t rows = static_cast<int64_t>(bls) * T;
    const int64_t per = p.order == FG_ORDER_BLOCK ? rows : static_cast<int64_t>(p.gbs) * T;
    const size_t tk = topk_scratch(phase, p.topk_pct, per / T, w->H, pos);
    const LayerWs need = layer_ws_layout(w, rows, per, nullptr, tk);
    FG_REQUIRE(workspace != nullptr && ws_bytes >= need.total, FG_ERR_WORKSPACE,
               "layer_step: workspace %zu < %zu bytes", ws_bytes, need.total);
    FG_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, FG_ERR_ALIGN,
               "layer_step: workspace must be 256-byte aligned");
    const LayerWs L = layer_ws_layout(w, rows, per, static_cast<char*>(workspace), tk);
    const cudaStream_t st = S(stream);
    const int64_t h1 = w->h1;

    const int nbatch = p.order == FG_ORDER_BLOCK ? 1 : p.k;
    const int32_t nb = p.order == FG_ORDER_BLOCK ? bls : p.gbs;
    for (int it = 0; it < nbatch; ++it) {
        const int bi = p.order == FG_ORDER_BATCHES_REV ? nbatch - 1 - it : it;
        const int32_t b0 = bi * nb;
        const int64_t r0 = static_cast<int64_t>(b0) * T, nr = static_cast<int64_t>(nb) * T;
        const Cache c = sub_cache(cache, b0, nb);
        const int32_t* pb = pad ? pad + b0 : nullptr;
        const __half* xin = H(x_in) + r0 * h1;
        __half* xout = Hm(x_out) + r0 * h1;
        __half* a = L.a + r0 * h1;
        __half* qkv = L.qkv + r0 * 3 * h1;
        __half* attn = L.attn + r0 * h1;
        __half* hh = L.h + r0 * h1;
        __half* u = L.u + r0 * w->h2;
#define FG_RUN(expr)                     \
    do {                                 \
        fg_status _s = (expr);           \
        if (_s != FG_OK) return _s;      \
    } while (0)
        FG_RUN(fg::launch_layernorm(xin, nr, h1, h1, H(w->ln1_g), H(w->ln1_b), w->ln_eps, a, st));
        FG_RUN(fg::launch_gemm_g4(a, nr, &w->qkv, H(w->b_qkv), nullptr, FG_ACT_NONE, qkv, L.gemm,
                                  L.gemm_bytes, st, rows));
        if (phase == FG_PHASE_PREFILL) {
            FG_RUN(fg::launch_prefill_attn(qkv, nb, T, w->H, d, pb, attn, st));
            FG_RUN(kv_prefill_store(qkv, 3 * h1, nb, T, w->H, d, &c, st));
        } else {
            FG_RUN(kv_decode_attn(qkv, 3 * h1, &c, pos, pb, p.topk_pct, L.topk, L.topk_bytes, attn,
                                  st));
        }
        FG_RUN(fg::launch_gemm_g4(attn, nr, &w->out, H(w->b_out), xin, FG_ACT_NONE, hh, L.gemm,
                                  L.gemm_bytes, st, rows));
        FG_RUN(fg::launch_layernorm(hh, nr, h1, h1, H(w->ln2_g), H(w->ln2_b), w->ln_eps, a, st));
        FG_RUN(fg::launch_gemm_g4(a, nr, &w->fc1, H(w->b_fc1), nullptr, FG_ACT_RELU, u, L.gemm,
                                  L.gemm_bytes, st, rows));
        FG_RUN(fg::launch_gemm_g4(u, nr, &w->fc2, H(w->b_fc2), hh, FG_ACT_NONE, xout, L.gemm,
                                  L.gemm_bytes, st, rows));
#undef FG_RUN
    }
    return FG_OK;
}

extern "C" {

const char* fg_status_str(fg_status s) {
    switch (s) {
        case FG_OK: return "ok";
        case FG_ERR_NULL: return "null pointer";
        case FG_ERR_SHAPE: return "bad shape";
        case FG_ERR_ALIGN: return "misaligned";
        case FG_ERR_UNSUPPORTED: return "unsupported";
        case FG_ERR_CUDA: return "cuda error";
        case FG_ERR_TIMEOUT: return "device wait timed out";
        case FG_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

const char* fg_last_error(void) { return g_err; }

int32_t fg_version(void) { return (4 << 16) | 0; }

fg_status fg_check(fg_stream stream) {
    cudaError_t e = cudaStreamSynchronize(S(stream));
    if (e != cudaSuccess) return fg::cuda_error(e, "fg_check stream");
    int* p = fg::device_status_ptr();
    if (!p) return fg::set_error(FG_ERR_CUDA, "fg_check: no device status word");
    int v = 0;
    e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fg::cuda_error(e, "fg_check read");
    if (v != 0) {
        int gen = 0;
        cudaMemcpy(&gen, p + 1, sizeof(int), cudaMemcpyDeviceToHost);
        const int words[2] = {0, gen + 1};
        cudaMemcpy(p, words, sizeof(words), cudaMemcpyHostToDevice);
        return fg::set_error(FG_ERR_TIMEOUT, "a bounded device wait expired (code %d)", v);
    }
    return FG_OK;
}

fg_status fg_trace_begin(int32_t timed_mask) {
    fg::Tracer& t = fg::tracer();
    std::lock_guard<std::mutex> lk(t.mu);
    t.on = true;
    t.timed_mask = timed_mask;
    t.st = fg_trace_stats{};
    t.recs.clear();
    t.used = 0;
    return FG_OK;
}

fg_status fg_trace_end(fg_trace_stats* out) {
    fg::Tracer& t = fg::tracer();
    std::lock_guard<std::mutex> lk(t.mu);
    t.on = false;
    for (const auto& r : t.recs) {
        cudaError_t e = cudaEventSynchronize(r.b);
        if (e != cudaSuccess) return fg::cuda_error(e, "fg_trace_end sync");
        float ms = 0.0f;
        e = cudaEventElapsedTime(&ms, r.a, r.b);
        if (e != cudaSuccess) return fg::cuda_error(e, "fg_trace_end elapsed");
        t.st.ms[r.cls] += ms;
    }
    t.recs.clear();
    t.used = 0;
    if (out) *out = t.st;
    return FG_OK;
}

fg_status fg_debug_set(int32_t knob, int64_t value) {
    if (knob == FG_KNOB_DROP_ARRIVE) {
        g_drop_arrive.store(value ? 1 : 0);
        return FG_OK;
    }
    if (knob == FG_KNOB_WAIT_NS) {
        g_wait_ns.store(value > 0 ? value : 0);
        return FG_OK;
    }
    return fg::set_error(FG_ERR_UNSUPPORTED, "unknown knob %d", knob);
}

fg_status fg_quantize_g4(const fg_f16* x, int64_t rows, int64_t cols, const fg_q4* out,
                         fg_stream stream) {
    FG_REQUIRE(x != nullptr, FG_ERR_NULL, "quantize_g4: null x");
    fg_status s = check_q4(out, "quantize_g4");
    if (s != FG_OK) return s;
    FG_REQUIRE(rows >= 0 && out->rows == rows && out->cols == cols, FG_ERR_SHAPE,
               "quantize_g4: out is [%lld][%lld], x is [%lld][%lld]", (long long)out->rows,
               (long long)out->cols, (long long)rows, (long long)cols);
    FG_REQUIRE(fg::aligned16(x), FG_ERR_ALIGN, "quantize_g4: x must be 16-byte aligned");
    return fg::launch_quantize_g4(H(x), rows * (cols / 64), out->codes, out->meta, S(stream));
}

fg_status fg_dequant_g4(const fg_q4* in, fg_f16* x, fg_stream stream) {
    fg_status s = check_q4(in, "dequant_g4");
    if (s != FG_OK) return s;
    FG_REQUIRE(x != nullptr, FG_ERR_NULL, "dequant_g4: null x");
    FG_REQUIRE(fg::aligned16(x), FG_ERR_ALIGN, "dequant_g4: x must be 16-byte aligned");
    return fg::launch_dequant_g4(in->codes, in->meta, in->rows * (in->cols / 64), Hm(x), S(stream));
}

size_t fg_dequant_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return fg::plan_gemm(M, N, K).ws_bytes;
}

fg_status fg_dequant_gemm_g4(const fg_f16* X, int64_t M, const fg_q4* W, const fg_f16* bias,
                             const fg_f16* residual, int32_t act, fg_f16* Y, void* workspace,
                             size_t ws_bytes, fg_stream stream) {
    fg_status s = check_q4(W, "dequant_gemm_g4");
    if (s != FG_OK) return s;
    FG_REQUIRE(M >= 0, FG_ERR_SHAPE, "dequant_gemm_g4: M < 0");
    if (M == 0) return FG_OK;
    FG_REQUIRE(X != nullptr && Y != nullptr, FG_ERR_NULL, "dequant_gemm_g4: null X or Y");
    FG_REQUIRE(W->rows > 0 && W->rows % 16 == 0, FG_ERR_SHAPE,
               "dequant_gemm_g4: N = %lld must be a positive multiple of 16", (long long)W->rows);
    FG_REQUIRE(M < (1LL << 31) && W->rows < (1LL << 31) && W->cols < (1LL << 31),
               FG_ERR_SHAPE, "dequant_gemm_g4: sizes out of range");
    FG_REQUIRE(act == FG_ACT_NONE || act == FG_ACT_RELU, FG_ERR_SHAPE, "dequant_gemm_g4: bad act");
    FG_REQUIRE(fg::aligned16(X) && fg::aligned16(Y) && (!residual || fg::aligned16(residual)),
               FG_ERR_ALIGN, "dequant_gemm_g4: X, Y, residual must be 16-byte aligned");
    FG_REQUIRE(!residual || (residual != Y && residual != X), FG_ERR_SHAPE,
               "dequant_gemm_g4: residual may not alias X or Y");
    return fg::launch_gemm_g4(H(X), M, W, H(bias), H(residual), act, Hm(Y), workspace, ws_bytes,
                              S(stream));
}

fg_status fg_gemm_f16_f32out(const fg_f16* X, int64_t M, const fg_f16* W, int64_t N, int64_t K,
                             float* Y, fg_stream stream) {
    FG_REQUIRE(M >= 0 && N > 0 && K > 0 && K % 64 == 0 && M < (1LL << 31) && N < (1LL << 31),
               FG_ERR_SHAPE, "gemm_f16_f32out: need K %% 64 == 0");
    if (M == 0) return FG_OK;
    FG_REQUIRE(X && W && Y, FG_ERR_NULL, "gemm_f16_f32out: null pointer");
    FG_REQUIRE(fg::aligned16(X) && fg::aligned16(W) && fg::aligned16(Y), FG_ERR_ALIGN,
               "gemm_f16_f32out: pointers must be 16-byte aligned");
    return fg::launch_gemm_f16_f32out(H(X), M, H(W), N, K, Y, S(stream));
}

fg_status fg_layernorm(const fg_f16* x, int64_t rows, int64_t cols, int64_t x_ld,
                       const fg_f16* gamma, const fg_f16* beta, float eps, fg_f16* y,
                       fg_stream stream) {
    FG_REQUIRE(x && gamma && beta && y, FG_ERR_NULL, "layernorm: null pointer");
    FG_REQUIRE(rows >= 0 && cols > 0 && cols % 8 == 0 && x_ld >= cols && x_ld % 8 == 0,
               FG_ERR_SHAPE, "layernorm: need cols %% 8 == 0 and x_ld >= cols, x_ld %% 8 == 0");
    FG_REQUIRE(fg::aligned16(x) && fg::aligned16(y) && fg::aligned16(gamma) && fg::aligned16(beta),
               FG_ERR_ALIGN, "layernorm: pointers must be 16-byte aligned");
    return fg::launch_layernorm(H(x), rows, cols, x_ld, H(gamma), H(beta), eps, Hm(y), S(stream));
}

fg_status fg_embed(const int32_t* ids, int64_t ntok, int32_t T, int32_t pos0, const int32_t* pad,
                   const fg_f16* e_tok, int64_t vocab, const fg_f16* e_pos, int64_t npos,
                   int32_t h1, fg_f16* y, fg_stream stream) {
    FG_REQUIRE(ids && e_tok && e_pos && y, FG_ERR_NULL, "embed: null pointer");
    FG_REQUIRE(ntok >= 0 && T > 0 && ntok % T == 0 && pos0 >= 0 && h1 > 0 && h1 % 8 == 0 &&
                   vocab > 0 && pos0 + T <= npos,
               FG_ERR_SHAPE, "embed: bad sizes (ntok %lld, T %d, pos0 %d, npos %lld)",
               (long long)ntok, T, pos0, (long long)npos);
    FG_REQUIRE(fg::aligned16(e_tok) && fg::aligned16(e_pos) && fg::aligned16(y), FG_ERR_ALIGN,
               "embed: tables and y must be 16-byte aligned");
    return fg::launch_embed(ids, ntok, T, pos0, pad, H(e_tok), H(e_pos), h1, Hm(y), S(stream));
}

fg_status fg_argmax(const float* logits, int64_t B, int64_t V, int32_t* out, fg_stream stream) {
    FG_REQUIRE(B >= 0 && V > 0 && V < (1LL << 31) && B < (1LL << 31), FG_ERR_SHAPE,
               "argmax: bad sizes (B %lld, V %lld)", (long long)B, (long long)V);
    if (B == 0) return FG_OK;
    FG_REQUIRE(logits && out, FG_ERR_NULL, "argmax: null pointer");
    FG_REQUIRE((reinterpret_cast<uintptr_t>(logits) & 3u) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & 3u) == 0,
               FG_ERR_ALIGN, "argmax: pointers must be 4-byte aligned");
    return fg::launch_argmax(logits, B, V, out, S(stream));
}

fg_status fg_kv_append_g4(const fg_f16* qkv, int64_t qkv_ld, const fg_kv4* cache, int32_t pos,
                          fg_stream stream) {
    fg_status s = check_kv(cache, "kv_append_g4");
    if (s != FG_OK) return s;
    FG_REQUIRE(qkv != nullptr, FG_ERR_NULL, "kv_append_g4: null qkv");
    const int64_t h1 = static_cast<int64_t>(cache->H) * cache->d;
    FG_REQUIRE(qkv_ld >= 3 * h1 && qkv_ld % 8 == 0, FG_ERR_SHAPE,
               "kv_append_g4: qkv_ld %lld must be >= 3*h1 and a multiple of 8", (long long)qkv_ld);
    FG_REQUIRE(pos >= 0 && pos < cache->cap, FG_ERR_SHAPE, "kv_append_g4: pos %d outside [0, %d)",
               pos, cache->cap);
    FG_REQUIRE(fg::aligned16(qkv), FG_ERR_ALIGN, "kv_append_g4: qkv must be 16-byte aligned");
    return fg::launch_kv_store(H(qkv), qkv_ld, cache->B, 1, cache->H, cache->d, cache, pos,
                               S(stream));
}

fg_status fg_decode_attn_g4(const fg_f16* qkv, int64_t qkv_ld, const fg_kv4* cache, int32_t pos,
                            const int32_t* pad, int32_t fuse_append, fg_f16* out,
                            fg_stream stream) {
    fg_status s = check_kv(cache, "decode_attn_g4");
    if (s != FG_OK) return s;
    FG_REQUIRE(qkv && out, FG_ERR_NULL, "decode_attn_g4: null qkv or out");
    const int64_t h1 = static_cast<int64_t>(cache->H) * cache->d;
    FG_REQUIRE(qkv_ld >= 3 * h1 && qkv_ld % 8 == 0, FG_ERR_SHAPE,
               "decode_attn_g4: qkv_ld %lld must be >= 3*h1 and a multiple of 8", (long long)qkv_ld);
    FG_REQUIRE(pos >= 0 && pos < cache->cap, FG_ERR_SHAPE,
               "decode_attn_g4: pos %d outside [0, %d)", pos, cache->cap);
    FG_REQUIRE(cache->cap <= 50000, FG_ERR_UNSUPPORTED, "decode_attn_g4: cap %d > 50000", cache->cap);
    FG_REQUIRE(fg::aligned16(qkv) && fg::aligned16(out), FG_ERR_ALIGN,
               "decode_attn_g4: qkv and out must be 16-byte aligned");
    FG_REQUIRE((reinterpret_cast<uintptr_t>(pad) & 3u) == 0, FG_ERR_ALIGN,
               "decode_attn_g4: pad must be 4-byte aligned");
    return fg::launch_decode_attn(H(qkv), qkv_ld, cache, pos, pad, fuse_append, Hm(out),
                                  S(stream));
}

size_t fg_decode_attn_topk_workspace_bytes(int32_t B, int32_t H, int32_t pos) {
    if (B < 0 || H <= 0 || pos < 0) return 0;
    return fg::decode_topk_ws_bytes(B, H, pos);
}

fg_status fg_decode_attn_topk_g4(const fg_f16* qkv, int64_t qkv_ld, const fg_kv4* cache,
                                 int32_t pos, const int32_t* pad, int32_t keep_pct,
                                 int32_t fuse_append, fg_f16* out, int32_t* sel_out,
                                 void* workspace, size_t ws_bytes, fg_stream stream) {
    fg_status s = check_kv(cache, "decode_attn_topk_g4");
    if (s != FG_OK) return s;
    FG_REQUIRE(qkv && out, FG_ERR_NULL, "decode_attn_topk_g4: null qkv or out");
    const int64_t h1 = static_cast<int64_t>(cache->H) * cache->d;
    FG_REQUIRE(qkv_ld >= 3 * h1 && qkv_ld % 8 == 0, FG_ERR_SHAPE,
               "decode_attn_topk_g4: qkv_ld %lld must be >= 3*h1 and a multiple of 8", (long long)qkv_ld);
    FG_REQUIRE(pos >= 0 && pos < cache->cap, FG_ERR_SHAPE,
               "decode_attn_topk_g4: pos %d outside [0, %d)", pos, cache->cap);
    FG_REQUIRE(keep_pct >= 1 && keep_pct <= 100, FG_ERR_SHAPE,
               "decode_attn_topk_g4: keep_pct %d outside [1, 100]", keep_pct);
    FG_REQUIRE(cache->cap <= 50000, FG_ERR_UNSUPPORTED, "decode_attn_topk_g4: cap %d > 50000", cache->cap);
    FG_REQUIRE(fg::aligned16(qkv) && fg::aligned16(out), FG_ERR_ALIGN,
               "decode_attn_topk_g4: qkv and out must be 16-byte aligned");
    FG_REQUIRE((reinterpret_cast<uintptr_t>(pad) & 3u) == 0 &&
                   (reinterpret_cast<uintptr_t>(sel_out) & 3u) == 0,
               FG_ERR_ALIGN, "decode_attn_topk_g4: pad and sel_out must be 4-byte aligned");
    FG_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, FG_ERR_ALIGN,
               "decode_attn_topk_g4: workspace must be 256-byte aligned");
    return fg::launch_decode_attn_topk(H(qkv), qkv_ld, cache, pos, pad, fuse_append, keep_pct,
                                       sel_out, workspace, ws_bytes, Hm(out), S(stream));
}

int32_t fg_topk_count(int32_t n, int32_t keep_pct) {
    if (n < 0 || keep_pct < 1 || keep_pct > 100) return -1;
    return static_cast<int32_t>((static_cast<int64_t>(n) * keep_pct + 99) / 100);
}

fg_status fg_prefill_attn(const fg_f16* qkv, int32_t B, int32_t s_len, int32_t Hh, int32_t d,
                          const int32_t* pad, const fg_kv4* cache, fg_f16* out,
                          fg_stream stream) {
    FG_REQUIRE(qkv && out, FG_ERR_NULL, "prefill_attn: null qkv or out");
    FG_REQUIRE(B >= 0 && s_len >= 0 && Hh > 0, FG_ERR_SHAPE, "prefill_attn: bad B/s/H");
    FG_REQUIRE(d == 64 || d == 128, FG_ERR_UNSUPPORTED, "prefill_attn: head dim %d not in {64,128}", d);
    FG_REQUIRE(fg::aligned16(qkv) && fg::aligned16(out), FG_ERR_ALIGN,
               "prefill_attn: qkv and out must be 16-byte aligned");
    if (cache) {
        fg_status s = check_kv(cache, "prefill_attn");
        if (s != FG_OK) return s;
        FG_REQUIRE(cache->B == B && cache->H == Hh && cache->d == d && s_len <= cache->cap,
                   FG_ERR_SHAPE, "prefill_attn: cache shape does not match");
    }
    FG_REQUIRE((reinterpret_cast<uintptr_t>(pad) & 3u) == 0, FG_ERR_ALIGN,
               "prefill_attn: pad must be 4-byte aligned");
    fg_status s = fg::launch_prefill_attn(H(qkv), B, s_len, Hh, d, pad, Hm(out), S(stream));
    if (s != FG_OK || !cache) return s;
    return fg::launch_kv_store(H(qkv), 3LL * Hh * d, B, s_len, Hh, d, cache, 0, S(stream));
}

size_t fg_layer_workspace_bytes(const fg_layer* w, int32_t phase, int32_t bls, int32_t T,
                                int32_t cap, fg_policy p) {
    if (!w || bls <= 0 || T <= 0 || p.gbs <= 0 || p.k <= 0 || w->H <= 0) return 0;
    const int64_t rows = static_cast<int64_t>(bls) * T;
    const int64_t per = p.order == FG_ORDER_BLOCK ? rows : static_cast<int64_t>(p.gbs) * T;
    const size_t tk = cap > 0 ? topk_scratch(phase, p.topk_pct, per / T, w->H, cap - 1) : 0;
    return layer_ws_layout(w, rows, per, nullptr, tk).total;
}

fg_status fg_layer_step(const fg_layer* w, const fg_kv4* cache, const fg_f16* x_in, fg_f16* x_out,
                        int32_t phase, int32_t T, int32_t pos, const int32_t* pad, fg_policy p,
                        void* workspace, size_t ws_bytes, fg_stream stream) {
    fg_status s = check_kv(cache, "layer_step");
    if (s != FG_OK) return s;
    return layer_step_impl(w, cache, x_in, x_out, phase, T, pos, pad, p, workspace, ws_bytes, stream);
}

fg_status fg_layer_step_kv16(const fg_layer* w, const fg_kv16* cache, const fg_f16* x_in,
                             fg_f16* x_out, int32_t phase, int32_t T, int32_t pos,
                             const int32_t* pad, fg_policy p, void* workspace, size_t ws_bytes,
                             fg_stream stream) {
    fg_status s = check_kv16(cache, "layer_step_kv16");
    if (s != FG_OK) return s;
    FG_REQUIRE(p.topk_pct == 0, FG_ERR_UNSUPPORTED,
               "layer_step_kv16: top-K attention (topk_pct %d) needs the 4-bit cache", p.topk_pct);
    FG_REQUIRE(cache->cap <= 50000, FG_ERR_UNSUPPORTED, "layer_step_kv16: cap %d > 50000", cache->cap);
    return layer_step_impl(w, cache, x_in, x_out, phase, T, pos, pad, p, workspace, ws_bytes, stream);
}

fg_status fg_kv_store_f16(const fg_f16* qkv, int64_t qkv_ld, int32_t T, const fg_kv16* cache,
                          int32_t slot0, fg_stream stream) {
    fg_status s = check_kv16(cache, "kv_store_f16");
    if (s != FG_OK) return s;
    FG_REQUIRE(qkv != nullptr, FG_ERR_NULL, "kv_store_f16: null qkv");
    const int64_t h1 = static_cast<int64_t>(cache->H) * cache->d;
    FG_REQUIRE(qkv_ld >= 3 * h1 && qkv_ld % 8 == 0, FG_ERR_SHAPE,
               "kv_store_f16: qkv_ld %lld must be >= 3*h1 and a multiple of 8", (long long)qkv_ld);
    FG_REQUIRE(T >= 0 && slot0 >= 0 && static_cast<int64_t>(slot0) + T <= cache->cap, FG_ERR_SHAPE,
               "kv_store_f16: slots [%d, %d + %d) outside [0, %d)", slot0, slot0, T, cache->cap);
    FG_REQUIRE(fg::aligned16(qkv), FG_ERR_ALIGN, "kv_store_f16: qkv must be 16-byte aligned");
    return fg::launch_kv_store_f16(H(qkv), qkv_ld, T, cache, slot0, S(stream));
}

fg_status fg_decode_attn_f16(const fg_f16* qkv, int64_t qkv_ld, const fg_kv16* cache, int32_t pos,
                             const int32_t* pad, int32_t fuse_append, fg_f16* out,
                             fg_stream stream) {
    fg_status s = check_kv16(cache, "decode_attn_f16");
    if (s != FG_OK) return s;
    FG_REQUIRE(qkv && out, FG_ERR_NULL, "decode_attn_f16: null qkv or out");
    const int64_t h1 = static_cast<int64_t>(cache->H) * cache->d;
    FG_REQUIRE(qkv_ld >= 3 * h1 && qkv_ld % 8 == 0, FG_ERR_SHAPE,
               "decode_attn_f16: qkv_ld %lld must be >= 3*h1 and a multiple of 8", (long long)qkv_ld);
    FG_REQUIRE(pos >= 0 && pos < cache->cap, FG_ERR_SHAPE,
               "decode_attn_f16: pos %d outside [0, %d)", pos, cache->cap);
    FG_REQUIRE(cache->cap <= 50000, FG_ERR_UNSUPPORTED, "decode_attn_f16: cap %d > 50000", cache->cap);
    FG_REQUIRE(fg::aligned16(qkv) && fg::aligned16(out), FG_ERR_ALIGN,
               "decode_attn_f16: qkv and out must be 16-byte aligned");
    FG_REQUIRE((reinterpret_cast<uintptr_t>(pad) & 3u) == 0, FG_ERR_ALIGN,
               "decode_attn_f16: pad must be 4-byte aligned");
    return fg::launch_decode_attn_f16(H(qkv), qkv_ld, cache, pos, pad, fuse_append, Hm(out),
                                      S(stream));
}

}  // extern "C"
