/*
 * fg.h -- C ABI of libfg: the GB300 (sm_103a) hot path of 4-bit group-
 * quantised, block-scheduled OPT decoding.
 *
 * What the library computes is defined on the pages it follows:
 *   "FlexGen 完全拆解" (pinghaoyang.com.cn), sections
 *     - "权重压缩与 KV Cache 压缩": group-wise asymmetric min/max 4-bit
 *       quantisation of weights and KV cache, groups of 64 contiguous
 *       values, dequantisation to FP16 before compute;
 *     - "从 Transformer 推理的数据流重新定义卸载": prefill Q, K, V
 *       projections of all prompt tokens; each decode step appends one K/V
 *       row and attends one query over s+t cached rows;
 *     - "FlexGen 的核心：计算图分块与张量生命周期": the zig-zag block schedule,
 *       one layer's weights kept while the k GPU batches of a block
 *       (bls = gbs * k sequences) pass through it;
 *   "bjbfmj.com/news/40234", section 6.3: two 4-bit codes per byte plus a
 *   per-group scale tensor.
 *
 * Conventions shared by every call
 *  - Pointers are DEVICE pointers unless stated otherwise; struct arguments
 *    themselves live in host memory and are read before the call returns.
 *  - The caller owns every buffer.  No call allocates or frees device
 *    memory; scratch space comes from a caller-provided workspace sized by
 *    the matching *_workspace_bytes query.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *  - Host-side validation runs before any launch; on failure nothing is
 *    launched and a status is returned.  fg_last_error() gives a one-line
 *    detail for the calling thread.  A failed launch returns FG_ERR_CUDA.
 *  - Device-side waits are bounded.  A wait that expires records
 *    FG_ERR_TIMEOUT in a per-device status word that fg_check() returns
 *    and clears; until then, launches that wait on the device skip their
 *    work (their outputs are unspecified).
 *  - fp16 tensors are IEEE binary16, passed as fg_f16 (uint16_t bit
 *    patterns, layout-identical to CUDA's __half).
 *  - 4-bit layout (part of the ABI): for a [rows][cols] tensor grouped
 *    along cols in groups of 64, codes are [rows][cols/2] bytes, element 2j
 *    in the low nibble of byte j and element 2j+1 in the high nibble; meta
 *    is [rows][cols/64][2] fp32 = (min, scale) per group.
 *  - Inputs must be finite; NaN or Inf inputs give unspecified outputs.
 *  - Left padding (prompts of different lengths in one block, padded to the
 *    common length s as the pages' workloads are, "FlexGen 完全拆解",
 *    section on reading the experimental results).  Calls that take
 *    `const int32_t* pad` accept NULL (no padding) or a DEVICE array of one
 *    count per sequence, 4-byte aligned: sequence b's prompt occupies slots
 *    pad[b]..s-1, its tokens take positions counted from slot pad[b],
 *    every query attends only keys at slots >= pad[b], and prefill queries
 *    in padding slots output zeros.  A padded prompt gives the results of
 *    the same prompt run unpadded.  The counts are read on the device and
 *    cannot be validated on the host: a count outside [0, s) (or, at decode,
 *    [0, pos]) is clamped into that range, never read out of bounds.
 */
#ifndef FG_H
#define FG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t fg_f16;                 /* IEEE binary16 bit pattern */
typedef struct CUstream_st* fg_stream;   /* same type as cudaStream_t */

typedef enum fg_status {
    FG_OK = 0,
    FG_ERR_NULL = 1,         /* a required pointer is NULL */
    FG_ERR_SHAPE = 2,        /* a size or index is outside what the call supports */
    FG_ERR_ALIGN = 3,        /* a pointer or leading dimension is misaligned */
    FG_ERR_UNSUPPORTED = 4,  /* valid request this build does not implement */
    FG_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
    FG_ERR_TIMEOUT = 6,      /* a bounded device-side wait expired */
    FG_ERR_WORKSPACE = 7     /* workspace missing or smaller than required */
} fg_status;

/* 4-bit group-quantised matrix [rows][cols], grouped along cols (for a
 * weight in torch Linear layout [out][in], cols = in = the contraction
 * dimension K).  cols % 64 == 0.  codes and meta are 16-byte aligned. */
typedef struct fg_q4 {
    uint8_t* codes;   /* [rows][cols/2] */
    float* meta;      /* [rows][cols/64][2] = (min, scale) */
    int64_t rows;
    int64_t cols;
} fg_q4;

/* One layer's 4-bit KV cache for B sequences, H heads of size d, cap slots.
 * codes [B][H][cap][d/2], meta [B][H][cap][d/64][2]; grouped along the head
 * dimension (64 values per group).  d in {64, 128}. */
typedef struct fg_kv4 {
    uint8_t* k_codes;
    uint8_t* v_codes;
    float* k_meta;
    float* v_meta;
    int32_t B, H, d, cap;
} fg_kv4;

/* One layer's uncompressed KV cache (the setting the pages compare the 4-bit
 * cache against, "FlexGen 完全拆解", results for input length 512): k and v
 * fp16 [B][H][cap][d], each row as the QKV projection produced it.  d in
 * {64, 128}; k and v 16-byte aligned. */
typedef struct fg_kv16 {
    fg_f16* k;
    fg_f16* v;
    int32_t B, H, d, cap;
} fg_kv16;

/* Block schedule: bls = gbs * k sequences per block.
 * order FG_ORDER_BLOCK: each projection is ONE launch over all bls rows, so
 *   each weight tile is fetched from HBM and dequantised once per block.
 * order FG_ORDER_BATCHES / FG_ORDER_BATCHES_REV: the k GPU batches run as k
 *   launches per projection in ascending / descending batch order (the
 *   zig-zag schedule alternates the two at each token step).
 * Every order gives bit-identical results: every launch of a block plans
 * its K split from the block's row count (bls * T), so the batches and the
 * whole block sum each output in the same order. */
enum { FG_ORDER_BLOCK = 0, FG_ORDER_BATCHES = 1, FG_ORDER_BATCHES_REV = 2 };
/* topk_pct: 0 (or 100) for dense decode attention; 1..99 runs each decode
 * step's attention as fg_decode_attn_topk_g4 at that percentage (the prefill
 * stays dense; the layer workspace then holds the scores).  (ABI 3.0 added
 * this field.) */
typedef struct fg_policy {
    int32_t gbs;
    int32_t k;
    int32_t order;
    int32_t topk_pct;
} fg_policy;

/* One OPT decoder layer (pre-LayerNorm, ReLU FFN).  qkv: [3*h1][h1] with
 * rows q | k | v (head h = rows [h*d, (h+1)*d) of each block); out [h1][h1];
 * fc1 [h2][h1]; fc2 [h1][h2]; biases and LayerNorm parameters fp16. */
typedef struct fg_layer {
    fg_q4 qkv, out, fc1, fc2;
    const fg_f16 *b_qkv, *b_out, *b_fc1, *b_fc2;
    const fg_f16 *ln1_g, *ln1_b, *ln2_g, *ln2_b;
    int32_t h1, H, h2;
    float ln_eps;
} fg_layer;

enum { FG_PHASE_PREFILL = 0, FG_PHASE_DECODE = 1 };
enum { FG_ACT_NONE = 0, FG_ACT_RELU = 1 };

/* ------------------------------------------------------------------ misc */

const char* fg_status_str(fg_status s);
/* Detail of the calling thread's last failed call ("" if none). */
const char* fg_last_error(void);
/* ABI version: (major << 16) | minor. */
int32_t fg_version(void);
/* Synchronise `stream`, then read and clear the current device's status
 * word: FG_ERR_TIMEOUT if a bounded device wait expired since the last
 * check, FG_ERR_CUDA if the stream reports an error, else FG_OK. */
fg_status fg_check(fg_stream stream);

/* ------------------------------------------------------------------ quantiser */

/* Group-wise 4-bit quantisation ("FlexGen 完全拆解", section on weight and
 * KV-cache compression; packing per "bjbfmj.com/news/40234" section 6.3).
 * For each group of 64 consecutive values of a row: m = min, M = max (fp32,
 * IEEE total order, -0 below +0); scale = (M - m) / 15 (IEEE fp32 divide);
 * code = clamp(rint((x - m) / scale), 0, 15), all codes 0 when scale == 0.
 * x: [rows][cols] fp16, 16-byte aligned; cols % 64 == 0.
 * out: rows/cols must equal (rows, cols); codes/meta 16-byte aligned.
 * Bit-exact: identical codes, meta and bytes to the reference definition. */
fg_status fg_quantize_g4(const fg_f16* x, int64_t rows, int64_t cols,
                         const fg_q4* out, fg_stream stream);

/* Dequantisation x^ = fp16(fma(code, scale, min)) (fp32 fused multiply-add,
 * one rounding to fp16).  Test and inspection utility: the hot path fuses
 * dequantisation into its consumers.  x: [rows][cols] fp16. */
fg_status fg_dequant_g4(const fg_q4* in, fg_f16* x, fg_stream stream);

/* ------------------------------------------------------------------ GEMMs */

/* Y = act(X W^T + bias) + residual, with W stored 4-bit (dequantised to
 * fp16 on chip, fp16 x fp16 products accumulated in fp32 on the tensor
 * cores, epilogue in fp32, one rounding to fp16).  This is every projection
 * of the decoder ("FlexGen 完全拆解", dataflow section: K = XW_K etc.).
 * X: [M][K] fp16 (K = W->cols), row stride K, 16-byte aligned.
 * W: [N][K] 4-bit (N = W->rows).  bias: [N] fp16 or NULL.
 * residual: [M][N] fp16 or NULL (may alias neither X nor Y), 16-byte
 * aligned (tiles of it are copied by TMA).
 * act: FG_ACT_NONE or FG_ACT_RELU (applied to acc + bias, before residual).
 * Y: [M][N] fp16, 16-byte aligned.  M >= 0 (M == 0 launches nothing);
 * N % 16 == 0.  FG_ERR_ALIGN for a misaligned X, Y or residual.
 * workspace: device scratch of at least
 * fg_dequant_gemm_workspace_bytes(M, N, K) bytes (NULL allowed when that is
 * 0), 256-byte aligned.  From M = 8192 rows that size is 2*N*K bytes: the
 * weights are dequantised once into it and the fp16 tensor-core pipeline
 * multiplies them (a prefill-sized block would otherwise dequantise every
 * weight tile once per 256 rows); with less (or NULL) the same product is
 * computed with the dequantisation fused per tile.
 * Each output is fp32-accumulated fp16(x) * fp16(w^) products with
 * w^ = fp16(fma(q, scale, min)) exactly as fg_dequant_g4 gives it.  The
 * result of a row never depends on the other rows; it depends on M only
 * through which regime M falls in -- at most 144 rows with K a multiple of
 * 256 (the dequantised weights go to TMEM and K is split over persistent
 * CTA clusters, parts summed in a fixed order), at most 256 rows (K split
 * across CTAs, fixed-order sum), more than 256 rows (whole tiles), 8192 rows
 * or more with the full workspace (fp16 weights) -- so launches in the same
 * regime agree bit for bit.  The K split depends on (N, K) and the device's
 * SM count.
 * In the first regime (at most 144 rows) the tiles split over clusters are
 * finished by the cluster holding their first part, which waits for the
 * later parts behind flags in the workspace; the grid is sized so that
 * every cluster can be resident at once.  If another context on the same
 * GPU keeps some clusters from being scheduled, those waits expire after
 * the bounded-wait limit and the call reports FG_ERR_TIMEOUT through
 * fg_check, with Y unspecified (never a hang). */
size_t fg_dequant_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
fg_status fg_dequant_gemm_g4(const fg_f16* X, int64_t M, const fg_q4* W,
                             const fg_f16* bias, const fg_f16* residual,
                             int32_t act, fg_f16* Y, void* workspace,
                             size_t ws_bytes, fg_stream stream);

/* The same computation as fg_dequant_gemm_g4, for callers that must not
 * allocate device memory: a plugin inside a host program that owns the
 * device-memory budget through its own pool and forbids other allocations,
 * or a latency-critical loop where cudaMalloc/cudaFree would synchronise the
 * device.  No counterpart in the paper: it exists only for such callers.
 * Inputs and outputs are as for fg_dequant_gemm_g4 (the caller still
 * passes X, W, bias, residual and Y); the K-split scratch comes from a
 * fixed 16 MiB device array inside the library (held on every GPU that
 * loads it until the process exits), so no workspace is passed and nothing
 * is allocated.  The call offers the GEMM only the scratch the shape cannot
 * do without, so M >= 8192 always takes the fused path (the weights are
 * never copied into the array as fp16).  Shapes whose K-split scratch
 * exceeds 16 MiB are rejected with FG_ERR_WORKSPACE before any launch.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the array and it keeps the
 * last call's contents.  No call relies on them: every partial sum read is
 * written earlier in the same call, and the decode kernel's fixup flags
 * carry a per-launch tag that also changes after fg_check reports a
 * timeout.  Calls that overlap on the GPU -- on different streams of one
 * device -- race on it and must be serialised by the caller. */
fg_status fg_dequant_gemm_g4_noalloc(const fg_f16* X, int64_t M, const fg_q4* W,
                                     const fg_f16* bias, const fg_f16* residual,
                                     int32_t act, fg_f16* Y, fg_stream stream);

/* Y = X W^T with fp16 W [N][K] and an fp32 result (the LM head against the
 * tied token embedding).  X [M][K] fp16; Y [M][N] fp32; K % 64 == 0; any
 * N >= 1 (the vocabulary need not be a multiple of the tile). */
fg_status fg_gemm_f16_f32out(const fg_f16* X, int64_t M, const fg_f16* W,
                             int64_t N, int64_t K, float* Y, fg_stream stream);

/* ------------------------------------------------------------------ small ops */

/* y = (x - mean) / sqrt(var + eps) * gamma + beta per row; mean and biased
 * variance in fp32 (the OPT layer's pre-LayerNorm and final LayerNorm).
 * Row r of x starts at x + r * x_ld (x_ld >= cols, x_ld % 8 == 0), so the
 * last token of each sequence can be normalised in place; y: [rows][cols]
 * contiguous fp16.  cols % 8 == 0, cols <= 16384. */
fg_status fg_layernorm(const fg_f16* x, int64_t rows, int64_t cols,
                       int64_t x_ld, const fg_f16* gamma, const fg_f16* beta,
                       float eps, fg_f16* y, fg_stream stream);

/* y[r] = e_tok[ids[r]] + e_pos[p] for r in [0, ntok): the token embedding
 * plus the learned position embedding of sequence-major rows of T tokens in
 * slots pos0.., with p = max(pos0 + r % T - pad[r / T], 0) (pad NULL: p =
 * pos0 + r % T).  ids: [ntok] int32 in [0, vocab).  pad: NULL or [ntok / T].
 * e_tok [vocab][h1], e_pos [npos][h1], y [ntok][h1] fp16; h1 % 8 == 0;
 * pos0 + T <= npos. */
fg_status fg_embed(const int32_t* ids, int64_t ntok, int32_t T, int32_t pos0,
                   const int32_t* pad, const fg_f16* e_tok, int64_t vocab,
                   const fg_f16* e_pos, int64_t npos, int32_t h1, fg_f16* y,
                   fg_stream stream);

/* Greedy choice of the next token: out[b] = the index of the largest of
 * logits[b][0..V), the lowest such index when several are equal (so the
 * result does not depend on the order of the reduction).  logits: [B][V]
 * fp32, out: [B] int32, both device, 4-byte aligned.  1 <= V < 2^31. */
fg_status fg_argmax(const float* logits, int64_t B, int64_t V, int32_t* out,
                    fg_stream stream);

/* ------------------------------------------------------------------ KV cache and attention */

/* Quantise the new token's k and v (one row per sequence) into cache slot
 * pos, per head, in groups of 64 along the head dimension (the decode-step
 * append of "FlexGen 完全拆解", dataflow section).  qkv: [B][qkv_ld] fp16
 * holding q | k | v of width h1 = H*d each; qkv_ld >= 3*h1, qkv_ld % 8 == 0.
 * 0 <= pos < cap.  Bit-exact with fg_quantize_g4 on the same values. */
fg_status fg_kv_append_g4(const fg_f16* qkv, int64_t qkv_ld,
                          const fg_kv4* cache, int32_t pos, fg_stream stream);

/* Decode attention over the 4-bit cache: for each sequence b and head h,
 * out = sum_j softmax_j(q . k^_j / sqrt(d)) v^_j over slots j = pad[b]..pos
 * (pad NULL: 0..pos), with k^, v^ the dequantised cache rows.  If
 * fuse_append != 0 the new k, v are first appended into slot pos exactly as
 * fg_kv_append_g4 does (in the same launch).  qkv as for fg_kv_append_g4;
 * pad: NULL or [B]; out: [B][h1] fp16. */
fg_status fg_decode_attn_g4(const fg_f16* qkv, int64_t qkv_ld,
                            const fg_kv4* cache, int32_t pos,
                            const int32_t* pad, int32_t fuse_append,
                            fg_f16* out, fg_stream stream);

/* Top-K sparse decode attention over the 4-bit cache ("FlexGen 完全拆解",
 * section on the paper's further approximations: the scores of every cached
 * key are computed, and only the V rows with the highest scores are loaded).
 * For each sequence b and head h with n = pos + 1 - pad[b] attended slots:
 * the scores s_j = q . k^_j / sqrt(d) and the full softmax weights
 * p_j = exp(s_j - max s) / sum_all exp(s - max s) over all n slots, as in
 * fg_decode_attn_g4; the kept set S = the fg_topk_count(n, keep_pct) slots
 * with the highest fp32 scores (equal scores: lower slot first); and
 * out = sum_{j in S} p_j v^_j -- rows outside S add nothing, the weights are
 * not renormalised over S.  Only the V rows of S are read from memory.
 * Two launches: a scores pass over K (the append fused) writes every score
 * to the workspace, then one warp per (b, h) selects and gathers.
 * keep_pct in [1, 100]; 100 keeps every row (the result then agrees with
 * fg_decode_attn_g4 within rounding).  sel_out: NULL, or device
 * [B][H][kmax] int32 with kmax = fg_topk_count(pos + 1, keep_pct),
 * receiving each (b, h)'s kept slots ascending, -1 after its own count.
 * workspace: device scratch of at least
 * fg_decode_attn_topk_workspace_bytes(B, H, pos) bytes, 256-byte aligned,
 * owned by the caller.  Other arguments, layouts and fusion as for
 * fg_decode_attn_g4.  Errors: FG_ERR_SHAPE for keep_pct outside [1, 100];
 * FG_ERR_ALIGN if pad or sel_out is not 4-byte aligned or the workspace
 * not 256-byte aligned; FG_ERR_WORKSPACE if it is missing or too small;
 * FG_ERR_UNSUPPORTED if the kept list exceeds the selecting warps' shared
 * memory (more than about 6,600 kept slots). */
size_t fg_decode_attn_topk_workspace_bytes(int32_t B, int32_t H, int32_t pos);
fg_status fg_decode_attn_topk_g4(const fg_f16* qkv, int64_t qkv_ld,
                                 const fg_kv4* cache, int32_t pos,
                                 const int32_t* pad, int32_t keep_pct,
                                 int32_t fuse_append, fg_f16* out,
                                 int32_t* sel_out, void* workspace,
                                 size_t ws_bytes, fg_stream stream);

/* Rows kept by top-K attention out of n: ceil(n * keep_pct / 100) (at least
 * one for n >= 1).  Returns -1 for n < 0 or keep_pct outside [1, 100]. */
int32_t fg_topk_count(int32_t n, int32_t keep_pct);

/* Store rows of k and v into the fp16 cache: token t (0 <= t < T) of
 * sequence b, row b*T + t of qkv ([B*T][qkv_ld] fp16 holding q | k | v of
 * width h1 = H*d each), goes to slot slot0 + t of sequence b, copied as is.
 * qkv_ld >= 3*h1, qkv_ld % 8 == 0; qkv 16-byte aligned; 0 <= slot0 and
 * slot0 + T <= cap.  The prefill stores T = s rows at slot 0; a decode step
 * that does not fuse its append stores T = 1 row at slot pos. */
fg_status fg_kv_store_f16(const fg_f16* qkv, int64_t qkv_ld, int32_t T,
                          const fg_kv16* cache, int32_t slot0, fg_stream stream);

/* Decode attention over the fp16 cache: for each sequence b and head h,
 * out = sum_j softmax_j(q . k_j / sqrt(d)) v_j over slots j = pad[b]..pos
 * (pad NULL: 0..pos), the rows read as stored.  If fuse_append != 0 the new
 * k, v rows (qkv row b) are first stored into slot pos, as fg_kv_store_f16
 * with T = 1 does, in the same launch.  qkv as for fg_kv_store_f16 with
 * B = cache->B rows; pad: NULL or [B] (4-byte aligned); out: [B][h1] fp16,
 * 16-byte aligned.  0 <= pos < cap <= 50000.  Device waits are bounded and
 * report FG_ERR_TIMEOUT through fg_check. */
fg_status fg_decode_attn_f16(const fg_f16* qkv, int64_t qkv_ld,
                             const fg_kv16* cache, int32_t pos,
                             const int32_t* pad, int32_t fuse_append,
                             fg_f16* out, fg_stream stream);

/* Causal prefill attention for B sequences of s prompt tokens over the fp16
 * K, V straight from the QKV projection: out_i = sum_{pad[b]<=j<=i}
 * softmax_j(q_i . k_j / sqrt(d)) v_j for slots i >= pad[b], and out_i = 0
 * for padding slots i < pad[b] (pad NULL: no padding).  qkv: [B*s][3*h1]
 * fp16 (sequence-major rows); pad: NULL or [B]; out: [B*s][h1] fp16.  If
 * cache is not NULL, the K and V rows of every slot are also quantised into
 * slots 0..s-1 (s <= cap, cache->B == B, H and d must match). */
fg_status fg_prefill_attn(const fg_f16* qkv, int32_t B, int32_t s, int32_t H,
                          int32_t d, const int32_t* pad, const fg_kv4* cache,
                          fg_f16* out, fg_stream stream);

/* ------------------------------------------------------------------ layer step */

/* One decoder layer for bls = p.gbs * p.k sequences of T new tokens:
 *   h = x + OutProj(Attn(LN1(x)));  y = h + FC2(ReLU(FC1(LN2(h)))).
 * phase FG_PHASE_PREFILL: T = s prompt tokens in slots 0..T-1 (the K/V rows
 * are stored into slots 0..T-1).  phase FG_PHASE_DECODE: T = 1; the new
 * token's K/V are appended at slot pos and attended over slots pad[b]..pos.
 * pad: NULL or [bls] left-padding counts (the attention masks; the layer
 * is otherwise row-wise, so positions enter only through fg_embed).
 * x_in, x_out: [bls*T][h1] fp16, sequence-major rows (may not alias).
 * cache->B must equal bls.  The k GPU batches are rows / cache sequences
 * [i*gbs, (i+1)*gbs).  workspace: device scratch of at least
 * fg_layer_workspace_bytes(w, phase, bls, T, cap, p) bytes, 256-byte
 * aligned, cap the cache capacity (it sizes the scores of top-K decode
 * attention, p.topk_pct in 1..99; otherwise it may be 0). */
size_t fg_layer_workspace_bytes(const fg_layer* w, int32_t phase, int32_t bls,
                                int32_t T, int32_t cap, fg_policy p);
fg_status fg_layer_step(const fg_layer* w, const fg_kv4* cache,
                        const fg_f16* x_in, fg_f16* x_out, int32_t phase,
                        int32_t T, int32_t pos, const int32_t* pad,
                        fg_policy p, void* workspace, size_t ws_bytes,
                        fg_stream stream);

/* fg_layer_step over the uncompressed fp16 cache: the same layer, schedule,
 * workspace and errors, with the prefill storing the K/V rows as
 * fg_kv_store_f16 does and each decode step attending as fg_decode_attn_f16
 * does (append fused).  p.topk_pct must be 0 (top-K attention is an option
 * of the 4-bit cache; FG_ERR_UNSUPPORTED otherwise). */
fg_status fg_layer_step_kv16(const fg_layer* w, const fg_kv16* cache,
                             const fg_f16* x_in, fg_f16* x_out, int32_t phase,
                             int32_t T, int32_t pos, const int32_t* pad,
                             fg_policy p, void* workspace, size_t ws_bytes,
                             fg_stream stream);

/* ------------------------------------------------------------------ tracing */

/* Kernel classes for tracing (bit mask). */
enum {
    FG_TRACE_GEMM_PREFILL = 1 << 0,  /* dequant GEMM launches with M > 256 rows */
    FG_TRACE_GEMM_DECODE = 1 << 1,   /* dequant GEMM launches with M <= 256 rows */
    FG_TRACE_ATTN_DECODE = 1 << 2,
    FG_TRACE_ATTN_PREFILL = 1 << 3,
    FG_TRACE_OTHER = 1 << 4,         /* quantiser, KV store, LayerNorm, embedding, LM head, reductions */
    FG_TRACE_NCLASS = 5
};

/* Per-class totals since the last fg_trace_begin. */
typedef struct fg_trace_stats {
    int64_t launches[FG_TRACE_NCLASS];   /* kernel launches, counted on the host */
    double ms[FG_TRACE_NCLASS];          /* summed device time of the timed classes */
    double flops[FG_TRACE_NCLASS];       /* algorithmic FLOPs of the launches */
    double bytes[FG_TRACE_NCLASS];       /* algorithmic HBM bytes of the launches */
} fg_trace_stats;

/* Start counting launches of every class and, for the classes in
 * `timed_mask`, record a CUDA event pair around each launch on its stream.
 * Host-side only; nothing is allocated on the device (CUDA events are
 * created once and reused). */
fg_status fg_trace_begin(int32_t timed_mask);
/* Stop, wait for the recorded events and return the totals. */
fg_status fg_trace_end(fg_trace_stats* out);

/* ------------------------------------------------------------------ test knobs */

/* Host-side test knobs (0 = off).  FG_KNOB_DROP_ARRIVE: the next
 * fg_dequant_gemm_g4 launch makes its producer skip one barrier arrive, so
 * the consumers' bounded waits expire and the launch reports
 * FG_ERR_TIMEOUT through fg_check() instead of hanging.
 * FG_KNOB_WAIT_NS: override the device wait limit in nanoseconds (0 =
 * default, about 2 s). */
enum { FG_KNOB_DROP_ARRIVE = 1, FG_KNOB_WAIT_NS = 2 };
fg_status fg_debug_set(int32_t knob, int64_t value);

#ifdef __cplusplus
}
#endif

#endif /* FG_H */
