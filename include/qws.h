/*
 * qws.h -- quantized weight streaming for single-token decode on GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels that multiply packed GGUF-style
 * weight matrices (Q4_K, Q6_K, Q4_0) by f32 activation vectors, decoding the
 * blocks in registers as they stream from HBM.  The calls restate the compute
 * backend of the "infer" project (crates/infer-compute/README.md, §Quick Start:
 * q4k_matvec(W, x, rows, hidden), decode_token(layers, x, hidden, inter, q_dim,
 * kv_dim, ...); §Shaders: q4k_matvec, q6k_matvec, Q4_0 matvec, q4k_qkv_proj,
 * q4k_ffn_gate_up, q4k_geglu_gelu_tanh_down, rms_norm, residual_add).
 *
 * Conventions shared by every call
 *  - Pointers named W*, x, y, h, q, k, v, w_* and ws are DEVICE pointers owned
 *    by the caller (for example torch tensors' data_ptr()).  The library never
 *    allocates, frees or retains them.  `layers` and `dims` are HOST pointers,
 *    read during the call only.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *    is asynchronous on that stream: a QWS_OK return means the work was
 *    enqueued.  Calls that overlap on the GPU must not share output or
 *    workspace buffers.
 *  - Weight layout: row-major; row r is the contiguous run of hidden/QK blocks
 *    that covers columns 0..hidden-1 (QK = 256 for Q4_K and Q6_K, 32 for
 *    Q4_0).  Block layouts are the public GGUF ones:
 *        Q4_K 144 B: f16 d, f16 dmin, 12 B packed 6-bit scales/mins, 128 B nibbles
 *        Q6_K 210 B: 128 B low nibbles, 64 B high 2-bit fields, 16 int8 scales, f16 d
 *        Q4_0  18 B: f16 d, 16 B nibbles
 *  - Activations: x is f32 [batch][hidden], y is f32 [batch][rows], both
 *    row-major and dense.
 *  - Accuracy: every result is an f32 accumulation of exact products; it stays
 *    within 1e-5 * sum_i |w_i x_i| of the exact value per output for |x| in
 *    [2^-66, 2^38] (outside that range products lose bits or overflow).
 *  - Errors: arguments are checked on the host before anything is enqueued.
 *      QWS_ERR_NULL      a required pointer is NULL
 *      QWS_ERR_SHAPE     a size is negative, zero where it may not be, or not a
 *                        multiple of 256 (hidden / inter), or above a limit
 *      QWS_ERR_ALIGN     W* not 16-byte aligned, or an f32 pointer not 4-byte aligned
 *      QWS_ERR_FORMAT    unknown qws_format
 *      QWS_ERR_WORKSPACE ws NULL or ws_bytes below qws_workspace_bytes(...)
 *      QWS_ERR_CUDA      the CUDA runtime refused the launch (message in
 *                        qws_last_error())
 *    Nothing is enqueued when a call returns an error.  rows == 0 returns
 *    QWS_OK without a launch.  A bounded wait that expires inside a kernel
 *    (a wedged pipeline) records a code that qws_device_error() returns.
 *  - Limits: every consumer thread owns one lane unit of 64 columns:
 *    batch * hidden / 64 <= 320 per pass, so hidden <= 20480 at batch 1 and
 *    hidden <= 2560 at batch 8; larger products need split_k (qws_matvec,
 *    qws_q4_0_matvec), which divides hidden into column slices.  The
 *    decode-once kernel for 2..8 vectors (Q4_0 and Q4_K weights, or the
 *    8-bit path) has no lane limit; it takes hidden % 256 == 0, <= 3072.
 */
#ifndef QWS_H
#define QWS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* qws_stream; /* = cudaStream_t */

typedef enum {
  QWS_OK = 0,
  QWS_ERR_NULL = 1,
  QWS_ERR_SHAPE = 2,
  QWS_ERR_ALIGN = 3,
  QWS_ERR_FORMAT = 4,
  QWS_ERR_WORKSPACE = 5,
  QWS_ERR_CUDA = 6,
  QWS_ERR_TIMEOUT = 7
} qws_status;

/* GGUF type ids. */
typedef enum { QWS_Q4_0 = 2, QWS_Q8_0 = 8, QWS_Q4_K = 12, QWS_Q6_K = 14 } qws_format;
/* QWS_Q8_0 is accepted only by the 8-bit path (qws_q8_matvec,
 * qws_q8_qkv_proj); the f32-activation entry points reject it. */

/* Operations for qws_workspace_bytes(). */
typedef enum {
  QWS_OP_MATVEC = 0,      /* qws_matvec / qws_q4_0_matvec with split_k > 1 */
  QWS_OP_FFN = 1,         /* qws_q4k_ffn_gate_up_geglu_down                */
  QWS_OP_DECODE_CHAIN = 2, /* qws_decode_chain                             */
  QWS_OP_PREFILL = 3,      /* qws_q4k_prefill_matmul (batch = n_tokens)     */
  QWS_OP_KV_ATTENTION = 4  /* qws_kv_attention: rows = n_ctx, hidden =
                              head_dim, inter = n_q_heads, batch = n_kv_heads */
} qws_op;

/* ------------------------------------------------------------------------
 * Quantized matrix-vector products.
 * infer-compute README §Quick Start "backend.q4k_matvec(&q4k_data, &x, rows,
 * hidden)" and §Shaders rows "Q4_0 matvec", "Q4_K/Q6_K" (q4k_matvec,
 * q6k_matvec):   y[b][r] = sum_i dequant(W)[r][i] * x[b][i].
 *   W      rows x hidden weights in `fmt` (device, 16-byte aligned)
 *   x      [batch][hidden] f32 (device, 4-byte aligned)
 *   y      [batch][rows]   f32 (device, 4-byte aligned), overwritten
 *   rows   >= 0;  hidden > 0, hidden % 256 == 0;  1 <= batch
 * ---------------------------------------------------------------------- */
qws_status qws_q4k_matvec(const void* W, const float* x, float* y, int64_t rows, int64_t hidden,
                          int batch, qws_stream stream);
qws_status qws_q6k_matvec(const void* W, const float* x, float* y, int64_t rows, int64_t hidden,
                          int batch, qws_stream stream);

/* Q4_0 matvec with an optional split-K path (the 262144-row lm_head).
 *   split_k  0 = library choice, 1 = single pass, S > 1 = S partial sums over
 *            hidden slices of hidden/S columns (S must divide hidden/256),
 *            written to the workspace and then added in a fixed order, so
 *            results are run-to-run identical.
 *   With 2..8 vectors, hidden <= 3072 and split_k 0 or 1, Q4_0 and Q4_K
 *   run a kernel that decodes each weight once for all vectors (tensor-core
 *   products of the exact codes with x split into two f16 parts after a
 *   per-vector power-of-two scale); the result meets the same tolerance
 *   for any finite x, the 320-lane limit does not apply and ws is unused.
 *   ws, ws_bytes  workspace of at least
 *            qws_workspace_bytes(QWS_OP_MATVEC, rows, hidden, 0, batch, S)
 *            bytes (device, 16-byte aligned); may be NULL when split_k == 1. */
qws_status qws_q4_0_matvec(const void* W, const float* x, float* y, int64_t rows, int64_t hidden,
                           int batch, int split_k, void* ws, size_t ws_bytes, qws_stream stream);

/* Any format, with the same split-K option. */
qws_status qws_matvec(qws_format fmt, const void* W, const float* x, float* y, int64_t rows,
                      int64_t hidden, int batch, int split_k, void* ws, size_t ws_bytes,
                      qws_stream stream);

/* ------------------------------------------------------------------------
 * Fused Q/K/V projection (infer-compute README §Shaders, q4k_qkv_proj): the
 * three Q4_K matrices share x and are streamed in one launch.
 *   q = Wq x (q_dim rows), k = Wk x (kv_dim rows), v = Wv x (kv_dim rows)
 *   Wq q_dim x hidden, Wk and Wv kv_dim x hidden, Q4_K (device, 16-B aligned)
 *   x [hidden], q [q_dim], k [kv_dim], v [kv_dim] f32 (device)
 * ---------------------------------------------------------------------- */
qws_status qws_q4k_qkv_proj(const void* Wq, const void* Wk, const void* Wv, const float* x,
                            float* q, float* k, float* v, int64_t hidden, int64_t q_dim,
                            int64_t kv_dim, qws_stream stream);

/* ------------------------------------------------------------------------
 * The 8-bit path (infer-compute README §Architecture: the Q4_0 FFN goes
 * "through legacy Q8 path"; §Shaders rows "Q8" (q8_matvec, q8_qkv_proj) and
 * "Element-wise" (quantize_q8)).  Activations are first quantized to Q8_0
 * blocks; the matvecs then multiply integer codes exactly (dp4a) and apply
 * the two block scales:
 *   y[b][r] = sum_k dw[r][k] * dx[b][k] * sum_j qw[r][k][j] * qx[b][k][j]
 * with qw = q - 8 for Q4_0 weights and qw = q for Q8_0 weights.
 *
 * Q8_0 block (34 bytes, 32 values): binary16 d, then 32 int8 codes; x ~ d*q.
 *
 * qws_quantize_q8_0: x [batch][n] f32 (device, 4-byte aligned, finite) ->
 *   xq [batch][n / 32 * 34] bytes (device, 2-byte aligned).  Per block of
 *   32, all in f32:
 *   amax = max |x|, d = amax / 127, id = (d != 0 ? 1 / d : 0),
 *   q = round(x * id) (halves away from zero); d is stored rounded to
 *   binary16 (nearest, ties to even).  The pages give no rounding rule; this
 *   is the symmetric absmax reading.  n > 0, n % 32 == 0, batch >= 1.
 *   Output bytes are identical run to run.
 *
 * qws_q8_matvec: W rows x hidden in wfmt (QWS_Q4_0 or QWS_Q8_0; device,
 *   16-byte aligned), xq [batch][hidden / 32 * 34] bytes (device, 4-byte
 *   aligned), y [batch][rows] f32 (device, 4-byte aligned), overwritten.
 *   hidden % 64 == 0, 0 < hidden <= 20480, batch * hidden / 64 <= 320.
 *   With 2..8 vectors, hidden % 256 == 0 and hidden <= 3072 a kernel that
 *   decodes each weight once for all vectors runs instead (tensor-core
 *   products of the exact integer codes, each block scaled by dw * dx in
 *   f32; no lane limit); the tolerance is the same.
 *   Any other format returns QWS_ERR_FORMAT.
 *
 * qws_q8_qkv_proj: the fused Q/K/V projection of the 8-bit path (batch 1):
 *   q = Wq xq (q_dim rows), k = Wk xq, v = Wv xq (kv_dim rows each), all
 *   three matrices in wfmt, streamed in one launch.
 * ---------------------------------------------------------------------- */
qws_status qws_quantize_q8_0(const float* x, void* xq, int64_t n, int batch, qws_stream stream);

/* Fused norm + quantize (infer-compute README §Shaders "Fused ops":
 * rms_norm_q8, residual_norm_q8): the rms_norm of qws_rms_norm (after h <- h + y
 * for the residual form, as qws_residual_rms_norm) quantized to Q8_0 blocks
 * as qws_quantize_q8_0 does, in one launch; the f32 normalized vector is not
 * stored.  x / h, y [batch][n] f32 (device, 4-byte aligned; h updated in
 * place), w [n] f32, xq [batch][n / 32 * 34] bytes (device, 2-byte aligned);
 * n > 0, n % 32 == 0, 1 <= batch <= 65535, eps >= 0. */
qws_status qws_rms_norm_q8(const float* x, const float* w, void* xq, int64_t n, float eps,
                           int batch, qws_stream stream);
qws_status qws_residual_rms_norm_q8(float* h, const float* y, const float* w, void* xq,
                                    int64_t n, float eps, int batch, qws_stream stream);
qws_status qws_q8_matvec(qws_format wfmt, const void* W, const void* xq, float* y, int64_t rows,
                         int64_t hidden, int batch, qws_stream stream);
qws_status qws_q8_qkv_proj(qws_format wfmt, const void* Wq, const void* Wk, const void* Wv,
                           const void* xq, float* q, float* k, float* v, int64_t hidden,
                           int64_t q_dim, int64_t kv_dim, qws_stream stream);

/* ------------------------------------------------------------------------
 * Prefill: the Q4_K product for many tokens at once (infer-compute README
 * §Quick Start and §Architecture, prefill_q4: the seq > 1 GPU path), on the
 * tensor cores:   Y[n][r] = sum_k dequant(W)[r][k] * X[n][k].
 *   W  rows x hidden Q4_K (device, 16-byte aligned)
 *   X  [n_tokens][hidden] f32 (device, 16-byte aligned)
 *   Y  [n_tokens][rows] f32 (device, 4-byte aligned), overwritten
 *   ws >= qws_workspace_bytes(QWS_OP_PREFILL, 0, hidden, 0, n_tokens, 0)
 *      bytes (device, 16-byte aligned): X split into f16 hi and lo parts, in
 *      tiles, and one scale per token
 *   rows >= 0; 0 < hidden <= 20480, hidden % 256 == 0; n_tokens >= 1.
 * Precision: the matvecs' bound, |Y - Y_exact| <= 1e-5 * sum_k |w x| per
 * output.  Each operand is split into two f16 parts (the weight, dequantized
 * in f32, scaled by 2^10; each token scaled by a power of two that puts its
 * largest |x| in [2^14, 2^15)); three f16 products per pair (hi*hi, hi*lo,
 * lo*hi) accumulate in f32.  The split needs |w| < 64 (every sub-block's
 * |d*sc|*15 + |dmin*m| < 64); a larger one records device error code 256
 * (read by qws_device_error).  Results are identical run to run.  The pages
 * do not state the precision of their prefill path; this keeps the one they
 * state for the matvecs.
 * ---------------------------------------------------------------------- */
qws_status qws_q4k_prefill_matmul(const void* W, const float* X, float* Y, int64_t rows,
                                  int64_t hidden, int64_t n_tokens, void* ws, size_t ws_bytes,
                                  qws_stream stream);

/* ------------------------------------------------------------------------
 * Decode attention over a KV cache, sequence length > 1 (infer-compute README
 * §Shaders rows "RoPE" (rope_at_pos) and "Attention" (kv_append,
 * kv_attention: GQA, softcap); infer-inference README §BLAS-Fused Attention).
 * Caches are f32 [n_kv_heads][max_seq][head_dim] (device); vectors f32.
 *
 * qws_rope_at_pos: x [n_heads][head_dim] (device) rotated in place at
 *   position pos: for i < rot_dim / 2, theta_i = pos * base^(-2i / rot_dim),
 *   (x_i, x_{i+rot/2}) <- (x_i cos - x_{i+rot/2} sin, x_i sin + x_{i+rot/2} cos);
 *   dimensions rot_dim.. unchanged (partial RoPE).  Angle, sine, cosine and
 *   the rotation in f64, rounded once to f32 (the angles' sines and cosines
 *   are evaluated on the host, once per call).  rot_dim even, 0 < rot_dim <=
 *   min(head_dim, 512), else QWS_ERR_SHAPE; pos >= 0; base > 0.  (The pages
 *   give no formula: this is the standard half-split rotary embedding.)
 * qws_kv_append: k, v [n_kv_heads][head_dim] written at position pos of the
 *   caches (0 <= pos < max_seq).
 * qws_kv_attention: one query token q [n_q_heads][head_dim] over cache
 *   positions 0 .. n_ctx-1; query head h reads kv head h / (n_q / n_kv):
 *     s_t = scale * q_h . k_t;  s_t <- softcap * tanh(s_t / softcap) if
 *     softcap > 0;  out_h = sum_t softmax(s)_t v_t.
 *   out [n_q_heads][head_dim] (device, overwritten); ws >=
 *   qws_workspace_bytes(QWS_OP_KV_ATTENTION, n_ctx, head_dim, n_q_heads,
 *   n_kv_heads, 0) bytes (device, 16-byte aligned).  head_dim in {32, 64,
 *   128, 256}; n_q_heads / n_kv_heads in 1..4; 1 <= n_ctx <= max_seq; caches
 *   and q 16-byte aligned.  Split along the positions, merged in a fixed
 *   order: identical run to run.
 * ---------------------------------------------------------------------- */
qws_status qws_rope_at_pos(float* x, int n_heads, int head_dim, int rot_dim, int64_t pos,
                           double base, qws_stream stream);
qws_status qws_kv_append(float* k_cache, float* v_cache, const float* k, const float* v,
                         int n_kv_heads, int head_dim, int64_t max_seq, int64_t pos,
                         qws_stream stream);
qws_status qws_kv_attention(const float* q, const float* k_cache, const float* v_cache,
                            float* out, int n_q_heads, int n_kv_heads, int head_dim,
                            int64_t max_seq, int64_t n_ctx, float scale, float softcap,
                            void* ws, size_t ws_bytes, qws_stream stream);

/* ------------------------------------------------------------------------
 * Gated FFN (infer-compute README §Shaders "Q4_K fused FFN": q4k_ffn_gate_up,
 * q4k_geglu_gelu_tanh_down; infer-inference README §WalkFfn steps 1-3):
 *   g = Wg x, u = Wu x            (one pass over x for both, inter rows)
 *   m = gelu_tanh(g) * u          (in the epilogue of the gate/up pass)
 *   y = Wd m                      (hidden rows, inter columns)
 *   Wg, Wu inter x hidden Q4_K; Wd hidden x inter in wd_fmt (Q6_K or Q4_K)
 *   x [hidden], y [hidden] f32; ws >= qws_workspace_bytes(QWS_OP_FFN, 0,
 *   hidden, inter, 1, 0) bytes; m is left in the first inter floats of ws.
 * ---------------------------------------------------------------------- */
qws_status qws_q4k_ffn_gate_up_geglu_down(const void* Wg, const void* Wu, const void* Wd,
                                          qws_format wd_fmt, const float* x, float* y,
                                          int64_t hidden, int64_t inter, void* ws,
                                          size_t ws_bytes, qws_stream stream);

/* First half of the FFN alone: m = gelu_tanh(Wg x) * (Wu x), m [inter]. */
qws_status qws_q4k_ffn_gate_up_geglu(const void* Wg, const void* Wu, const float* x, float* m,
                                     int64_t hidden, int64_t inter, qws_stream stream);

/* ------------------------------------------------------------------------
 * The SiLU-gated FFN for SiLU models (infer-compute README §Shaders, the
 * SiLU-gated down variant; infer-inference PERFORMANCE.md §Activation
 * Function Support): as qws_q4k_ffn_gate_up_geglu_down with
 *   m = silu(g) * u,   silu(t) = t / (1 + exp(-t)).
 * Arguments, layouts, workspace and errors as the GELU entry points.
 * ---------------------------------------------------------------------- */
qws_status qws_q4k_ffn_gate_up_silu_down(const void* Wg, const void* Wu, const void* Wd,
                                         qws_format wd_fmt, const float* x, float* y,
                                         int64_t hidden, int64_t inter, void* ws,
                                         size_t ws_bytes, qws_stream stream);

/* First half of the SiLU FFN alone: m = silu(Wg x) * (Wu x), m [inter]. */
qws_status qws_q4k_ffn_gate_up_silu(const void* Wg, const void* Wu, const float* x, float* m,
                                    int64_t hidden, int64_t inter, qws_stream stream);

/* ------------------------------------------------------------------------
 * The gated FFN above for callers that cannot allocate device memory.  The
 * pages have no counterpart; this is a convenience of this library.  It is for
 * callers that may not allocate at call time and have no spare device buffer
 * to lend as workspace (for example a serving runtime whose device memory pool
 * is fixed at start-up, or a plugin whose host forbids device allocations
 * outside its own allocator).  The intermediate m lives in a fixed array
 * inside the library: every device that loads the library holds
 * QWS_FFN_NOALLOC_MAX_INTER floats (80 KiB) of it until the process exits.
 *   Arguments, layouts and results as qws_q4k_ffn_gate_up_geglu_down, without
 *   ws / ws_bytes; inter <= QWS_FFN_NOALLOC_MAX_INTER, else QWS_ERR_SHAPE.
 *   Allocates nothing: no cudaMalloc / cudaFree and no allocating library call.
 *   Each call looks up the array's device address in the current device's
 *   context (the lookup allocates nothing, and a context recreated after a
 *   device reset gets its own address); the first call on a device may load
 *   the library's module there, so make that first call before any stream
 *   capture.  Every call on a device shares the one array, and m is rewritten
 *   from scratch by each call; calls that overlap on the GPU (streams with no
 *   ordering between them) race on it and must be serialised by the caller.
 * ---------------------------------------------------------------------- */
#define QWS_FFN_NOALLOC_MAX_INTER 20480

qws_status qws_q4k_ffn_gate_up_geglu_down_noalloc(const void* Wg, const void* Wu, const void* Wd,
                                                  qws_format wd_fmt, const float* x, float* y,
                                                  int64_t hidden, int64_t inter,
                                                  qws_stream stream);

/* ------------------------------------------------------------------------
 * rms_norm (infer-compute README §Shaders "Normalization"):
 *   y[b][i] = x[b][i] / sqrt(mean_j x[b][j]^2 + eps) * w[i]
 * x, y [batch][n], w [n] f32 (device); y may equal x.  n > 0, batch >= 1.
 * residual_add (§Shaders "Element-wise"):  h[b][i] += y[b][i].
 * ---------------------------------------------------------------------- */
qws_status qws_rms_norm(const float* x, const float* w, float* y, int64_t n, float eps,
                        int batch, qws_stream stream);
qws_status qws_residual_add(float* h, const float* y, int64_t n, int batch, qws_stream stream);

/* ------------------------------------------------------------------------
 * residual_norm (infer-compute README §Shaders "residual_norm"): the residual
 * add and the RMS norm of its result in one launch:
 *   h[b][i] += y[b][i];   x[b][i] = h[b][i] / sqrt(mean_j h[b][j]^2 + eps) * w[i]
 * h (in/out), y, x [batch][n], w [n] f32 (device, 4-byte aligned); x must not
 * alias h or y.  n > 0, 1 <= batch <= 65535, eps >= 0; errors as rms_norm.
 * ---------------------------------------------------------------------- */
qws_status qws_residual_rms_norm(float* h, const float* y, const float* w, float* x, int64_t n,
                                 float eps, int batch, qws_stream stream);

/* ------------------------------------------------------------------------
 * Decoder chain at sequence length 1 (infer-compute README §Architecture:
 * "single command buffer ... for all 34 layers", §Quick Start decode_token;
 * infer-inference PERFORMANCE.md §Post-Norm Architecture).  Per layer:
 *   n1 = rms_norm(h, w_in); q, k, v = QKV(n1); a = v broadcast to the query
 *   heads (one key: softmax = 1; head i reads kv head i / (nq / nkv));
 *   o = Wo a;  h1 = h + rms_norm(o, w_post_attn)      (post_norms = 1)
 *              h1 = h + o                              (post_norms = 0)
 *   n2 = rms_norm(h1, w_pre_ffn); f = FFN(n2);
 *   h  = h1 + rms_norm(f, w_post_ffn)  (post_norms = 1)  or  h1 + f.
 * All layers run in ONE persistent cooperative launch; weights of the next
 * step stream into shared memory while the grid waits at a step boundary.
 *   layers   host array of n_layers descriptors (1 <= n_layers <= 64)
 *   h        [hidden] f32 device, in/out
 *   ws       >= qws_workspace_bytes(QWS_OP_DECODE_CHAIN, 0, hidden, inter, 1, 0)
 * Limits: formats Q4_K for q/k/v/o/gate/up, Q4_K or Q6_K for down; hidden,
 * inter, n_q_heads*head_dim multiples of 256 and <= 20480; n_q_heads a
 * multiple of n_kv_heads.
 * ---------------------------------------------------------------------- */
typedef struct {
  const void *Wq, *Wk, *Wv, *Wo, *Wg, *Wu, *Wd;
  qws_format fmt_qkv, fmt_o, fmt_gu, fmt_down;
  const float *w_in, *w_post_attn, *w_pre_ffn, *w_post_ffn; /* [hidden] each */
} qws_layer;

typedef struct {
  int64_t hidden, inter;
  int n_q_heads, n_kv_heads, head_dim;
  float eps;
  int post_norms;
} qws_dims;

qws_status qws_decode_chain(const qws_layer* layers, int n_layers, float* h,
                            const qws_dims* dims, void* ws, size_t ws_bytes, qws_stream stream);

/* qws_decode_chain followed by the model's final norm in the same launch
 * (infer-compute README §Architecture: the decode path ends with the final
 * norm before the lm_head): after the last layer,
 *   hn = rms_norm(h, w_final) = h * (mean(h^2) + eps)^-1/2 * w_final,
 * computed by the CTA that writes h, so a following lm_head reads hn with no
 * norm launch in between.  h, layers, dims, ws: as for qws_decode_chain (h
 * holds the last layer's output on return, bit-identical to that call's).
 *   w_final  [hidden] f32 device, 4-byte aligned
 *   hn       [hidden] f32 device, 4-byte aligned, out; must not overlap h
 * Errors: those of qws_decode_chain; QWS_ERR_NULL if w_final or hn is NULL,
 * QWS_ERR_ALIGN if either is misaligned, QWS_ERR_SHAPE if hn overlaps h (all
 * checked before any launch). */
qws_status qws_decode_chain_final_norm(const qws_layer* layers, int n_layers, float* h,
                                      const float* w_final, float* hn, const qws_dims* dims,
                                      void* ws, size_t ws_bytes, qws_stream stream);

/* ------------------------------------------------------------------------
 * One decode step at sequence position pos with a KV cache (infer-compute
 * README §Architecture: decode is norm -> QKV -> attend -> O -> FFN per layer;
 * §Shaders rows "RoPE" rope_at_pos and "Attention" kv_append, kv_attention;
 * infer-compute §Quick Start decode_token(..., rope_base)).  Per layer, the
 * layer of qws_decode_chain with the sequence-1 broadcast replaced by real
 * attention:
 *   n = rms_norm(h, w_in); [q|k|v] = W n; q, k <- RoPE at pos (the first
 *   rot_dim dimensions of every head, half-split pairs, base rope_base);
 *   caches[l][pos] <- k, v; a = attention of q over positions 0..pos (scale
 *   attn_scale, optional softcap, query head h reads kv head h / (n_q / n_kv));
 *   o = Wo a; then the residuals and norms of qws_decode_chain (sandwich norms
 *   when dims->post_norms) and the GEGLU FFN.
 *   h [hidden] f32 device, in: the token's input, out: the last layer's output.
 *   kv->k_caches[l], kv->v_caches[l]: device pointers (an array of n_layers on
 *   the host) to f32 [n_kv_heads][max_seq][head_dim], 16-byte aligned,
 *   caller-owned; positions 0..pos-1 are read, position pos is written.
 *   ws: device, >= qws_decode_kv_workspace_bytes(dims, max_seq) bytes,
 *   16-byte aligned, scratch (its contents on return are unspecified).
 *   Runs on the decode chain's kernel: with head_dim 256 and at most 2
 *   query heads per kv head, or head_dim 128 and 1, 2 or 4, the attention
 *   (RoPE at pos, the K/V append, the softmax over positions 0..pos) runs
 *   inside it and a token is one launch (per 64 layers); other head shapes
 *   take one chain launch per layer with the attention launches between
 *   them; layers whose down projections differ in format take a sequence of
 *   standalone launches with the same results' bounds.
 *   Shapes: as qws_decode_chain; head_dim in {32, 64, 128, 256};
 *   n_q_heads / n_kv_heads in 1..4; 0 <= pos < max_seq; rot_dim even in
 *   (0, head_dim]; rope_base > 0; attn_scale finite; softcap >= 0 (0 = off).
 *   Asynchronous on stream; errors as above, nothing enqueued on an error.
 * ---------------------------------------------------------------------- */
typedef struct {
  float* const* k_caches;
  float* const* v_caches;
  int64_t max_seq;
  int64_t pos;
  int rot_dim;
  double rope_base;
  float attn_scale;
  float softcap;
} qws_kv;

size_t qws_decode_kv_workspace_bytes(const qws_dims* dims, int64_t max_seq);
qws_status qws_decode_kv(const qws_layer* layers, int n_layers, float* h, const qws_dims* dims,
                         const qws_kv* kv, void* ws, size_t ws_bytes, qws_stream stream);

/* ------------------------------------------------------------------------
 * Bookkeeping.
 * qws_workspace_bytes: bytes of workspace an op needs (0 if none); for
 *   QWS_OP_MATVEC pass the split count in split_k (0 = the library's choice).
 * qws_last_error: message of the calling thread's last failed call ("" if
 *   none).  The pointer stays valid until that thread's next call.
 * qws_device_error: waits for the device, returns the OR of the error codes
 *   recorded by kernels since the last call (1 = a consumer gave up waiting
 *   for data, 2 = a producer gave up waiting for a free stage, 4 = a grid
 *   barrier gave up, 8 = a producer gave up draining its copies; 16..128 the
 *   prefill kernel's waits; 256 = a prefill weight outside the f16 split's
 *   range) and clears them.  Returns QWS_ERR_TIMEOUT when the code is
 *   non-zero.
 * qws_version: library version string.
 * ---------------------------------------------------------------------- */
size_t qws_workspace_bytes(qws_op op, int64_t rows, int64_t hidden, int64_t inter, int batch,
                           int split_k);

/* ------------------------------------------------------------------------
 * Self-test of the failure path (no counterpart on the pages; the pages'
 * checked buffer access, infer-compute README §Safe Buffer Access, is the
 * convention this extends to device-side waits).  Runs one of the library's
 * bounded wait primitives on something that never becomes ready, with a wait
 * limit of limit_cycles clock cycles instead of the kernels' ~1 s default:
 *   kind 0: the streaming engine's mbarrier wait, on a barrier that no thread
 *           and no copy ever completes;
 *   kind 1: the decode chain's stamped-word poll, on the 8-byte word at word8
 *           (device memory, 8-byte aligned, caller-owned; the call clears it
 *           first, so its stamp never matches).
 * The wait gives up, records code 1 (a consumer gave up waiting for data) for
 * qws_device_error() and the kernel returns; nothing else is in flight, so
 * the context stays usable.  limit_cycles in [1, ~2e9]; errors as above.
 * ---------------------------------------------------------------------- */
qws_status qws_selftest_wait_timeout(int kind, long long limit_cycles, void* word8,
                                     qws_stream stream);
const char* qws_last_error(void);
qws_status qws_device_error(unsigned* code);
const char* qws_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QWS_H */
