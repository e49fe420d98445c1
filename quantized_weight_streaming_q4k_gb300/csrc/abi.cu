// abi.cu -- the C ABI declared in include/qws.h: argument checks (on the host,
// before anything is enqueued), workspace sizing and dispatch to launchers.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/qws.h"
#include "launch.h"

namespace {

thread_local std::string tl_error;

qws_status fail(qws_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  tl_error = buf;
  return st;
}

qws_status ok() {
  tl_error.clear();
  return QWS_OK;
}

qws_status cuda_fail(cudaError_t e, const char* what, const std::string& why) {
  if (!why.empty())
    return fail(e == cudaErrorInvalidValue ? QWS_ERR_SHAPE : QWS_ERR_CUDA, "%s: %s", what,
                why.c_str());
  return fail(QWS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool known_format(int fmt) { return fmt == QWS_Q4_0 || fmt == QWS_Q4_K || fmt == QWS_Q6_K; }

constexpr int64_t kMaxHidden = 20480;  // 320 lane units of 64 columns

#define QWS_CHECK_PTR(p) \
  if (!(p)) return fail(QWS_ERR_NULL, "%s: %s is NULL", fn, #p)
#define QWS_CHECK_W(p)                                                         \
  do {                                                                         \
    QWS_CHECK_PTR(p);                                                          \
    if (!aligned(p, 16)) return fail(QWS_ERR_ALIGN, "%s: %s is not 16-byte aligned", fn, #p); \
  } while (0)
#define QWS_CHECK_F(p)                                                         \
  do {                                                                         \
    QWS_CHECK_PTR(p);                                                          \
    if (!aligned(p, 4)) return fail(QWS_ERR_ALIGN, "%s: %s is not 4-byte aligned", fn, #p); \
  } while (0)

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// Split count the library picks: 1 unless batch * lane units per row
// (hidden / S / unit width) must shrink to fit the 320 consumer lanes.
int auto_splits(int fmt, int64_t hidden, int batch) {
  const int64_t nb = hidden / 256;
  const int64_t uw = qws::unit_weights(fmt);
  for (int64_t s = 1; s <= nb; ++s) {
    if (nb % s) continue;
    if ((hidden / s / uw) * batch <= 320) return static_cast<int>(s);
  }
  return -1;
}

qws_status check_matvec(const char* fn, int fmt, const void* W, const float* x, const float* y,
                        int64_t rows, int64_t hidden, int batch) {
  if (!known_format(fmt)) return fail(QWS_ERR_FORMAT, "%s: unknown format %d", fn, fmt);
  QWS_CHECK_W(W);
  QWS_CHECK_F(x);
  QWS_CHECK_F(y);
  if (rows < 0) return fail(QWS_ERR_SHAPE, "%s: rows = %lld < 0", fn, (long long)rows);
  if (hidden <= 0 || hidden % 256)
    return fail(QWS_ERR_SHAPE, "%s: hidden = %lld is not a positive multiple of 256", fn,
                (long long)hidden);
  if (batch < 1) return fail(QWS_ERR_SHAPE, "%s: batch = %d < 1", fn, batch);
  if (rows > (int64_t(1) << 31) / batch)
    return fail(QWS_ERR_SHAPE, "%s: rows * batch above 2^31", fn);
  return QWS_OK;
}

qws_status run_matvec(const char* fn, int fmt, const void* W, const float* x, float* y,
                      int64_t rows, int64_t hidden, int batch, int split_k, void* ws,
                      size_t ws_bytes, cudaStream_t st) {
  qws_status rc = check_matvec(fn, fmt, W, x, y, rows, hidden, batch);
  if (rc != QWS_OK) return rc;
  if (split_k < 0) return fail(QWS_ERR_SHAPE, "%s: split_k = %d < 0", fn, split_k);
  if (split_k <= 1 && qws::batch_q4_eligible(fmt, hidden, batch)) {
    // 2..8 vectors: every weight decoded once for all of them (no lane limit)
    if (rows == 0) return ok();
    const cudaError_t e = qws::launch_batch_q4_matvec(fmt, static_cast<const uint8_t*>(W), x, y,
                                                      rows, hidden, batch, st);
    if (e != cudaSuccess) return cuda_fail(e, fn, "");
    return ok();
  }
  int S = split_k == 0 ? auto_splits(fmt, hidden, batch) : split_k;
  if (S < 1)
    return fail(QWS_ERR_SHAPE, "%s: batch %d too large for hidden %lld", fn, batch,
                (long long)hidden);
  if ((hidden / 256) % S)
    return fail(QWS_ERR_SHAPE, "%s: split_k = %d does not divide hidden/256 = %lld", fn, S,
                (long long)(hidden / 256));
  const int64_t Ks = hidden / S;
  if (Ks > kMaxHidden)
    return fail(QWS_ERR_SHAPE, "%s: hidden / split_k = %lld above %lld; use split_k", fn,
                (long long)Ks, (long long)kMaxHidden);
  const int64_t lanes = (Ks / qws::unit_weights(fmt)) * batch;
  if (lanes > 320)
    return fail(QWS_ERR_SHAPE,
                "%s: batch * lane units per row = %lld above 320 (use split_k, or a smaller batch)",
                fn, (long long)lanes);
  if (S > 1) {
    if (qws::row_bytes_of(fmt, hidden) % 16 || qws::row_bytes_of(fmt, Ks) % 16)
      return fail(QWS_ERR_SHAPE, "%s: split rows are not 16-byte multiples for this format", fn);
    const size_t need = qws_workspace_bytes(QWS_OP_MATVEC, rows, hidden, 0, batch, S);
    if (!ws || ws_bytes < need)
      return fail(QWS_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", fn, ws_bytes, need);
    if (!aligned(ws, 16)) return fail(QWS_ERR_ALIGN, "%s: ws is not 16-byte aligned", fn);
  }
  if (rows == 0) return ok();
  std::string why;
  qws::Seg seg{static_cast<const uint8_t*>(W), S > 1 ? static_cast<float*>(ws) : y, rows, 0};
  cudaError_t e = qws::launch_matvec(fmt, qws::EPI_STORE, &seg, 1, nullptr, x, hidden, batch, S,
                                     st, &why);
  if (e != cudaSuccess) return cuda_fail(e, fn, why);
  if (S > 1) {
    e = qws::launch_splitk_reduce(static_cast<const float*>(ws), y, rows * batch, S, st);
    if (e != cudaSuccess) return cuda_fail(e, fn, "");
  }
  return ok();
}

}  // namespace

void qws::set_last_error(const char* msg) { tl_error = msg ? msg : ""; }

extern "C" {

qws_status qws_q4k_matvec(const void* W, const float* x, float* y, int64_t rows, int64_t hidden,
                          int batch, qws_stream stream) {
  return run_matvec("qws_q4k_matvec", QWS_Q4_K, W, x, y, rows, hidden, batch, 1, nullptr, 0,
                    reinterpret_cast<cudaStream_t>(stream));
}

qws_status qws_q6k_matvec(const void* W, const float* x, float* y, int64_t rows, int64_t hidden,
                          int batch, qws_stream stream) {
  return run_matvec("qws_q6k_matvec", QWS_Q6_K, W, x, y, rows, hidden, batch, 1, nullptr, 0,
                    reinterpret_cast<cudaStream_t>(stream));
}

qws_status qws_q4_0_matvec(const void* W, const float* x, float* y, int64_t rows, int64_t hidden,
                           int batch, int split_k, void* ws, size_t ws_bytes, qws_stream stream) {
  return run_matvec("qws_q4_0_matvec", QWS_Q4_0, W, x, y, rows, hidden, batch, split_k, ws,
                    ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

qws_status qws_matvec(qws_format fmt, const void* W, const float* x, float* y, int64_t rows,
                      int64_t hidden, int batch, int split_k, void* ws, size_t ws_bytes,
                      qws_stream stream) {
  return run_matvec("qws_matvec", fmt, W, x, y, rows, hidden, batch, split_k, ws, ws_bytes,
                    reinterpret_cast<cudaStream_t>(stream));
}

qws_status qws_q4k_qkv_proj(const void* Wq, const void* Wk, const void* Wv, const float* x,
                            float* q, float* k, float* v, int64_t hidden, int64_t q_dim,
                            int64_t kv_dim, qws_stream stream) {
  const char* fn = "qws_q4k_qkv_proj";
  QWS_CHECK_W(Wq);
  QWS_CHECK_W(Wk);
  QWS_CHECK_W(Wv);
  QWS_CHECK_F(x);
  QWS_CHECK_F(q);
  QWS_CHECK_F(k);
  QWS_CHECK_F(v);
  if (hidden <= 0 || hidden % 256 || hidden > kMaxHidden)
    return fail(QWS_ERR_SHAPE, "%s: hidden = %lld (need a multiple of 256 in (0, 20480])", fn,
                (long long)hidden);
  if (q_dim < 0 || kv_dim < 0) return fail(QWS_ERR_SHAPE, "%s: negative q_dim / kv_dim", fn);
  if (q_dim + 2 * kv_dim == 0) return ok();
  qws::Seg segs[3];
  int n = 0;
  if (q_dim) segs[n++] = qws::Seg{static_cast<const uint8_t*>(Wq), q, q_dim, 0};
  if (kv_dim) {
    segs[n++] = qws::Seg{static_cast<const uint8_t*>(Wk), k, kv_dim, 0};
    segs[n++] = qws::Seg{static_cast<const uint8_t*>(Wv), v, kv_dim, 0};
  }
  std::string why;
  cudaError_t e = qws::launch_matvec(QWS_Q4_K, qws::EPI_STORE, segs, n, nullptr, x, hidden, 1, 1,
                                     reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, fn, why);
  return ok();
}

qws_status qws_quantize_q8_0(const float* x, void* xq, int64_t n, int batch, qws_stream stream) {
  const char* fn = "qws_quantize_q8_0";
  QWS_CHECK_F(x);
  QWS_CHECK_PTR(xq);
  if (!aligned(xq, 2)) return fail(QWS_ERR_ALIGN, "%s: xq is not 2-byte aligned", fn);
  if (n <= 0 || n % 32)
    return fail(QWS_ERR_SHAPE, "%s: n = %lld is not a positive multiple of 32", fn, (long long)n);
  if (batch < 1) return fail(QWS_ERR_SHAPE, "%s: batch = %d < 1", fn, batch);
  if (n > (int64_t(1) << 40) / batch) return fail(QWS_ERR_SHAPE, "%s: n * batch too large", fn);
  cudaError_t e = qws::launch_quantize_q8_0(x, static_cast<uint8_t*>(xq), n / 32 * batch,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn, "");
  return ok();
}

static qws_status check_q8_shape(const char* fn, int wfmt, int64_t hidden, int batch) {
  if (wfmt != QWS_Q4_0 && wfmt != QWS_Q8_0)
    return fail(QWS_ERR_FORMAT, "%s: weights must be Q4_0 or Q8_0 (got %d)", fn, wfmt);
  if (hidden <= 0 || hidden % 64 || hidden > kMaxHidden)
    return fail(QWS_ERR_SHAPE, "%s: hidden = %lld (need a multiple of 64 in (0, 20480])", fn,
                (long long)hidden);
  if (batch < 1) return fail(QWS_ERR_SHAPE, "%s: batch = %d < 1", fn, batch);
  // the decode-once kernel (2..8 vectors) has no lane limit
  if ((hidden / 64) * batch > 320 && !qws::batch_q4_eligible(100 + wfmt, hidden, batch))
    return fail(QWS_ERR_SHAPE, "%s: batch * hidden / 64 = %lld above 320", fn,
                (long long)((hidden / 64) * batch));
  return QWS_OK;
}

qws_status qws_q8_matvec(qws_format wfmt, const void* W, const void* xq, float* y, int64_t rows,
                         int64_t hidden, int batch, qws_stream stream) {
  const char* fn = "qws_q8_matvec";
  qws_status rc = check_q8_shape(fn, wfmt, hidden, batch);
  if (rc != QWS_OK) return rc;
  QWS_CHECK_W(W);
  QWS_CHECK_F(xq);
  QWS_CHECK_F(y);
  if (rows < 0) return fail(QWS_ERR_SHAPE, "%s: rows = %lld < 0", fn, (long long)rows);
  if (rows > (int64_t(1) << 31) / batch)
    return fail(QWS_ERR_SHAPE, "%s: rows * batch above 2^31", fn);
  if (rows == 0) return ok();
  if (qws::batch_q4_eligible(100 + wfmt, hidden, batch)) {
    // 2..8 vectors: every weight decoded once for all of them
    const cudaError_t e = qws::launch_batch_q4_matvec(
        100 + wfmt, static_cast<const uint8_t*>(W), nullptr, y, rows, hidden, batch,
        reinterpret_cast<cudaStream_t>(stream), static_cast<const uint8_t*>(xq));
    if (e != cudaSuccess) return cuda_fail(e, fn, "");
    return ok();
  }
  std::string why;
  qws::Seg seg{static_cast<const uint8_t*>(W), y, rows, 0};
  cudaError_t e = qws::launch_matvec_q8(wfmt, &seg, 1, static_cast<const uint8_t*>(xq), hidden,
                                        batch, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, fn, why);
  return ok();
}

qws_status qws_q8_qkv_proj(qws_format wfmt, const void* Wq, const void* Wk, const void* Wv,
                           const void* xq, float* q, float* k, float* v, int64_t hidden,
                           int64_t q_dim, int64_t kv_dim, qws_stream stream) {
  const char* fn = "qws_q8_qkv_proj";
  qws_status rc = check_q8_shape(fn, wfmt, hidden, 1);
  if (rc != QWS_OK) return rc;
  QWS_CHECK_W(Wq);
  QWS_CHECK_W(Wk);
  QWS_CHECK_W(Wv);
  QWS_CHECK_F(xq);
  QWS_CHECK_F(q);
  QWS_CHECK_F(k);
  QWS_CHECK_F(v);
  if (q_dim < 0 || kv_dim < 0) return fail(QWS_ERR_SHAPE, "%s: negative q_dim / kv_dim", fn);
  if (q_dim + 2 * kv_dim == 0) return ok();
  qws::Seg segs[3];
  int n = 0;
  if (q_dim) segs[n++] = qws::Seg{static_cast<const uint8_t*>(Wq), q, q_dim, 0};
  if (kv_dim) {
    segs[n++] = qws::Seg{static_cast<const uint8_t*>(Wk), k, kv_dim, 0};
    segs[n++] = qws::Seg{static_cast<const uint8_t*>(Wv), v, kv_dim, 0};
  }
  std::string why;
  cudaError_t e = qws::launch_matvec_q8(wfmt, segs, n, static_cast<const uint8_t*>(xq), hidden, 1,
                                        reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, fn, why);
  return ok();
}

qws_status qws_q4k_prefill_matmul(const void* W, const float* X, float* Y, int64_t rows,
                                  int64_t hidden, int64_t n_tokens, void* ws, size_t ws_bytes,
                                  qws_stream stream) {
  const char* fn = "qws_q4k_prefill_matmul";
  QWS_CHECK_W(W);
  QWS_CHECK_PTR(X);
  if (!aligned(X, 16)) return fail(QWS_ERR_ALIGN, "%s: X is not 16-byte aligned", fn);
  QWS_CHECK_F(Y);
  if (rows < 0) return fail(QWS_ERR_SHAPE, "%s: rows = %lld < 0", fn, (long long)rows);
  if (hidden <= 0 || hidden % 256 || hidden > kMaxHidden)
    return fail(QWS_ERR_SHAPE, "%s: hidden = %lld (need a multiple of 256 in (0, 20480])", fn,
                (long long)hidden);
  if (n_tokens < 1 || n_tokens > (int64_t(1) << 30))
    return fail(QWS_ERR_SHAPE, "%s: n_tokens = %lld outside [1, 2^30]", fn,
                (long long)n_tokens);
  if (rows > (int64_t(1) << 40) / n_tokens)
    return fail(QWS_ERR_SHAPE, "%s: rows * n_tokens too large", fn);
  const size_t need = qws::prefill_workspace_bytes(hidden, n_tokens);
  if (!ws || ws_bytes < need)
    return fail(QWS_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", fn, ws_bytes, need);
  if (!aligned(ws, 16)) return fail(QWS_ERR_ALIGN, "%s: ws is not 16-byte aligned", fn);
  if ((rows + 127) / 128 * ((n_tokens + 255) / 256) > (int64_t(1) << 31) - 1)
    return fail(QWS_ERR_SHAPE, "%s: too many tiles", fn);
  if (rows == 0) return ok();
  cudaError_t e = qws::launch_prefill_q4k(static_cast<const uint8_t*>(W), X, Y, rows, hidden,
                                          n_tokens, static_cast<uint8_t*>(ws),
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn, "");
  return ok();
}

qws_status qws_rope_at_pos(float* x, int n_heads, int head_dim, int rot_dim, int64_t pos,
                           double base, qws_stream stream) {
  const char* fn = "qws_rope_at_pos";
  QWS_CHECK_F(x);
  if (n_heads < 1 || head_dim < 2 || rot_dim < 2 || rot_dim % 2 || rot_dim > head_dim ||
      rot_dim > 512)
    return fail(QWS_ERR_SHAPE,
                "%s: need n_heads >= 1 and an even 0 < rot_dim <= min(head_dim, 512)", fn);
  if (pos < 0 || !(base > 0.0)) return fail(QWS_ERR_SHAPE, "%s: need pos >= 0 and base > 0", fn);
  cudaError_t e = qws::launch_rope(x, n_heads, head_dim, rot_dim, pos, base,
                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn, "");
  return ok();
}

qws_status qws_kv_append(float* k_cache, float* v_cache, const float* k, const float* v,
                         int n_kv_heads, int head_dim, int64_t max_seq, int64_t pos,
                         qws_stream stream) {
  const char* fn = "qws_kv_append";
  QWS_CHECK_F(k_cache);
  QWS_CHECK_F(v_cache);
  QWS_CHECK_F(k);
  QWS_CHECK_F(v);
  if (n_kv_heads < 1 || head_dim < 1 || max_seq < 1)
    return fail(QWS_ERR_SHAPE, "%s: empty cache shape", fn);
  if (pos < 0 || pos >= max_seq)
    return fail(QWS_ERR_SHAPE, "%s: pos = %lld outside [0, max_seq = %lld)", fn, (long long)pos,
                (long long)max_seq);
  cudaError_t e = qws::launch_kv_append(k_cache, v_cache, k, v, n_kv_heads, head_dim, max_seq,
                                        pos, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn, "");
  return ok();
}

qws_status qws_kv_attention(const float* q, const float* k_cache, const float* v_cache,
                            float* out, int n_q_heads, int n_kv_heads, int head_dim,
                            int64_t max_seq, int64_t n_ctx, float scale, float softcap,
                            void* ws, size_t ws_bytes, qws_stream stream) {
  const char* fn = "qws_kv_attention";
  QWS_CHECK_PTR(q);
  QWS_CHECK_PTR(k_cache);
  QWS_CHECK_PTR(v_cache);
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(QWS_ERR_ALIGN, "%s: q and the caches must be 16-byte aligned", fn);
  QWS_CHECK_F(out);
  if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(QWS_ERR_SHAPE, "%s: head_dim = %d not in {32, 64, 128, 256}", fn, head_dim);
  if (n_kv_heads < 1 || n_q_heads < n_kv_heads || n_q_heads % n_kv_heads ||
      n_q_heads / n_kv_heads > 4)
    return fail(QWS_ERR_SHAPE, "%s: n_q_heads / n_kv_heads must be an integer in 1..4", fn);
  if (n_ctx < 1 || n_ctx > max_seq)
    return fail(QWS_ERR_SHAPE, "%s: need 1 <= n_ctx <= max_seq", fn);
  if (!std::isfinite(scale) || !(softcap >= 0.f) || !std::isfinite(softcap))
    return fail(QWS_ERR_SHAPE, "%s: scale must be finite and softcap >= 0", fn);
  const size_t need = qws::kv_attention_workspace_bytes(n_q_heads, n_kv_heads, head_dim, n_ctx);
  if (!ws || ws_bytes < need)
    return fail(QWS_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", fn, ws_bytes, need);
  if (!aligned(ws, 16)) return fail(QWS_ERR_ALIGN, "%s: ws is not 16-byte aligned", fn);
  cudaError_t e = qws::launch_kv_attention(q, k_cache, v_cache, out, n_q_heads, n_kv_heads,
                                           head_dim, max_seq, n_ctx, scale, softcap,
                                           static_cast<float*>(ws),
                                           reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn, "");
  return ok();
}

static qws_status check_ffn_shape(const char* fn, int64_t hidden, int64_t inter) {
  if (hidden <= 0 || hidden % 256 || hidden > kMaxHidden)
    return fail(QWS_ERR_SHAPE, "%s: hidden = %lld (need a multiple of 256 in (0, 20480])", fn,
                (long long)hidden);
  if (inter <= 0 || inter % 256 || inter > kMaxHidden)
    return fail(QWS_ERR_SHAPE, "%s: inter = %lld (need a multiple of 256 in (0, 20480])", fn,
                (long long)inter);
  return QWS_OK;
}

namespace {

// The gated FFN's first launch: m = act(Wg x) * (Wu x), act by epilogue.
qws_status ffn_gate_up(const char* fn, int epi, const void* Wg, const void* Wu, const float* x,
                       float* m, int64_t hidden, int64_t inter, qws_stream stream) {
  QWS_CHECK_W(Wg);
  QWS_CHECK_W(Wu);
  QWS_CHECK_F(x);
  QWS_CHECK_F(m);
  qws_status rc = check_ffn_shape(fn, hidden, inter);
  if (rc != QWS_OK) return rc;
  qws::Seg seg{static_cast<const uint8_t*>(Wg), m, inter, 0};
  std::string why;
  cudaError_t e = qws::launch_matvec(QWS_Q4_K, epi, &seg, 1, static_cast<const uint8_t*>(Wu), x,
                                     hidden, 1, 1, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, fn, why);
  return ok();
}

// The whole gated FFN: the first launch into the workspace, then the down
// projection.
qws_status ffn_full(const char* fn, int epi, const void* Wg, const void* Wu, const void* Wd,
                    qws_format wd_fmt, const float* x, float* y, int64_t hidden, int64_t inter,
                    void* ws, size_t ws_bytes, qws_stream stream) {
  QWS_CHECK_W(Wg);
  QWS_CHECK_W(Wu);
  QWS_CHECK_W(Wd);
  QWS_CHECK_F(x);
  QWS_CHECK_F(y);
  if (wd_fmt != QWS_Q4_K && wd_fmt != QWS_Q6_K)
    return fail(QWS_ERR_FORMAT, "%s: wd_fmt must be Q4_K or Q6_K", fn);
  qws_status rc = check_ffn_shape(fn, hidden, inter);
  if (rc != QWS_OK) return rc;
  const size_t need = qws_workspace_bytes(QWS_OP_FFN, 0, hidden, inter, 1, 0);
  if (!ws || ws_bytes < need)
    return fail(QWS_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", fn, ws_bytes, need);
  if (!aligned(ws, 16)) return fail(QWS_ERR_ALIGN, "%s: ws is not 16-byte aligned", fn);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float* m = static_cast<float*>(ws);
  qws::Seg seg{static_cast<const uint8_t*>(Wg), m, inter, 0};
  std::string why;
  cudaError_t e = qws::launch_matvec(QWS_Q4_K, epi, &seg, 1, static_cast<const uint8_t*>(Wu), x,
                                     hidden, 1, 1, st, &why);
  if (e != cudaSuccess) return cuda_fail(e, fn, why);
  qws::Seg dseg{static_cast<const uint8_t*>(Wd), y, hidden, 0};
  e = qws::launch_matvec(wd_fmt, qws::EPI_STORE, &dseg, 1, nullptr, m, inter, 1, 1, st, &why);
  if (e != cudaSuccess) return cuda_fail(e, fn, why);
  return ok();
}

}  // namespace

qws_status qws_q4k_ffn_gate_up_geglu(const void* Wg, const void* Wu, const float* x, float* m,
                                     int64_t hidden, int64_t inter, qws_stream stream) {
  return ffn_gate_up("qws_q4k_ffn_gate_up_geglu", qws::EPI_GEGLU, Wg, Wu, x, m, hidden, inter,
                     stream);
}

qws_status qws_q4k_ffn_gate_up_geglu_down(const void* Wg, const void* Wu, const void* Wd,
                                          qws_format wd_fmt, const float* x, float* y,
                                          int64_t hidden, int64_t inter, void* ws,
                                          size_t ws_bytes, qws_stream stream) {
  return ffn_full("qws_q4k_ffn_gate_up_geglu_down", qws::EPI_GEGLU, Wg, Wu, Wd, wd_fmt, x, y,
                  hidden, inter, ws, ws_bytes, stream);
}

qws_status qws_q4k_ffn_gate_up_silu(const void* Wg, const void* Wu, const float* x, float* m,
                                    int64_t hidden, int64_t inter, qws_stream stream) {
  return ffn_gate_up("qws_q4k_ffn_gate_up_silu", qws::EPI_SWIGLU, Wg, Wu, x, m, hidden, inter,
                     stream);
}

qws_status qws_q4k_ffn_gate_up_silu_down(const void* Wg, const void* Wu, const void* Wd,
                                         qws_format wd_fmt, const float* x, float* y,
                                         int64_t hidden, int64_t inter, void* ws,
                                         size_t ws_bytes, qws_stream stream) {
  return ffn_full("qws_q4k_ffn_gate_up_silu_down", qws::EPI_SWIGLU, Wg, Wu, Wd, wd_fmt, x, y,
                  hidden, inter, ws, ws_bytes, stream);
}

qws_status qws_rms_norm(const float* x, const float* w, float* y, int64_t n, float eps,
                        int batch, qws_stream stream) {
  const char* fn = "qws_rms_norm";
  QWS_CHECK_F(x);
  QWS_CHECK_F(w);
  QWS_CHECK_F(y);
  if (n <= 0) return fail(QWS_ERR_SHAPE, "%s: n = %lld <= 0", fn, (long long)n);
  if (batch < 1 || batch > 65535) return fail(QWS_ERR_SHAPE, "%s: batch = %d", fn, batch);
  if (!(eps >= 0.f)) return fail(QWS_ERR_SHAPE, "%s: eps must be >= 0", fn);
  cudaError_t e =
      qws::launch_rms_norm(x, w, y, n, eps, batch, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn, "");
  return ok();
}

qws_status qws_residual_add(float* h, const float* y, int64_t n, int batch, qws_stream stream) {
  const char* fn = "qws_residual_add";
  QWS_CHECK_F(h);
  QWS_CHECK_F(y);
  if (n < 0) return fail(QWS_ERR_SHAPE, "%s: n = %lld < 0", fn, (long long)n);
  if (batch < 1) return fail(QWS_ERR_SHAPE, "%s: batch = %d < 1", fn, batch);
  if (n == 0) return ok();
  cudaError_t e =
      qws::launch_residual_add(h, y, n, batch, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn, "");
  return ok();
}

qws_status qws_residual_rms_norm(float* h, const float* y, const float* w, float* x, int64_t n,
                                 float eps, int batch, qws_stream stream) {
  const char* fn = "qws_residual_rms_norm";
  QWS_CHECK_F(h);
  QWS_CHECK_F(y);
  QWS_CHECK_F(w);
  QWS_CHECK_F(x);
  if (n <= 0) return fail(QWS_ERR_SHAPE, "%s: n = %lld <= 0", fn, (long long)n);
  if (batch < 1 || batch > 65535) return fail(QWS_ERR_SHAPE, "%s: batch = %d", fn, batch);
  if (!(eps >= 0.f)) return fail(QWS_ERR_SHAPE, "%s: eps must be >= 0", fn);
  cudaError_t e = qws::launch_residual_rms_norm(h, y, w, x, n, eps, batch,
                                                reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn, "");
  return ok();
}

static qws_status run_norm_q8(const char* fn, float* h, const float* y, const float* w,
                              void* xq, int64_t n, float eps, int batch, bool residual,
                              qws_stream stream) {
  QWS_CHECK_F(h);
  if (residual) QWS_CHECK_F(y);
  QWS_CHECK_F(w);
  QWS_CHECK_PTR(xq);
  if (!aligned(xq, 2)) return fail(QWS_ERR_ALIGN, "%s: xq is not 2-byte aligned", fn);
  if (n <= 0 || n % 32)
    return fail(QWS_ERR_SHAPE, "%s: n = %lld is not a positive multiple of 32", fn, (long long)n);
  if (batch < 1 || batch > 65535) return fail(QWS_ERR_SHAPE, "%s: batch = %d", fn, batch);
  if (!(eps >= 0.f)) return fail(QWS_ERR_SHAPE, "%s: eps must be >= 0", fn);
  cudaError_t e = qws::launch_norm_q8(h, y, w, static_cast<uint8_t*>(xq), n, eps, batch,
                                      residual, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn, "");
  return ok();
}

qws_status qws_rms_norm_q8(const float* x, const float* w, void* xq, int64_t n, float eps,
                           int batch, qws_stream stream) {
  return run_norm_q8("qws_rms_norm_q8", const_cast<float*>(x), nullptr, w, xq, n, eps, batch,
                     false, stream);
}

qws_status qws_residual_rms_norm_q8(float* h, const float* y, const float* w, void* xq,
                                    int64_t n, float eps, int batch, qws_stream stream) {
  return run_norm_q8("qws_residual_rms_norm_q8", h, y, w, xq, n, eps, batch, true, stream);
}

qws_status qws_decode_chain(const qws_layer* layers, int n_layers, float* h,
                            const qws_dims* dims, void* ws, size_t ws_bytes, qws_stream stream) {
  std::string err;
  const qws_status st = qws::decode_chain(layers, n_layers, h, dims, ws, ws_bytes,
                                          reinterpret_cast<cudaStream_t>(stream), err);
  if (st != QWS_OK) return fail(st, "%s", err.c_str());
  return ok();
}

qws_status qws_decode_chain_final_norm(const qws_layer* layers, int n_layers, float* h,
                                      const float* w_final, float* hn, const qws_dims* dims,
                                      void* ws, size_t ws_bytes, qws_stream stream) {
  if (!w_final || !hn) return fail(QWS_ERR_NULL, "qws_decode_chain_final_norm: NULL argument");
  std::string err;
  const qws_status st = qws::decode_chain(layers, n_layers, h, dims, ws, ws_bytes,
                                          reinterpret_cast<cudaStream_t>(stream), err, w_final,
                                          hn, "qws_decode_chain_final_norm");
  if (st != QWS_OK) return fail(st, "%s", err.c_str());
  return ok();
}

size_t qws_workspace_bytes(qws_op op, int64_t rows, int64_t hidden, int64_t inter, int batch,
                           int split_k) {
  switch (op) {
    case QWS_OP_MATVEC: {
      if (rows <= 0 || hidden <= 0 || batch < 1) return 0;
      const int S = split_k == 0 ? auto_splits(QWS_Q4_K, hidden, batch) : split_k;
      if (S <= 1) return 0;
      return round256(sizeof(float) * static_cast<size_t>(S) * batch * rows);
    }
    case QWS_OP_FFN:
      return inter > 0 ? round256(sizeof(float) * static_cast<size_t>(inter)) : 0;
    case QWS_OP_DECODE_CHAIN:
      return qws::chain_workspace_bytes(hidden, inter);
    case QWS_OP_PREFILL:
      if (hidden <= 0 || hidden % 256 || batch < 1) return 0;
      return round256(qws::prefill_workspace_bytes(hidden, batch));
    case QWS_OP_KV_ATTENTION:
      if (rows < 1 || hidden <= 0 || inter <= 0 || batch <= 0 || inter % batch) return 0;
      return round256(qws::kv_attention_workspace_bytes(static_cast<int>(inter), batch,
                                                        static_cast<int>(hidden), rows));
  }
  return 0;
}

const char* qws_last_error(void) { return tl_error.c_str(); }

qws_status qws_device_error(unsigned* code) {
  if (!code) return fail(QWS_ERR_NULL, "qws_device_error: code is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "qws_device_error", "");
  *code = qws::read_clear_matvec_errors() | qws::read_clear_chain_errors() |
          qws::read_clear_prefill_errors() | qws::read_clear_attention_errors() |
          qws::read_clear_batchmv_errors();
  return *code ? fail(QWS_ERR_TIMEOUT, "device error code 0x%x", *code) : ok();
}

size_t qws_decode_kv_workspace_bytes(const qws_dims* dims, int64_t max_seq) {
  return qws::decode_kv_workspace_bytes(dims, max_seq);
}

qws_status qws_decode_kv(const qws_layer* layers, int n_layers, float* h, const qws_dims* dims,
                         const qws_kv* kv, void* ws, size_t ws_bytes, qws_stream stream) {
  std::string err;
  const qws_status st = qws::decode_kv(layers, n_layers, h, dims, kv, ws, ws_bytes,
                                       reinterpret_cast<cudaStream_t>(stream), err);
  if (st != QWS_OK) return fail(st, "%s", err.c_str());
  return ok();
}

qws_status qws_selftest_wait_timeout(int kind, long long limit_cycles, void* word8,
                                     qws_stream stream) {
  const char* fn = "qws_selftest_wait_timeout";
  if (kind != 0 && kind != 1) return fail(QWS_ERR_SHAPE, "%s: kind must be 0 or 1", fn);
  if (limit_cycles < 1 || limit_cycles > qws::kWaitCycles)
    return fail(QWS_ERR_SHAPE, "%s: limit_cycles must be in [1, %lld]", fn, qws::kWaitCycles);
  if (kind == 1 && !word8) return fail(QWS_ERR_NULL, "%s: word8 is NULL", fn);
  if (kind == 1 && reinterpret_cast<uintptr_t>(word8) % 8)
    return fail(QWS_ERR_ALIGN, "%s: word8 must be 8-byte aligned", fn);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = kind == 0 ? qws::launch_selftest_mbar(limit_cycles, s)
                                  : qws::launch_selftest_poll(word8, limit_cycles, s);
  if (e != cudaSuccess) return cuda_fail(e, fn, "");
  return ok();
}

const char* qws_version(void) { return "qws 0.1.0 (sm_103a)"; }

}  // extern "C"
