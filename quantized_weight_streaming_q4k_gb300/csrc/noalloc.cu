// noalloc.cu -- the gated FFN for callers that cannot allocate device memory.
//
// qws_q4k_ffn_gate_up_geglu_down needs a caller-provided workspace for its
// intermediate vector m = gelu(Wg x) * (Wu x).  Some callers have neither a
// spare device buffer nor permission to allocate one at call time (a serving
// runtime whose device memory pool is fixed at start-up, or a plugin whose host
// forbids device allocations outside its own allocator).  This variant keeps m
// in a fixed array that lives in this library's module: every device that
// loads the library holds kMaxInter floats (80 KiB) of it until the process
// exits.  It computes exactly what the workspace version computes, with the
// same kernels.
#include <cuda_runtime.h>

#include <cstdio>
#include <string>

#include "../../include/qws.h"
#include "launch.h"

namespace {

constexpr int64_t kMaxInter = QWS_FFN_NOALLOC_MAX_INTER;

// The scratch vector m.  Shared by every call on a device: calls that overlap
// on the GPU (different streams, no ordering between them) race on it.
static __device__ __align__(256) float g_ffn_scratch[kMaxInter];

// Device address of g_ffn_scratch in the current device's context.  In host
// code the array's name only stands for the symbol; the kernels need the
// address the runtime reports.  It is looked up on every call (the lookup
// allocates nothing), so a context that was destroyed and recreated -- after
// cudaDeviceReset, say -- never leaves a stale address behind.
qws_status scratch_address(float** out, std::string& err) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_ffn_scratch);
  if (e != cudaSuccess || !p) {
    err = std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e);
    return QWS_ERR_CUDA;
  }
  *out = static_cast<float*>(p);
  return QWS_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" qws_status qws_q4k_ffn_gate_up_geglu_down_noalloc(const void* Wg, const void* Wu,
                                                             const void* Wd, qws_format wd_fmt,
                                                             const float* x, float* y,
                                                             int64_t hidden, int64_t inter,
                                                             qws_stream stream) {
  const char* fn = "qws_q4k_ffn_gate_up_geglu_down_noalloc";
  char msg[256];
  auto fail = [&](qws_status st, const char* what) {
    snprintf(msg, sizeof(msg), "%s: %s", fn, what);
    qws::set_last_error(msg);
    return st;
  };
  if (!Wg || !Wu || !Wd || !x || !y) return fail(QWS_ERR_NULL, "a pointer argument is NULL");
  if (!aligned(Wg, 16) || !aligned(Wu, 16) || !aligned(Wd, 16))
    return fail(QWS_ERR_ALIGN, "weights must be 16-byte aligned");
  if (!aligned(x, 4) || !aligned(y, 4)) return fail(QWS_ERR_ALIGN, "x and y must be 4-byte aligned");
  if (wd_fmt != QWS_Q4_K && wd_fmt != QWS_Q6_K) return fail(QWS_ERR_FORMAT, "wd_fmt must be Q4_K or Q6_K");
  if (hidden <= 0 || hidden % 256 || hidden > 20480)
    return fail(QWS_ERR_SHAPE, "hidden must be a multiple of 256 in (0, 20480]");
  if (inter <= 0 || inter % 256)
    return fail(QWS_ERR_SHAPE, "inter must be a positive multiple of 256");
  if (inter > kMaxInter) {
    snprintf(msg, sizeof(msg), "%s: inter = %lld exceeds the fixed scratch of %lld floats", fn,
             static_cast<long long>(inter), static_cast<long long>(kMaxInter));
    qws::set_last_error(msg);
    return QWS_ERR_SHAPE;
  }
  std::string err;
  float* m = nullptr;
  qws_status st = scratch_address(&m, err);
  if (st != QWS_OK) return fail(st, err.c_str());
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::string why;
  qws::Seg seg{static_cast<const uint8_t*>(Wg), m, inter, 0};
  cudaError_t e = qws::launch_matvec(QWS_Q4_K, qws::EPI_GEGLU, &seg, 1,
                                     static_cast<const uint8_t*>(Wu), x, hidden, 1, 1, s, &why);
  if (e != cudaSuccess) return fail(QWS_ERR_CUDA, why.empty() ? cudaGetErrorString(e) : why.c_str());
  qws::Seg dseg{static_cast<const uint8_t*>(Wd), y, hidden, 0};
  e = qws::launch_matvec(wd_fmt, qws::EPI_STORE, &dseg, 1, nullptr, m, inter, 1, 1, s, &why);
  if (e != cudaSuccess) return fail(QWS_ERR_CUDA, why.empty() ? cudaGetErrorString(e) : why.c_str());
  qws::set_last_error("");
  return QWS_OK;
}
