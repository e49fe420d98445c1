// chain.cu -- persistent decode-chain kernel (placeholder until implemented).
#include <cuda_runtime.h>

#include "../../include/qws.h"
#include "launch.h"

namespace qws {
size_t chain_workspace_bytes(int64_t, int64_t) { return 0; }
unsigned read_clear_chain_errors() { return 0; }
}  // namespace qws

extern "C" qws_status qws_decode_chain(const qws_layer*, int, float*, const qws_dims*, void*,
                                       size_t, qws_stream) {
  return QWS_ERR_CUDA;
}
