// lmhead.cu -- fused LM head + top-16 (placeholder until the tensor-core kernel lands).
#include "common.cuh"
#include "launch.h"

namespace dflash2 {

size_t lmhead_workspace_bytes(int64_t M, int64_t V, int64_t d) {
  (void)M; (void)V; (void)d;
  return 256;
}

cudaError_t launch_lmhead_topk(const uint16_t* hidden, const uint16_t* W, int64_t M, int64_t V,
                               int64_t d, float* vals, int32_t* idx, void* workspace, int num_sms,
                               uint32_t* err, cudaStream_t stream) {
  (void)hidden; (void)W; (void)M; (void)V; (void)d; (void)vals; (void)idx; (void)workspace;
  (void)num_sms; (void)err; (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace dflash2
