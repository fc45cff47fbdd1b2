// FP8 pre-pass and forward (placeholder until the kernels land).
#include "common.h"

namespace attn {
attn_status_t launch_fp8_quantize(const Fp8QuantParams&, cudaStream_t) {
  return fail(ATTN_ERR_UNSUPPORTED, "FP8 pre-pass not built yet");
}
attn_status_t launch_fwd_fp8(const Fp8FwdParams&, cudaStream_t) {
  return fail(ATTN_ERR_UNSUPPORTED, "FP8 forward not built yet");
}
}  // namespace attn
