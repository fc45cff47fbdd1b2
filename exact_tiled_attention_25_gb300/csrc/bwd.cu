// BF16/FP16 attention backward (placeholder until the kernels land).
#include "common.h"

namespace attn {
attn_status_t launch_bwd(const BwdParams&, cudaStream_t) {
  return fail(ATTN_ERR_UNSUPPORTED, "backward pass not built yet");
}
}  // namespace attn
