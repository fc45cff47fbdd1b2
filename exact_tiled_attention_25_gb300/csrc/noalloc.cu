// attn_bwd_noalloc: the backward pass for callers that cannot allocate
// device memory -- for example code running inside a custom runtime with no
// allocator of its own, or a host library that must not call cudaMalloc on
// the caller's behalf.  The scratch attn_bwd needs (float32 dQ accumulator and
// the two padded row vectors) comes from a fixed array compiled into this
// library instead of a caller-provided workspace.
#include "common.h"

namespace attn {
namespace {

// Largest scratch the built-in array provides.  Every GPU that loads this
// library holds this much device memory until the process exits.
constexpr size_t kNoAllocScratchBytes = 64ull << 20;   // 64 MiB

__device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

// Device address of g_bwd_scratch in the current context.  In host code the
// symbol itself is only a host-side stand-in, so the address is looked up with
// the device current.  The lookup runs on every call (it is cheap once the
// module is loaded) instead of being cached per device ordinal: a cached
// address would go stale after cudaDeviceReset or under another context on the
// same device.
attn_status_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(built-in scratch)");
  *out = p;
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                          const void* o, const void* dout, const float* lse,
                                          void* dq, void* dk, void* dv, int B, int H, int N,
                                          int d, int causal, float softmax_scale,
                                          attn_dtype_t dtype, cudaStream_t stream) {
  const size_t need = attn_bwd_workspace_size(B, H, N, d);
  if (need == 0) return fail(ATTN_ERR_INVALID_ARG, "B, H, N and d must be >= 1");
  if (need > kNoAllocScratchBytes)
    return fail(ATTN_ERR_INVALID_ARG,
                "problem needs " + std::to_string(need) +
                    " bytes of backward scratch; the built-in scratch of attn_bwd_noalloc holds " +
                    std::to_string(kNoAllocScratchBytes) + " bytes (use attn_bwd with a workspace)");
  // the device check first, so a device of the wrong architecture gets
  // ATTN_ERR_ARCH rather than a failed symbol lookup
  attn_status_t s = check_device();
  if (s != ATTN_OK) return s;
  void* scratch = nullptr;
  s = scratch_address(&scratch);
  if (s != ATTN_OK) return s;
  return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, kNoAllocScratchBytes, B, H, N, d,
                  causal, softmax_scale, dtype, stream);
}
