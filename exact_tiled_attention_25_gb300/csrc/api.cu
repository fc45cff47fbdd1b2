// The C ABI: argument validation, device checks, tensor maps, status word.
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "common.h"
#include "sm103_prims.cuh"

namespace attn {

namespace {

thread_local std::string g_last_error;

// One status word per device; kernels record the first internal error here.
__device__ int g_device_status;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

constexpr int kMaxDevices = 64;
int g_arch_ok[kMaxDevices];   // 0 unknown, 1 ok, 2 wrong arch (a property of the device)
std::mutex g_dev_mutex;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Pure argument checks: no CUDA call is made here, so they also run on a
// machine without a GPU.
attn_status_t check_shape(int B, int H, int N, int d, int causal) {
  if (B < 1 || H < 1 || N < 1) return fail(ATTN_ERR_INVALID_ARG, "B, H and N must be >= 1");
  if (d != 64 && d != 128 && d != 256)
    return fail(ATTN_ERR_INVALID_ARG, "d must be 64, 128 or 256");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  const double elems = static_cast<double>(B) * H * N * d;
  if (elems >= 2147483648.0) return fail(ATTN_ERR_INVALID_ARG, "B*H*N*d must be < 2^31");
  return ATTN_OK;
}

attn_status_t check_heads(int H, int H_kv) {
  if (H_kv < 1 || H_kv > H || H % H_kv != 0)
    return fail(ATTN_ERR_INVALID_ARG, "H_kv must divide H (1 <= H_kv <= H)");
  return ATTN_OK;
}

// A packed batch: B sequences, the longest max_seqlen tokens, total tokens.
attn_status_t check_packed(int B, int max_seqlen, int total, int H, int d, int causal) {
  if (B < 1 || H < 1 || max_seqlen < 1 || total < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, max_seqlen and total must be >= 1");
  if (d != 64 && d != 128 && d != 256)
    return fail(ATTN_ERR_INVALID_ARG, "d must be 64, 128 or 256");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (static_cast<double>(total) * H * d >= 2147483648.0)
    return fail(ATTN_ERR_INVALID_ARG, "total*H*d must be < 2^31");
  if (static_cast<double>(B) * H * (max_seqlen + 127) / 128 * 128 >= 2147483648.0)
    return fail(ATTN_ERR_INVALID_ARG, "B*H*max_seqlen too large");
  return ATTN_OK;
}

attn_status_t check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs) {
    if (p == nullptr) return fail(ATTN_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(p)) return fail(ATTN_ERR_INVALID_ARG, "tensor pointer not 16-byte aligned");
  }
  return ATTN_OK;
}

attn_status_t check_scale(float s) {
  if (!(s > 0.f) || !std::isfinite(s))
    return fail(ATTN_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
  return ATTN_OK;
}

}  // namespace

// Device check: compute capability 10.3, cached per device ordinal (the
// architecture does not change with the context).
attn_status_t check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
    e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
    g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  if (g_arch_ok[dev] != 1)
    return fail(ATTN_ERR_ARCH, "this library runs on compute capability 10.3 (GB300) only");
  return ATTN_OK;
}

attn_status_t fail(attn_status_t code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

attn_status_t fail_cuda(cudaError_t err, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorName(err) + " (" +
                 cudaGetErrorString(err) + ")";
  return ATTN_ERR_CUDA;
}

// Looked up on every call rather than cached per device ordinal, so the
// address always belongs to the current context (a cached one would go stale
// after cudaDeviceReset or under another context on the same device).
int* device_status_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

attn_status_t make_tmap_3d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner,
                           uint64_t rows, uint64_t planes, uint32_t box_inner,
                           uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {inner, rows, planes};
  cuuint64_t strides[2] = {inner * elem_bytes, inner * rows * elem_bytes};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                           : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return ATTN_OK;
}

attn_status_t make_tmap_4d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner,
                           uint64_t rows, uint64_t heads, uint64_t batches, uint64_t row_bytes,
                           uint64_t head_bytes, uint64_t batch_bytes, uint32_t box_inner,
                           uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[4] = {inner, rows, heads, batches};
  cuuint64_t strides[3] = {row_bytes, head_bytes, batch_bytes};
  cuuint32_t box[4] = {box_inner, box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                           : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (4-D) failed with CUresult " + std::to_string(r));
  return ATTN_OK;
}

attn_status_t set_smem(const void* kernel, int bytes) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(max dynamic shared memory)");
  return ATTN_OK;
}

// One thread waits on a barrier that nothing arrives on, through the same
// bounded wait every kernel uses; the wait gives up after limit_ns and the
// kernel records the timeout in the status word and returns.
__global__ void selftest_wait_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(&bar, 1);
  fence_mbar_init();
  const Abort ab{&abort_flag, status};
  mbar_wait_limit(&bar, 0, ab, kDevTimeoutSelftest, limit_ns);
}

}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case ATTN_ERR_ARCH: return "device is not compute capability 10.3";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "a kernel wait exceeded its time limit";
  }
  return "unknown status";
}

const char* attn_last_error(void) { return g_last_error.c_str(); }

size_t attn_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  return bwd_workspace_layout(B, H, N, d).total;
}

attn_status_t attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int H_kv, int N, int d, int causal, float softmax_scale,
                           attn_dtype_t dtype, cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_shape(B, H, N, d, causal)) != ATTN_OK) return s;
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  if ((s = check_ptrs({q, k, v, o, lse})) != ATTN_OK) return s;
  if ((s = check_scale(softmax_scale)) != ATTN_OK) return s;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_BF16 or ATTN_FP16");
  if ((s = check_device()) != ATTN_OK) return s;
  FwdParams p{q, k, v, o, lse, B, H, N, d, H_kv, nullptr, 0, causal, softmax_scale,
              dtype == ATTN_FP16 ? 1 : 0};
  return launch_fwd(p, stream);
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N, int d, int causal, float softmax_scale, attn_dtype_t dtype,
                       cudaStream_t stream) {
  return attn_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, causal, softmax_scale, dtype, stream);
}

attn_status_t attn_fwd_schedule(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int N, int d, int causal, float softmax_scale,
                                attn_dtype_t dtype, int schedule, cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_shape(B, H, N, d, causal)) != ATTN_OK) return s;
  if ((s = check_ptrs({q, k, v, o, lse})) != ATTN_OK) return s;
  if ((s = check_scale(softmax_scale)) != ATTN_OK) return s;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_BF16 or ATTN_FP16");
  if (schedule < 0 || schedule > (ATTN_SCHED_ONE_TILE | ATTN_SCHED_EAGER_RESCALE))
    return fail(ATTN_ERR_INVALID_ARG, "schedule must combine ATTN_SCHED_* flags");
  if (dtype != ATTN_BF16 || d == 256)
    return fail(ATTN_ERR_UNSUPPORTED, "schedule variants: bfloat16, d = 64 or 128");
  if ((s = check_device()) != ATTN_OK) return s;
  FwdParams p{q, k, v, o, lse, B, H, N, d, H, nullptr, 0, causal, softmax_scale, 0};
  return launch_fwd_sched(p, schedule, stream);
}

attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int* cu_seqlens, int B, int max_seqlen, int total, int H,
                              int H_kv, int d, int causal, float softmax_scale,
                              attn_dtype_t dtype, cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_packed(B, max_seqlen, total, H, d, causal)) != ATTN_OK) return s;
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  if ((s = check_ptrs({q, k, v, o, lse})) != ATTN_OK) return s;
  if (cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens must be a non-null, 4-byte aligned device array");
  if ((s = check_scale(softmax_scale)) != ATTN_OK) return s;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_BF16 or ATTN_FP16");
  if ((s = check_device()) != ATTN_OK) return s;
  FwdParams p{q, k, v, o, lse, B, H, max_seqlen, d, H_kv, cu_seqlens, total, causal,
              softmax_scale, dtype == ATTN_FP16 ? 1 : 0};
  return launch_fwd(p, stream);
}

// Shared by the backward entry points after their own shape checks.
static attn_status_t bwd_common(const void* q, const void* k, const void* v, const void* o,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                void* workspace, size_t workspace_bytes, size_t workspace_need,
                                const BwdWorkspace& w, int B, int H, int H_kv, int N, int d,
                                const int* cu_seqlens, int total, int causal,
                                float softmax_scale, attn_dtype_t dtype, cudaStream_t stream) {
  attn_status_t s;
  if ((s = check_ptrs({q, k, v, o, dout, lse, dq, dk, dv, workspace})) != ATTN_OK) return s;
  if ((s = check_scale(softmax_scale)) != ATTN_OK) return s;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_BF16 or ATTN_FP16");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < workspace_need)
    return fail(ATTN_ERR_INVALID_ARG, "workspace smaller than the workspace-size query returns");
  if (d == 256) return fail(ATTN_ERR_UNSUPPORTED, "the backward pass supports d = 64 and 128");
  if ((s = check_device()) != ATTN_OK) return s;
  char* ws = static_cast<char*>(workspace);
  BwdParams p{q,  k,  v,  o,  dout, lse, dq, dk, dv, reinterpret_cast<float*>(ws + w.dq_acc),
              reinterpret_cast<float*>(ws + w.lse2), reinterpret_cast<float*>(ws + w.delta),
              B,  H,  N,  d,  H_kv, cu_seqlens, total, causal, softmax_scale,
              dtype == ATTN_FP16 ? 1 : 0};
  return launch_bwd(p, stream);
}

attn_status_t attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           void* workspace, size_t workspace_bytes, int B, int H, int H_kv, int N,
                           int d, int causal, float softmax_scale, attn_dtype_t dtype,
                           cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_shape(B, H, N, d, causal)) != ATTN_OK) return s;
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  return bwd_common(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
                    attn_bwd_workspace_size(B, H, N, d), bwd_workspace_layout(B, H, N, d), B, H,
                    H_kv, N, d, nullptr, 0, causal, softmax_scale, dtype, stream);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                       int causal, float softmax_scale, attn_dtype_t dtype,
                       cudaStream_t stream) {
  return attn_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, H, N,
                      d, causal, softmax_scale, dtype, stream);
}

size_t attn_bwd_varlen_workspace_size(int B, int max_seqlen, int total, int H, int d) {
  if (B < 1 || max_seqlen < 1 || total < 1 || H < 1 || d < 1) return 0;
  return bwd_workspace_layout_packed(B, max_seqlen, total, H, d).total;
}

attn_status_t attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              void* workspace, size_t workspace_bytes, const int* cu_seqlens,
                              int B, int max_seqlen, int total, int H, int H_kv, int d,
                              int causal, float softmax_scale, attn_dtype_t dtype,
                              cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_packed(B, max_seqlen, total, H, d, causal)) != ATTN_OK) return s;
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  if (cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens must be a non-null, 4-byte aligned device array");
  return bwd_common(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
                    attn_bwd_varlen_workspace_size(B, max_seqlen, total, H, d),
                    bwd_workspace_layout_packed(B, max_seqlen, total, H, d), B, H, H_kv,
                    max_seqlen, d, cu_seqlens, total, causal, softmax_scale, dtype, stream);
}

attn_status_t attn_fp8_quantize(const float* q, const float* k, const float* v,
                                const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                uint8_t* v8, float* q_descale, float* k_descale,
                                float* v_descale, int B, int H, int N, int d, int per_tensor,
                                cudaStream_t stream) {
  return attn_fp8_quantize_gqa(q, k, v, hadamard_signs, q8, k8, v8, q_descale, k_descale,
                               v_descale, B, H, H, N, d, per_tensor, stream);
}

// Shared by the fixed-length pre-pass entry points (float32 or bfloat16 inputs).
static attn_status_t fp8_quantize_common(const void* q, const void* k, const void* v,
                                         const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                         uint8_t* v8, float* q_descale, float* k_descale,
                                         float* v_descale, int B, int H, int H_kv, int N, int d,
                                         int per_tensor, int in_bf16, cudaStream_t stream);

attn_status_t attn_fp8_quantize_gqa(const float* q, const float* k, const float* v,
                                    const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                    uint8_t* v8, float* q_descale, float* k_descale,
                                    float* v_descale, int B, int H, int H_kv, int N, int d,
                                    int per_tensor, cudaStream_t stream) {
  return fp8_quantize_common(q, k, v, hadamard_signs, q8, k8, v8, q_descale, k_descale, v_descale,
                             B, H, H_kv, N, d, per_tensor, 0, stream);
}

attn_status_t attn_fp8_quantize_bf16(const void* q, const void* k, const void* v,
                                     const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                     uint8_t* v8, float* q_descale, float* k_descale,
                                     float* v_descale, int B, int H, int H_kv, int N, int d,
                                     int per_tensor, cudaStream_t stream) {
  return fp8_quantize_common(q, k, v, hadamard_signs, q8, k8, v8, q_descale, k_descale, v_descale,
                             B, H, H_kv, N, d, per_tensor, 1, stream);
}

static attn_status_t fp8_quantize_common(const void* q, const void* k, const void* v,
                                         const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                         uint8_t* v8, float* q_descale, float* k_descale,
                                         float* v_descale, int B, int H, int H_kv, int N, int d,
                                         int per_tensor, int in_bf16, cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_shape(B, H, N, d, 0)) != ATTN_OK) return s;
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  if ((s = check_ptrs({q, k, v, q8, k8, v8, q_descale, k_descale, v_descale})) != ATTN_OK)
    return s;
  if (per_tensor != 0 && per_tensor != 1)
    return fail(ATTN_ERR_INVALID_ARG, "per_tensor must be 0 or 1");
  if (per_tensor && hadamard_signs)
    return fail(ATTN_ERR_INVALID_ARG, "the per-tensor comparator takes no Hadamard signs");
  if (hadamard_signs && !aligned16(hadamard_signs))
    return fail(ATTN_ERR_INVALID_ARG, "hadamard_signs not 16-byte aligned");
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 path supports d = 128");
  if ((s = check_device()) != ATTN_OK) return s;
  Fp8QuantParams p{{q, k, v}, {q8, k8, v8}, {q_descale, k_descale, v_descale}, hadamard_signs,
                   B, H, N, d, per_tensor, nullptr, nullptr, H_kv, nullptr, 0, in_bf16};
  return launch_fp8_quantize(p, stream);
}

attn_status_t attn_fp8_quantize_varlen(const float* q, const float* k, const float* v,
                                       const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                       uint8_t* v8, float* q_descale, float* k_descale,
                                       float* v_descale, const int* cu_seqlens, int B,
                                       int max_seqlen, int total, int H, int H_kv, int d,
                                       cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_packed(B, max_seqlen, total, H, d, 0)) != ATTN_OK) return s;
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  if ((s = check_ptrs({q, k, v, q8, k8, v8, q_descale, k_descale, v_descale})) != ATTN_OK)
    return s;
  if (cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens must be a non-null, 4-byte aligned device array");
  if (hadamard_signs && !aligned16(hadamard_signs))
    return fail(ATTN_ERR_INVALID_ARG, "hadamard_signs not 16-byte aligned");
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 path supports d = 128");
  if ((s = check_device()) != ATTN_OK) return s;
  Fp8QuantParams p{{q, k, v}, {q8, k8, v8}, {q_descale, k_descale, v_descale}, hadamard_signs,
                   B, H, max_seqlen, d, 0, nullptr, nullptr, H_kv, cu_seqlens, total};
  return launch_fp8_quantize(p, stream);
}

attn_status_t attn_fp8_quantize_rope(const float* q, const float* k, const float* v,
                                     const float* rope_cos, const float* rope_sin,
                                     const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                     uint8_t* v8, float* q_descale, float* k_descale,
                                     float* v_descale, int B, int H, int N, int d,
                                     cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_shape(B, H, N, d, 0)) != ATTN_OK) return s;
  if ((s = check_ptrs({q, k, v, rope_cos, rope_sin, q8, k8, v8, q_descale, k_descale,
                       v_descale})) != ATTN_OK)
    return s;
  if (hadamard_signs && !aligned16(hadamard_signs))
    return fail(ATTN_ERR_INVALID_ARG, "hadamard_signs not 16-byte aligned");
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 path supports d = 128");
  if ((s = check_device()) != ATTN_OK) return s;
  Fp8QuantParams p{{q, k, v}, {q8, k8, v8}, {q_descale, k_descale, v_descale}, hadamard_signs,
                   B, H, N, d, 0, rope_cos, rope_sin};
  return launch_fp8_quantize(p, stream);
}

attn_status_t attn_fp8_quantize_ex(const void* q, const void* k, const void* v, int input_bf16,
                                   const float* rope_cos, const float* rope_sin,
                                   const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                   uint8_t* v8, float* q_descale, float* k_descale,
                                   float* v_descale, const int* cu_seqlens, int B, int N,
                                   int total, int H, int H_kv, int d, int per_tensor,
                                   cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if (input_bf16 != 0 && input_bf16 != 1)
    return fail(ATTN_ERR_INVALID_ARG, "input_bf16 must be 0 or 1");
  if (cu_seqlens) {
    if ((s = check_packed(B, N, total, H, d, 0)) != ATTN_OK) return s;
    if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)
      return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
  } else {
    if ((s = check_shape(B, H, N, d, 0)) != ATTN_OK) return s;
  }
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  if ((s = check_ptrs({q, k, v, q8, k8, v8, q_descale, k_descale, v_descale})) != ATTN_OK)
    return s;
  if ((rope_cos == nullptr) != (rope_sin == nullptr))
    return fail(ATTN_ERR_INVALID_ARG, "give both rope_cos and rope_sin, or neither");
  if (rope_cos && (!aligned16(rope_cos) || !aligned16(rope_sin)))
    return fail(ATTN_ERR_INVALID_ARG, "rope tables must be 16-byte aligned");
  if (hadamard_signs && !aligned16(hadamard_signs))
    return fail(ATTN_ERR_INVALID_ARG, "hadamard_signs not 16-byte aligned");
  if (per_tensor != 0 && per_tensor != 1)
    return fail(ATTN_ERR_INVALID_ARG, "per_tensor must be 0 or 1");
  if (per_tensor && (hadamard_signs || rope_cos || cu_seqlens))
    return fail(ATTN_ERR_INVALID_ARG,
                "the per-tensor comparator takes fixed-length inputs without Hadamard or rotation");
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 path supports d = 128");
  if ((s = check_device()) != ATTN_OK) return s;
  Fp8QuantParams p{{q, k, v}, {q8, k8, v8}, {q_descale, k_descale, v_descale}, hadamard_signs,
                   B, H, N, d, per_tensor, rope_cos, rope_sin, H_kv, cu_seqlens,
                   cu_seqlens ? total : 0, input_bf16};
  return launch_fp8_quantize(p, stream);
}

size_t attn_decode_workspace_size(int B, int H, int H_kv, int n_q, int d, int max_seqlen) {
  if (B < 1 || H < 1 || H_kv < 1 || n_q < 1 || d < 1 || max_seqlen < 1) return 0;
  return decode_workspace_bytes(B, H, H_kv, n_q, d, max_seqlen);
}

attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int* block_table, const int* seq_lens, void* o, float* lse,
                                void* workspace, size_t workspace_bytes, int B, int H, int H_kv,
                                int n_q, int d, int num_pages, int page_size, int max_pages,
                                int max_seqlen, int causal, float softmax_scale,
                                attn_dtype_t dtype, cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if (B < 1 || H < 1 || n_q < 1 || num_pages < 1 || max_pages < 1 || max_seqlen < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, n_q, num_pages, max_pages and max_seqlen must be >= 1");
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  if (d != 64 && d != 128) return fail(ATTN_ERR_INVALID_ARG, "decode supports d = 64 and 128");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if ((H / H_kv) * n_q > 128)
    return fail(ATTN_ERR_UNSUPPORTED, "(H / H_kv) * n_q must be <= 128 (one query tile)");
  if (page_size < 8 || page_size > 65536 || (page_size & (page_size - 1)) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "page_size must be a power of two in [8, 65536]");
  if (static_cast<long long>(max_pages) * page_size > 2147483647LL ||
      static_cast<double>(num_pages) * page_size * H_kv * d >= 9.0e15)
    return fail(ATTN_ERR_INVALID_ARG, "cache too large");
  if (static_cast<double>(B) * H * n_q * d >= 2147483648.0)
    return fail(ATTN_ERR_INVALID_ARG, "B*H*n_q*d must be < 2^31");
  if ((s = check_ptrs({q, k_cache, v_cache, o, lse, workspace})) != ATTN_OK) return s;
  if (!block_table || !seq_lens || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "block_table and seq_lens must be non-null, 4-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < attn_decode_workspace_size(B, H, H_kv, n_q, d, max_seqlen))
    return fail(ATTN_ERR_INVALID_ARG, "workspace smaller than attn_decode_workspace_size()");
  if ((s = check_scale(softmax_scale)) != ATTN_OK) return s;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_BF16 or ATTN_FP16");
  if ((s = check_device()) != ATTN_OK) return s;
  const DecodeSplits sp = decode_splits(B, H_kv, max_seqlen);
  const size_t rows = static_cast<size_t>(B) * H * n_q * sp.splits;
  char* ws = static_cast<char*>(workspace);
  DecodeParams p{q, k_cache, v_cache, block_table, seq_lens, o, lse,
                 reinterpret_cast<float*>(ws),
                 reinterpret_cast<float*>(ws + align_up(rows * d * sizeof(float), 256)),
                 B, H, H_kv, n_q, d, num_pages, page_size, max_pages, max_seqlen, causal,
                 softmax_scale, dtype == ATTN_FP16 ? 1 : 0};
  return launch_decode(p, stream);
}

attn_status_t attn_decode_paged_fp8(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                    const float* k_descale, const float* v_descale,
                                    const float* hadamard_signs, const int* block_table,
                                    const int* seq_lens, void* o, float* lse, void* workspace,
                                    size_t workspace_bytes, int B, int H, int H_kv, int n_q, int d,
                                    int num_pages, int page_size, int max_pages, int max_seqlen,
                                    int causal, float softmax_scale, attn_dtype_t dtype,
                                    cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if (B < 1 || H < 1 || n_q < 1 || num_pages < 1 || max_pages < 1 || max_seqlen < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, n_q, num_pages, max_pages and max_seqlen must be >= 1");
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 decode supports d = 128");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if ((H / H_kv) * n_q > 128)
    return fail(ATTN_ERR_UNSUPPORTED, "(H / H_kv) * n_q must be <= 128 (one query tile)");
  if (page_size < 16 || page_size > 65536 || (page_size & (page_size - 1)) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "page_size must be a power of two in [16, 65536] for an FP8 cache");
  if (static_cast<long long>(max_pages) * page_size > 2147483647LL ||
      static_cast<double>(num_pages) * page_size * H_kv * d >= 9.0e15)
    return fail(ATTN_ERR_INVALID_ARG, "cache too large");
  if (static_cast<double>(B) * H * n_q * d >= 2147483648.0)
    return fail(ATTN_ERR_INVALID_ARG, "B*H*n_q*d must be < 2^31");
  if ((s = check_ptrs({q, k_cache, v_cache, o, lse, workspace, k_descale, v_descale})) != ATTN_OK)
    return s;
  if (hadamard_signs && (reinterpret_cast<uintptr_t>(hadamard_signs) & 15u))
    return fail(ATTN_ERR_INVALID_ARG, "hadamard_signs must be 16-byte aligned");
  if (!block_table || !seq_lens || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "block_table and seq_lens must be non-null, 4-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < attn_decode_workspace_size(B, H, H_kv, n_q, d, max_seqlen))
    return fail(ATTN_ERR_INVALID_ARG, "workspace smaller than attn_decode_workspace_size()");
  if ((s = check_scale(softmax_scale)) != ATTN_OK) return s;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_BF16 or ATTN_FP16");
  if ((s = check_device()) != ATTN_OK) return s;
  const DecodeSplits sp = decode_splits(B, H_kv, max_seqlen);
  const size_t rows = static_cast<size_t>(B) * H * n_q * sp.splits;
  char* ws = static_cast<char*>(workspace);
  DecodeParams p{q, k_cache, v_cache, block_table, seq_lens, o, lse,
                 reinterpret_cast<float*>(ws),
                 reinterpret_cast<float*>(ws + align_up(rows * d * sizeof(float), 256)),
                 B, H, H_kv, n_q, d, num_pages, page_size, max_pages, max_seqlen, causal,
                 softmax_scale, dtype == ATTN_FP16 ? 1 : 0,
                 1, k_descale, v_descale, hadamard_signs};
  return launch_decode(p, stream);
}

attn_status_t attn_fwd_fp8(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                           const float* q_descale, const float* k_descale,
                           const float* v_descale, void* o, float* lse, int B, int H, int N,
                           int d, int causal, float softmax_scale, cudaStream_t stream) {
  return attn_fwd_fp8_gqa(q8, k8, v8, q_descale, k_descale, v_descale, o, lse, B, H, H, N, d,
                          causal, softmax_scale, stream);
}

attn_status_t attn_fwd_fp8_schedule(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                                    const float* q_descale, const float* k_descale,
                                    const float* v_descale, void* o, float* lse, int B, int H,
                                    int N, int d, int causal, float softmax_scale, int schedule,
                                    cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_shape(B, H, N, d, causal)) != ATTN_OK) return s;
  if ((s = check_ptrs({q8, k8, v8, o, lse})) != ATTN_OK) return s;
  if (!q_descale || !k_descale || !v_descale)
    return fail(ATTN_ERR_INVALID_ARG, "null descale pointer");
  if ((s = check_scale(softmax_scale)) != ATTN_OK) return s;
  // 0, ATTN_SCHED_EXP2_NONE, or ATTN_SCHED_EXP2_POLY with an optional share of 1..4
  // eighths in bits 8..11
  const int eighths = (schedule >> 8) & 15;
  if (schedule != 0 && schedule != ATTN_SCHED_EXP2_NONE &&
      ((schedule & ~(15 << 8)) != ATTN_SCHED_EXP2_POLY || eighths > 4))
    return fail(ATTN_ERR_INVALID_ARG,
                "schedule must be 0, ATTN_SCHED_EXP2_NONE, ATTN_SCHED_EXP2_POLY or "
                "ATTN_SCHED_EXP2_EIGHTHS(1..4)");
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 path supports d = 128");
  if ((s = check_device()) != ATTN_OK) return s;
  Fp8FwdParams p{q8, k8, v8, q_descale, k_descale, v_descale, o, lse, B, H, N, d, causal,
                 softmax_scale, H};
  // the kernels count the share in sixteenths
  p.exp2_poly = schedule == 0 ? -1 : schedule == ATTN_SCHED_EXP2_NONE ? 0 : 2 * (eighths == 0 ? 2 : eighths);
  return launch_fwd_fp8(p, stream);
}

attn_status_t attn_selftest_exp2(const float* x, float* y_poly, float* y_mufu, long long n,
                                 cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if (n < 1 || n > (1ll << 30)) return fail(ATTN_ERR_INVALID_ARG, "n must be in [1, 2^30]");
  if (!x || !y_poly || !y_mufu) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if ((s = check_device()) != ATTN_OK) return s;
  return launch_exp2_selftest(x, y_poly, y_mufu, n, stream);
}

attn_status_t attn_fwd_fp8_varlen(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                                  const float* q_descale, const float* k_descale,
                                  const float* v_descale, void* o, float* lse,
                                  const int* cu_seqlens, int B, int max_seqlen, int total, int H,
                                  int H_kv, int d, int causal, float softmax_scale,
                                  cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_packed(B, max_seqlen, total, H, d, causal)) != ATTN_OK) return s;
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  if ((s = check_ptrs({q8, k8, v8, o, lse})) != ATTN_OK) return s;
  if (!q_descale || !k_descale || !v_descale)
    return fail(ATTN_ERR_INVALID_ARG, "null descale pointer");
  if (cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens must be a non-null, 4-byte aligned device array");
  if ((s = check_scale(softmax_scale)) != ATTN_OK) return s;
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 path supports d = 128");
  if ((s = check_device()) != ATTN_OK) return s;
  Fp8FwdParams p{q8, k8, v8, q_descale, k_descale, v_descale, o, lse, B, H, max_seqlen, d, causal,
                 softmax_scale, H_kv, cu_seqlens, total};
  return launch_fwd_fp8(p, stream);
}

attn_status_t attn_fwd_fp8_gqa(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                               const float* q_descale, const float* k_descale,
                               const float* v_descale, void* o, float* lse, int B, int H,
                               int H_kv, int N, int d, int causal, float softmax_scale,
                               cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_shape(B, H, N, d, causal)) != ATTN_OK) return s;
  if ((s = check_heads(H, H_kv)) != ATTN_OK) return s;
  if ((s = check_ptrs({q8, k8, v8, o, lse})) != ATTN_OK) return s;
  if (!q_descale || !k_descale || !v_descale)
    return fail(ATTN_ERR_INVALID_ARG, "null descale pointer");
  if ((s = check_scale(softmax_scale)) != ATTN_OK) return s;
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 path supports d = 128");
  if ((s = check_device()) != ATTN_OK) return s;
  Fp8FwdParams p{q8, k8, v8, q_descale, k_descale, v_descale, o, lse, B, H, N, d, causal,
                 softmax_scale, H_kv};
  return launch_fwd_fp8(p, stream);
}

attn_status_t attn_selftest_wait_timeout(unsigned limit_us, cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if (limit_us < 1 || limit_us > 1000000)
    return fail(ATTN_ERR_INVALID_ARG, "limit_us must be in [1, 1000000]");
  if ((s = check_device()) != ATTN_OK) return s;
  int* status = device_status_word();
  if (!status) return fail(ATTN_ERR_CUDA, "status word unavailable");
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status, static_cast<uint64_t>(limit_us) * 1000ull);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "self-test launch");
  return ATTN_OK;
}

attn_status_t attn_get_device_status(cudaStream_t stream) {
  g_last_error.clear();
  attn_status_t s;
  if ((s = check_device()) != ATTN_OK) return s;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
  int* word = device_status_word();
  if (!word) return fail(ATTN_ERR_CUDA, "status word unavailable");
  int value = 0;
  e = cudaMemcpy(&value, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e, "reading the status word");
  if (value == 0) return ATTN_OK;
  const int zero = 0;
  e = cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail_cuda(e, "clearing the status word");
  static const char* roles[] = {"?",        "load",   "mma",
                                "softmax",  "epilogue", "reduce",
                                "shared-memory alignment", "self-test"};
  const int role = (value >> 8) & 0xF;
  if (value == kDevBadSeqlens)
    return fail(ATTN_ERR_INVALID_ARG,
                "cu_seqlens inconsistent (an entry outside [0, total], decreasing, or a sequence "
                "longer than max_seqlen), or a decode seq_lens / block_table entry out of range; "
                "those sequences or pages were skipped");
  return fail(ATTN_ERR_TIMEOUT, std::string("kernel wait timed out in role ") +
                                    (role < 8 ? roles[role] : "?") + " (code " +
                                    std::to_string(value) + ")");
}

}  // extern "C"
