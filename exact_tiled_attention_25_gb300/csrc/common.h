// Host-side internals shared by the kernel translation units and the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>

#include "../../include/attn_gb300.h"

namespace attn {

// Record a detail message for attn_last_error() and return `code`.
attn_status_t fail(attn_status_t code, const std::string& msg);
attn_status_t fail_cuda(cudaError_t err, const char* what);

// Device address of the status word in the current context (nullptr if the
// lookup fails).
int* device_status_word();

// Compute capability 10.3 check of the current device (ATTN_ERR_ARCH if not).
attn_status_t check_device();

// 3-D tensor map over a contiguous [planes][rows][inner] array with a
// (box_inner x box_rows x 1) box and 128-byte swizzle.  elem_bytes is 1 or 2
// (raw bytes / 16-bit words), or 4 (float32, the type a reduce-add needs).
attn_status_t make_tmap_3d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner,
                           uint64_t rows, uint64_t planes, uint32_t box_inner,
                           uint32_t box_rows);

// 4-D map over {d, rows, heads, batches} with byte strides for rows, heads and
// batches (each a multiple of 16); box {box_inner, box_rows, 1, 1}, 128-byte
// swizzle.  Covers [B, H, N, d] and packed [total, H, d] alike.
attn_status_t make_tmap_4d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner,
                           uint64_t rows, uint64_t heads, uint64_t batches, uint64_t row_bytes,
                           uint64_t head_bytes, uint64_t batch_bytes, uint32_t box_inner,
                           uint32_t box_rows);

// Opt a kernel into more than 48 KB of dynamic shared memory (once per kernel).
attn_status_t set_smem(const void* kernel, int bytes);

struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, N, d;     // N: sequence length, or the longest one of a packed batch
  int H_kv;           // key/value heads (H % H_kv == 0)
  const int* cu_seqlens;   // device [B + 1] for a packed batch, else nullptr
  int total;          // tokens of a packed batch (cu_seqlens[B])
  int causal;
  float scale;
  int fp16;   // 0 = bf16, 1 = fp16
};

struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;   // float32 scratch in dQ's layout
  float* lse2;     // [B, H, Npad] float32 scratch: -LSE * log2(e), -inf padding
  float* delta;    // [B, H, Npad] float32 scratch: -rowsum(dO * O), 0 padding
  int B, H, N, d;  // N: sequence length, or the longest one of a packed batch
  int H_kv;        // key/value heads (H % H_kv == 0)
  const int* cu_seqlens;   // device [B + 1] for a packed batch, else nullptr
  int total;       // tokens of a packed batch
  int causal;
  float scale;
  int fp16;
};

struct Fp8QuantParams {
  const void* src[3];                // float32, or bfloat16 when in_bf16
  uint8_t* dst[3];
  float* descale[3];
  const float* signs;
  int B, H, N, d;
  int per_tensor;
  const float* rope_cos = nullptr;   // [N, d/2] rotary tables (block mode), or nullptr
  const float* rope_sin = nullptr;
  int H_kv = 0;                      // heads of K and V (0: H)
  const int* cu_seqlens = nullptr;   // packed batch: device [B + 1] offsets (N = longest)
  int total = 0;                     // packed batch: tokens
  int in_bf16 = 0;                   // inputs are bfloat16 (block and per-tensor modes)
};

struct Fp8FwdParams {
  const uint8_t* q8;
  const uint8_t* k8;
  const uint8_t* v8;
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  void* o;
  float* lse;
  int B, H, N, d;
  int causal;
  float scale;
  int H_kv;   // heads of K and V (H % H_kv == 0)
  const int* cu_seqlens = nullptr;   // packed batch: device [B + 1] offsets (N = longest)
  int total = 0;                     // packed batch: tokens
  int exp2_poly = -1;                // sixteenths of the exponentials on the FMA pipe (0, 1, 2, 4, 6, 8); -1: the library's choice
};

attn_status_t launch_fwd(const FwdParams& p, cudaStream_t stream);
// exp2_poly2 and ex2.approx on the same n inputs (diagnostic).
attn_status_t launch_exp2_selftest(const float* x, float* y_poly, float* y_mufu, long long n,
                                   cudaStream_t stream);
// Schedule variants of the forward kernel (ATTN_SCHED_* flags), for measurement.
attn_status_t launch_fwd_sched(const FwdParams& p, int sched, cudaStream_t stream);
// Persistent forward (cluster launch control) for packed causal batches.
attn_status_t launch_fwd_persistent(const FwdParams& p, cudaStream_t stream);
attn_status_t launch_bwd(const BwdParams& p, cudaStream_t stream);
attn_status_t launch_fp8_quantize(const Fp8QuantParams& p, cudaStream_t stream);
attn_status_t launch_fwd_fp8(const Fp8FwdParams& p, cudaStream_t stream);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Backward scratch layout: dQ accumulator, then L*log2(e) and D, each padded
// to a multiple of 128 rows per head; every part 256-byte aligned.
struct BwdWorkspace {
  size_t dq_acc, lse2, delta, total;
};
// dq_rows: rows of d floats in the dQ accumulator; rows_pad: entries of each
// padded row vector.
inline BwdWorkspace bwd_workspace_layout_rows(size_t dq_rows, size_t rows_pad, int d) {
  const size_t rows = dq_rows;
  BwdWorkspace w;
  w.dq_acc = 0;
  w.lse2 = align_up(rows * d * sizeof(float), 256);
  w.delta = w.lse2 + align_up(rows_pad * sizeof(float), 256);
  w.total = w.delta + align_up(rows_pad * sizeof(float), 256);
  return w;
}

inline BwdWorkspace bwd_workspace_layout(int B, int H, int N, int d) {
  return bwd_workspace_layout_rows(static_cast<size_t>(B) * H * N,
                                   static_cast<size_t>(B) * H * ((static_cast<size_t>(N) + 127) / 128 * 128), d);
}

// A packed batch: dQ accumulator [total, H, d]; row vectors padded per (b, h)
// to the longest sequence.
inline BwdWorkspace bwd_workspace_layout_packed(int B, int max_seqlen, int total, int H, int d) {
  return bwd_workspace_layout_rows(static_cast<size_t>(total) * H,
                                   static_cast<size_t>(B) * H *
                                       ((static_cast<size_t>(max_seqlen) + 127) / 128 * 128), d);
}

// Paged decode (few new query tokens per sequence against a paged cache).
struct DecodeParams {
  const void* q;            // [B, H, n_q, d]
  const void* k_cache;      // [num_pages, page_size, H_kv, d]
  const void* v_cache;
  const int* block_table;   // [B, max_pages]
  const int* seq_lens;      // [B]
  void* o;                  // [B, H, n_q, d]
  float* lse;               // [B, H, n_q]
  float* o_part;            // workspace: [B, H, n_q, splits, d] float32
  float* lse_part;          // workspace: [B, H, n_q, splits] float32
  int B, H, H_kv, n_q, d;
  int num_pages, page_size, max_pages, max_seqlen;
  int causal;
  float scale;
  int fp16;
  // e4m3 cache (d = 128): codes in k_cache / v_cache, one float32 descale per
  // (physical page, key/value head), optional key-transform signs
  int fp8 = 0;
  const float* k_descale = nullptr;   // [num_pages, H_kv]
  const float* v_descale = nullptr;
  const float* signs = nullptr;       // [d] of +-1, or nullptr
};

// Key-range splits of a decode call, each a whole number of 128-key tiles.
// One CTA runs per SM at a time, so the split size minimises the modelled time
// ceil(CTAs / 152) waves x (tiles per CTA + about 1.5 tiles of per-CTA start-up
// and drain), trading the last wave's idle SMs against start-up costs.
struct DecodeSplits {
  int splits, tiles_per_split;
};
inline DecodeSplits decode_splits(int B, int H_kv, int max_seqlen) {
  const int ntiles = (max_seqlen + 127) / 128;
  const long long base = static_cast<long long>(B) * H_kv;
  int best_tps = ntiles;
  double best = 1e300;
  for (int tps = 1; tps <= ntiles; ++tps) {
    const long long splits = (ntiles + tps - 1) / tps;
    if (tps > 1 && (ntiles + tps - 2) / (tps - 1) == splits) continue;   // same split count
    const long long waves = (base * splits + 151) / 152;
    const double cost = static_cast<double>(waves) * (tps + 1.5);
    if (cost < best) {
      best = cost;
      best_tps = tps;
    }
  }
  return {(ntiles + best_tps - 1) / best_tps, best_tps};
}

inline size_t decode_workspace_bytes(int B, int H, int H_kv, int n_q, int d, int max_seqlen) {
  const DecodeSplits sp = decode_splits(B, H_kv, max_seqlen);
  const size_t rows = static_cast<size_t>(B) * H * n_q * sp.splits;
  return align_up(rows * d * sizeof(float), 256) + align_up(rows * sizeof(float), 256);
}

attn_status_t launch_decode(const DecodeParams& p, cudaStream_t stream);

}  // namespace attn
