/*
 * attn_gb300 -- exact tiled softmax attention for one NVIDIA GB300 (sm_103a).
 *
 * Public C ABI of libattn_gb300.so.  Plain pointers and sizes only.
 *
 * What is computed.  For every batch b and head h, with S = softmax_scale * Q K^T
 * (N x N, keys j > i set to -inf when causal != 0):
 *     O   = softmax(S) V                        (row softmax)
 *     LSE = m + log(l)                          (natural log; m = row max of S,
 *                                                l = sum_j exp(S_ij - m))
 * "FlashAttention-3: Hopper Asynchrony and FP8 Attention", section "Symbol Map"
 * (O_i, m_i, l_i, L_i = m_i + log(l_i)) and "Putting It Together", step 7 (only O
 * and L are written).  The result is exact attention up to floating-point
 * rounding: S and P never reach global memory; the kernels walk key/value tiles
 * with the online-softmax recurrence.  The causal mask is lower-triangular with
 * top-left alignment (query i sees keys 0..i).
 *
 * Layout.  Every Q/K/V/O/dO/dQ/dK/dV tensor is [B, H, N, d], contiguous, d fastest
 * ("BHND").  LSE and the FP8 descales are contiguous [B, H, N] and
 * [B, H, ceil(N/128)] float32 arrays.  All pointers are DEVICE pointers on the
 * current CUDA device, 16-byte aligned (a TMA requirement); the caller owns them.
 *
 * Supported shapes.  d in {64, 128, 256} for the forward passes, d in {64, 128}
 * for the backward pass, d = 128 for the FP8 pass; N >= 1; B, H >= 1;
 * B * H * N * d < 2^31.
 *
 * Errors.  Arguments are validated before anything is launched; a bad argument
 * returns ATTN_ERR_INVALID_ARG, an unsupported (valid) shape ATTN_ERR_UNSUPPORTED,
 * a device that is not compute capability 10.3 ATTN_ERR_ARCH, a failed CUDA call
 * ATTN_ERR_CUDA (attn_last_error() then names it).  Launches are asynchronous on
 * `stream`; results are ready when the stream has reached them.  A kernel never
 * traps: if one of its internal waits exceeds its time limit it records the
 * fact in a device status word and returns early, and attn_get_device_status()
 * reports ATTN_ERR_TIMEOUT.
 *
 * Memory.  The library allocates no device memory per call.  It holds one
 * 4-byte status word per device (a static device variable).  Scratch for the
 * backward pass is supplied by the caller (attn_bwd_workspace_size()).
 *
 * Thread safety.  Calls may come from several host threads; the status word is
 * shared by all calls on a device.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t in the CUDA runtime headers.  NULL = legacy default stream. */
typedef struct CUstream_st* cudaStream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,
  ATTN_ERR_UNSUPPORTED = 2,
  ATTN_ERR_ARCH = 3,
  ATTN_ERR_CUDA = 4,
  ATTN_ERR_TIMEOUT = 5
} attn_status_t;

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1 } attn_dtype_t;

/*
 * attn_fwd -- BF16/FP16 forward.
 *   q, k, v : [B, H, N, d] in `dtype` (read only)
 *   o       : [B, H, N, d] in `dtype` (written)
 *   lse     : [B, H, N] float32 (written), natural-log LSE of the scaled,
 *             masked scores; input to attn_bwd.
 *   causal  : 0 or 1.   softmax_scale: > 0, finite (commonly 1/sqrt(d)).
 * Source: "FlashAttention-3: Hopper Asynchrony and FP8 Attention", sections
 * "Symbol Map", "Producer-consumer asynchrony", "Ping-pong scheduling",
 * "Two-stage WGMMA-softmax pipeline", "Putting It Together".
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int N, int d, int causal, float softmax_scale,
                       attn_dtype_t dtype, cudaStream_t stream);

/*
 * Schedule variants of attn_fwd, for measurement only (the ablation of the
 * forward pipeline); flags combine with bitwise or.
 */
enum {
  ATTN_SCHED_DEFAULT = 0,
  ATTN_SCHED_ONE_TILE = 1,       /* one 128-row query tile per CTA: while its softmax
                                    runs, the tensor core has no second tile to work on */
  ATTN_SCHED_EAGER_RESCALE = 2,  /* rescale the output accumulator whenever the row max
                                    grows, instead of only when it grows by more than 2^8 */
  ATTN_SCHED_EXP2_POLY = 4,      /* FP8 forward only: part of the exponentials on the FMA
                                    pipe (a fitted cubic) instead of the MUFU unit; the
                                    share is set in eighths by ATTN_SCHED_EXP2_EIGHTHS,
                                    a quarter when none is given */
  ATTN_SCHED_EXP2_NONE = 8       /* FP8 forward only: every exponential on the MUFU unit */
};

/* The FMA-pipe share of the FP8 forward's exponentials, k of every 8 (k = 1..4), as a
   schedule value: ATTN_SCHED_EXP2_POLY with k in bits 8..11. */
#define ATTN_SCHED_EXP2_EIGHTHS(k) (ATTN_SCHED_EXP2_POLY | ((k) << 8))

/*
 * attn_fwd_schedule -- attn_fwd with a schedule variant.  `schedule` is a
 * combination of the ATTN_SCHED_* flags; ATTN_SCHED_DEFAULT is exactly attn_fwd.
 * Every variant computes the same O and LSE (up to rounding); only the order of
 * work on the GPU changes.  Limits: bfloat16, d = 64 or 128 (other shapes return
 * ATTN_ERR_UNSUPPORTED); an unknown flag returns ATTN_ERR_INVALID_ARG.  Other
 * arguments, errors and semantics as attn_fwd.
 * Source: "FlashAttention-3: Hopper Asynchrony and FP8 Attention", sections
 * "How we know: H100 attention benchmarks" (the pipeline ablation: throughput
 * with and without the overlap of softmax and matrix multiplies),
 * "Ping-pong scheduling" (a second tile's matrix multiplies under one tile's
 * softmax) and "Symbol Map" (the numerator rescale when the running max grows).
 */
attn_status_t attn_fwd_schedule(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int N, int d, int causal, float softmax_scale,
                                attn_dtype_t dtype, int schedule, cudaStream_t stream);

/*
 * attn_fwd_gqa -- attn_fwd with grouped-query attention: the H query heads
 * share H_kv key/value heads (1 <= H_kv <= H, H % H_kv == 0); query head h
 * reads key/value head h / (H / H_kv).  H_kv = H is attn_fwd, H_kv = 1 is
 * multi-query attention.
 *   q, o : [B, H, N, d];   k, v : [B, H_kv, N, d];   lse : [B, H, N] float32.
 * Other arguments, errors and semantics as attn_fwd.
 * Source: "FlashAttention 3 Hardware Acceleration: Hopper GPU Strategies for
 * Long-Context Enterprise Inference Optimization", section "Runtime Kernel
 * Selection" (grouped query attention patterns).
 */
attn_status_t attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int H_kv, int N, int d, int causal, float softmax_scale,
                           attn_dtype_t dtype, cudaStream_t stream);

/*
 * attn_fwd_varlen -- forward over a batch of B sequences of different lengths
 * packed back to back without padding, with grouped-query attention.
 *   q, o       : [total, H, d] in `dtype` (token-major, d fastest)
 *   k, v       : [total, H_kv, d]
 *   lse        : [H, total] float32
 *   cu_seqlens : DEVICE int32 [B + 1]; sequence b is tokens [cu_seqlens[b],
 *                cu_seqlens[b+1]); cu_seqlens[0] = 0, non-decreasing,
 *                cu_seqlens[B] = total.  Empty sequences are allowed.
 *   max_seqlen : >= the longest sequence (it sizes the grid).
 * Attention and the causal mask act within each sequence (query i of a sequence
 * sees that sequence's keys 0..i).  The host checks shapes and pointers; the
 * device checks each sequence against total and max_seqlen, skips any that
 * does not fit, and reports it through attn_get_device_status()
 * (ATTN_ERR_INVALID_ARG).
 * Source: "FlashAttention 3 Hardware Acceleration: Hopper GPU Strategies for
 * Long-Context Enterprise Inference Optimization", sections "GPU Compatibility
 * and Enablement Matrix" (variable-length sequence handling) and "Runtime
 * Kernel Selection" (grouped query attention).
 */
attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int* cu_seqlens, int B, int max_seqlen, int total, int H,
                              int H_kv, int d, int causal, float softmax_scale,
                              attn_dtype_t dtype, cudaStream_t stream);

/*
 * attn_bwd_workspace_size -- bytes of device scratch attn_bwd needs:
 * a float32 dQ accumulator [B, H, N, d] and two float32 row vectors (-L * log2(e)
 * and -D, D = rowsum(dO * O)) padded to a multiple of 128 rows per head, each
 * part 256-byte aligned.  Returns 0 for invalid sizes.  Pure arithmetic on the
 * sizes: no CUDA call, usable before any device is chosen.
 * Source: the global dQ that "FlashAttention-3: Hopper Asynchrony and FP8
 * Attention", section "Backward warp specialization", has the dQ-writer add
 * local tiles into (here a float32 accumulator, converted at the end); the
 * caller allocates it once up front, as "FlashAttention 3 Hardware Acceleration:
 * Hopper GPU Strategies for Long-Context Enterprise Inference Optimization",
 * sections "Poor Memory Allocation" (pre-allocated workspace buffers) and
 * "Memory Fragmentation" (workspace kept apart from long-lived buffers) advise.
 */
size_t attn_bwd_workspace_size(int B, int H, int N, int d);

/*
 * attn_bwd -- BF16/FP16 backward: dQ, dK, dV of sum(O * dO).
 *   q, k, v, o, dout : [B, H, N, d] in `dtype`; o and lse from attn_fwd with
 *                      the same q, k, v, causal and softmax_scale.
 *   lse              : [B, H, N] float32.
 *   dq, dk, dv       : [B, H, N, d] in `dtype` (written).
 *   workspace        : device scratch of at least attn_bwd_workspace_size()
 *                      bytes, 256-byte aligned; its contents on entry do not
 *                      matter and are overwritten.
 * P and dS are recomputed from LSE ("FlashAttention-3: Hopper Asynchrony and
 * FP8 Attention", section "Backward warp specialization"): a row-dot pre-pass
 * D_i = dO_i . O_i, a key/value-tile-outer main kernel that accumulates dK, dV
 * on chip and adds dQ partial tiles into the float32 accumulator, and a final
 * conversion of dQ.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                       int causal, float softmax_scale, attn_dtype_t dtype,
                       cudaStream_t stream);

/*
 * attn_bwd_gqa -- attn_bwd with grouped-query attention (see attn_fwd_gqa):
 *   q, o, dout, dq : [B, H, N, d];   k, v, dk, dv : [B, H_kv, N, d];
 *   lse : [B, H, N].  dK and dV of a shared key/value head are the sums over
 *   the H / H_kv query heads that read it; one CTA per key tile and key/value
 *   head accumulates them over the whole group on chip, so they need no
 *   atomics.  The workspace is attn_bwd_workspace_size(B, H, N, d).
 * Source: as attn_bwd, and "FlashAttention 3 Hardware Acceleration: Hopper GPU
 * Strategies for Long-Context Enterprise Inference Optimization", section
 * "Runtime Kernel Selection" (grouped query attention).
 */
attn_status_t attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           void* workspace, size_t workspace_bytes, int B, int H, int H_kv, int N,
                           int d, int causal, float softmax_scale, attn_dtype_t dtype,
                           cudaStream_t stream);

/*
 * attn_bwd_varlen_workspace_size -- bytes of device scratch attn_bwd_varlen
 * needs: a float32 dQ accumulator [total, H, d] and two float32 row vectors
 * (-L * log2(e) and -D) of B * H * (max_seqlen rounded up to 128) entries,
 * each part 256-byte aligned.  Returns 0 for invalid sizes.
 */
size_t attn_bwd_varlen_workspace_size(int B, int max_seqlen, int total, int H, int d);

/*
 * attn_bwd_varlen -- backward of attn_fwd_varlen over the same packed batch:
 *   q, o, dout, dq : [total, H, d];   k, v, dk, dv : [total, H_kv, d];
 *   lse : [H, total] from attn_fwd_varlen;   cu_seqlens, max_seqlen, total as
 *   there (device-checked the same way).  d = 64 or 128.
 * Source: as attn_bwd and attn_fwd_varlen.
 */
attn_status_t attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              void* workspace, size_t workspace_bytes, const int* cu_seqlens,
                              int B, int max_seqlen, int total, int H, int H_kv, int d,
                              int causal, float softmax_scale, attn_dtype_t dtype,
                              cudaStream_t stream);

/*
 * attn_bwd_noalloc -- attn_bwd for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for code that
 * may not call cudaMalloc (or any allocating routine) itself, such as a
 * runtime without its own device allocator.  Arguments are those of attn_bwd
 * without the workspace: the scratch comes from a 64 MiB array built into the
 * library (held on every GPU that loads the library until the process exits).
 *   - Problems whose attn_bwd_workspace_size() exceeds 64 MiB are rejected with
 *     ATTN_ERR_INVALID_ARG and a message naming the sizes.
 *   - No device memory is allocated or freed by this call.
 *   - Each call checks the device (compute capability 10.3, else ATTN_ERR_ARCH)
 *     and then looks up the array's device address in the current context,
 *     with that device current.  The first lookup in a context loads the
 *     library's device code there; make that first call before any stream
 *     capture.
 *   - Every call shares the one array.  Calls whose work overlaps on the GPU
 *     (different streams, or different host threads on the same device) race on
 *     it; serialise them.  Each call clears what must start at zero itself.
 */
attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk,
                               void* dv, int B, int H, int N, int d, int causal,
                               float softmax_scale, attn_dtype_t dtype, cudaStream_t stream);

/*
 * attn_decode_workspace_size -- bytes of device scratch attn_decode_paged needs
 * for the partial results of its key-range splits (float32 O and log-sum-exp
 * per split and query row).  Returns 0 for invalid sizes.
 */
size_t attn_decode_workspace_size(int B, int H, int H_kv, int n_q, int d, int max_seqlen);

/*
 * attn_decode_paged -- decode step: n_q new query tokens per sequence against a
 * paged key/value cache, with grouped-query heads.
 *   q           : [B, H, n_q, d] in `dtype`; token t of sequence b is at position
 *                 seq_lens[b] - n_q + t (its keys and values are already in the
 *                 cache).
 *   k_cache,
 *   v_cache     : [num_pages, page_size, H_kv, d] in `dtype`.
 *   block_table : DEVICE int32 [B, max_pages]: logical page p of sequence b is
 *                 physical page block_table[b][p].
 *   seq_lens    : DEVICE int32 [B]: tokens of each sequence in the cache
 *                 (0 <= seq_lens[b] <= max_pages * page_size).
 *   o           : [B, H, n_q, d] in `dtype`;  lse : [B, H, n_q] float32 (natural
 *                 log of the scaled, masked scores; -inf and O = 0 for a row
 *                 that sees no key).
 *   workspace   : at least attn_decode_workspace_size(B, H, H_kv, n_q, d,
 *                 max_seqlen) bytes, 256-byte aligned.
 *   max_seqlen  : >= every seq_lens[b] (sizes the key-range split).
 *   causal      : 1 = query t sees keys 0 .. seq_lens[b] - n_q + t (bottom-right
 *                 aligned); 0 = every key of the sequence.
 * Limits: d = 64 or 128; (H / H_kv) * n_q <= 128; page_size a power of two in
 * [8, 65536].  Out-of-range seq_lens or block_table entries are skipped on the
 * device and reported by attn_get_device_status() as ATTN_ERR_INVALID_ARG.
 * Source: exact attention ("FlashAttention-3: Hopper Asynchrony and FP8
 * Attention", "Symbol Map"; its section "Where It Breaks" leaves a
 * decode-focused kernel as open work) over the paged cache of "FlashAttention 3
 * Hardware Acceleration: Hopper GPU Strategies for Long-Context Enterprise
 * Inference Optimization", sections "Memory Fragmentation" (the cache in
 * fixed-size blocks) and "Production Inference Engines" (separate decode
 * functions).
 */
attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int* block_table, const int* seq_lens, void* o, float* lse,
                                void* workspace, size_t workspace_bytes, int B, int H, int H_kv,
                                int n_q, int d, int num_pages, int page_size, int max_pages,
                                int max_seqlen, int causal, float softmax_scale,
                                attn_dtype_t dtype, cudaStream_t stream);

/*
 * attn_decode_paged_fp8 -- attn_decode_paged over a cache of e4m3 codes with
 * block scaling: one descale per (physical page, key/value head).
 *   q              : [B, H, n_q, d] in `dtype` (bf16 or fp16); the kernel
 *                    quantises each query row to e4m3 with its own descale
 *                    (row amax / 448), after multiplying it by M when
 *                    hadamard_signs is given.
 *   k_cache,
 *   v_cache        : uint8 e4m3 (OCP E4M3, "fn") codes [num_pages, page_size,
 *                    H_kv, d].  Value = code x descale of the block.
 *   k_descale,
 *   v_descale      : DEVICE float32 [num_pages, H_kv], positive and finite.
 *   hadamard_signs : DEVICE float32 [d] of +1 / -1, or NULL.  Give it when the
 *                    keys were stored transformed, K M with M = diag(signs)
 *                    H_d / sqrt(d) (H_d the Sylvester Hadamard matrix): the query
 *                    is transformed by the same M, and (q M)(K M)^T = q K^T.
 *                    Values are never transformed.
 *   Other arguments, outputs, workspace (attn_decode_workspace_size), masking
 *   and device-side error reporting as attn_decode_paged.  O is in `dtype`.
 * Limits: d = 128; (H / H_kv) * n_q <= 128; page_size a power of two in
 * [16, 65536].  Both products run on e4m3 operands (P rounded to e4m3, as in
 * attn_fwd_fp8); accuracy is that of the FP8 forward.
 * Source: the FP8 path of "FlashAttention-3: Hopper Asynchrony and FP8
 * Attention" ("FP8 accuracy controls": block quantisation, incoherent
 * processing) applied to the decode step that its section "Where It Breaks"
 * leaves open (persistent FP8 inference), over the paged cache of "FlashAttention
 * 3 Hardware Acceleration: ...", section "Memory Fragmentation".
 */
attn_status_t attn_decode_paged_fp8(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                    const float* k_descale, const float* v_descale,
                                    const float* hadamard_signs, const int* block_table,
                                    const int* seq_lens, void* o, float* lse, void* workspace,
                                    size_t workspace_bytes, int B, int H, int H_kv, int n_q, int d,
                                    int num_pages, int page_size, int max_pages, int max_seqlen,
                                    int causal, float softmax_scale, attn_dtype_t dtype,
                                    cudaStream_t stream);

/*
 * attn_fp8_quantize -- FP8 e4m3 pre-pass with block scaling and incoherent
 * processing ("FlashAttention-3: Hopper Asynchrony and FP8 Attention", section
 * "FP8 accuracy controls").
 *   q, k, v        : [B, H, N, d] float32 (read only); d must be 128.
 *   hadamard_signs : d float32 values, each +1 or -1, or NULL.  When given, every
 *                    row x of Q and of K becomes x M with M = diag(signs) H_d / sqrt(d)
 *                    (H_d the Sylvester Hadamard matrix) before quantisation;
 *                    V is never transformed.  (QM)(KM)^T = QK^T, so the FP8
 *                    forward needs no knowledge of the transform.
 *   q8, k8, v8     : [B, H, N, d] e4m3 bytes (written).
 *   q_descale, k_descale, v_descale : [B, H, ceil(N/128)] float32 (written):
 *                    per 128-row block, descale = amax / 448 (1 if amax = 0) and
 *                    code = e4m3_rn_satfinite(x / descale).
 *   per_tensor     : 0 = one scale per block; 1 = one scale per whole tensor (all
 *                    b, h, rows; every descale entry holds it) -- the per-tensor
 *                    comparator; hadamard_signs must then be NULL.
 */
attn_status_t attn_fp8_quantize(const float* q, const float* k, const float* v,
                                const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                uint8_t* v8, float* q_descale, float* k_descale,
                                float* v_descale, int B, int H, int N, int d, int per_tensor,
                                cudaStream_t stream);

/*
 * attn_fp8_quantize_gqa -- attn_fp8_quantize for grouped-query attention: Q has
 * H heads, K and V have H_kv (H % H_kv == 0; "FlashAttention 3 Hardware
 * Acceleration: ...", section "GPU Compatibility and Enablement Matrix",
 * grouped-query attention by template specialisation).
 *   q, q8          : [B, H, N, d];  q_descale : [B, H, ceil(N/128)].
 *   k, v, k8, v8   : [B, H_kv, N, d];  k_descale, v_descale : [B, H_kv, ceil(N/128)].
 * Blocks, transform, per-tensor mode and errors as attn_fp8_quantize (which is
 * this call with H_kv = H).
 */
attn_status_t attn_fp8_quantize_gqa(const float* q, const float* k, const float* v,
                                    const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                    uint8_t* v8, float* q_descale, float* k_descale,
                                    float* v_descale, int B, int H, int H_kv, int N, int d,
                                    int per_tensor, cudaStream_t stream);

/*
 * attn_fp8_quantize_bf16 -- attn_fp8_quantize_gqa on bfloat16 inputs: q
 * [B, H, N, d], k and v [B, H_kv, N, d] bfloat16 (each value widened exactly to
 * float32, then transformed and quantised as there); the same outputs, modes
 * and errors.  This is the pre-pass for activations held in bfloat16, e.g. the
 * very tensors the BF16 forward reads.
 */
attn_status_t attn_fp8_quantize_bf16(const void* q, const void* k, const void* v,
                                     const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                     uint8_t* v8, float* q_descale, float* k_descale,
                                     float* v_descale, int B, int H, int H_kv, int N, int d,
                                     int per_tensor, cudaStream_t stream);

/*
 * attn_fp8_quantize_varlen -- the block pre-pass (attn_fp8_quantize_gqa) for a
 * packed batch of B sequences stored back to back (the layout of
 * attn_fwd_varlen).
 *   q : [total, H, d] float32;  k, v : [total, H_kv, d] float32;  d = 128.
 *   q8, k8, v8 : the same shapes, e4m3 bytes (written).
 *   q_descale : [B, H, ceil(max_seqlen/128)];  k_descale, v_descale :
 *               [B, H_kv, ceil(max_seqlen/128)] float32 (written): a block is
 *               128 consecutive tokens of one sequence and head, starting at the
 *               sequence's first token; entries past a sequence's end hold 1.
 *   cu_seqlens : DEVICE int32 [B + 1] (as attn_fwd_varlen).
 * Block mode only (no per-tensor mode, no rotary embedding).  Offsets that are
 * not increasing, run past `total` or hold a sequence longer than max_seqlen
 * are reported by attn_get_device_status() as ATTN_ERR_INVALID_ARG.
 */
attn_status_t attn_fp8_quantize_varlen(const float* q, const float* k, const float* v,
                                       const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                       uint8_t* v8, float* q_descale, float* k_descale,
                                       float* v_descale, const int* cu_seqlens, int B,
                                       int max_seqlen, int total, int H, int H_kv, int d,
                                       cudaStream_t stream);

/*
 * attn_fp8_quantize_rope -- attn_fp8_quantize (block mode) with the rotary
 * position embedding of Q and K fused in front of the Hadamard transform
 * ("FlashAttention-3: Hopper Asynchrony and FP8 Attention", section "FP8
 * accuracy controls": the transform can be fused with rotary embedding; the
 * pages do not define the embedding, so the tables come from the caller).
 *   rope_cos, rope_sin : device float32 [N, d/2]: for the row at position n
 *                        (0 <= n < N, the same for every b, h) each pair
 *                        (x_i, x_{i+d/2}), i < d/2, becomes
 *                        (x_i c - x_{i+d/2} s,  x_{i+d/2} c + x_i s),
 *                        c = rope_cos[n][i], s = rope_sin[n][i].
 *   V is not rotated.  hadamard_signs may be NULL (rotation only).  Other
 *   arguments, outputs and errors as attn_fp8_quantize; d = 128.
 */
attn_status_t attn_fp8_quantize_rope(const float* q, const float* k, const float* v,
                                     const float* rope_cos, const float* rope_sin,
                                     const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                     uint8_t* v8, float* q_descale, float* k_descale,
                                     float* v_descale, int B, int H, int N, int d,
                                     cudaStream_t stream);

/*
 * attn_fp8_quantize_ex -- the FP8 pre-pass with every option in one call:
 * float32 or bfloat16 inputs, rotary embedding of Q and K, the Hadamard
 * transform, grouped-query heads, and fixed-length or packed batches.
 *   q, k, v        : input_bf16 = 0: float32; 1: bfloat16.
 *                    cu_seqlens == NULL: q [B, H, N, d], k and v [B, H_kv, N, d];
 *                    else a packed batch (the layout of attn_fwd_varlen): q
 *                    [total, H, d], k and v [total, H_kv, d], N = the longest
 *                    sequence (max_seqlen), cu_seqlens DEVICE int32 [B + 1].
 *   rope_cos,
 *   rope_sin       : DEVICE float32 [N, d/2] or both NULL (no rotation).  A row
 *                    at position n of its sequence (n = 0 at the sequence's first
 *                    token) has each pair (x_i, x_{i+d/2}), i < d/2, rotated to
 *                    (x_i c - x_{i+d/2} s, x_{i+d/2} c + x_i s), c, s =
 *                    rope_cos[n][i], rope_sin[n][i]; Q and K only, before the
 *                    Hadamard transform.  16-byte aligned.
 *   hadamard_signs : as attn_fp8_quantize, or NULL.
 *   q8, k8, v8     : e4m3 codes in the inputs' layout (written).
 *   *_descale      : fixed length: [B, H or H_kv, ceil(N/128)]; packed: as
 *                    attn_fp8_quantize_varlen (entries past a sequence's end hold 1).
 *   per_tensor     : 1 = the per-tensor comparator (fixed length, no rotation, no
 *                    Hadamard); else 0.
 * d = 128.  The codes are those of attn_fp8_quantize_gqa / _bf16 / _varlen /
 * _rope with the same options; the packed offsets are checked on the device
 * (reported by attn_get_device_status as ATTN_ERR_INVALID_ARG).
 * Source: "FlashAttention-3: Hopper Asynchrony and FP8 Attention", section "FP8
 * accuracy controls" (block scales; the transform "can be fused with rotary
 * embedding"); "FlashAttention 3 Hardware Acceleration: ...", sections "Torch
 * Compile" (rotary embedding fused with the transform) and "GPU Compatibility
 * and Enablement Matrix" (grouped-query heads, variable-length batches).
 */
attn_status_t attn_fp8_quantize_ex(const void* q, const void* k, const void* v, int input_bf16,
                                   const float* rope_cos, const float* rope_sin,
                                   const float* hadamard_signs, uint8_t* q8, uint8_t* k8,
                                   uint8_t* v8, float* q_descale, float* k_descale,
                                   float* v_descale, const int* cu_seqlens, int B, int N,
                                   int total, int H, int H_kv, int d, int per_tensor,
                                   cudaStream_t stream);

/*
 * attn_fwd_fp8 -- FP8 e4m3 forward on the output of attn_fp8_quantize.
 *   q8, k8, v8 : [B, H, N, d] e4m3; d must be 128.
 *   *_descale  : [B, H, ceil(N/128)] float32 block descales.
 *   o          : [B, H, N, d] bfloat16 (written); lse: [B, H, N] float32 (written).
 * Scores use the block descales of their query and key blocks; the
 * probabilities are rounded to e4m3 for the P V product.  causal, softmax_scale,
 * the asynchronous launch on `stream` and the errors are those of attn_fwd;
 * descales must be positive and finite (the pre-pass writes them so).
 * Source: "FlashAttention-3: Hopper Asynchrony and FP8 Attention", sections
 * "Symbol Map" (the same O and L as attn_fwd), "FP8 accuracy controls" (one
 * scale per Q, K or V block; Q and K may carry the transform M, which the
 * scores do not see since (QM)(KM)^T = QK^T) and "FP8 layout conformance" (the
 * P V product on FP8 operands); "FlashAttention 3 Hardware Acceleration: ...",
 * section "FP8 Assumptions": quantisation happens before the call and every
 * FP8 tensor travels with its scales.
 */
attn_status_t attn_fwd_fp8(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                           const float* q_descale, const float* k_descale,
                           const float* v_descale, void* o, float* lse, int B, int H, int N,
                           int d, int causal, float softmax_scale, cudaStream_t stream);

/*
 * attn_fwd_fp8_schedule -- attn_fwd_fp8 with a schedule variant, for
 * measurement.  `schedule` is 0 (exactly attn_fwd_fp8, which evaluates one
 * sixteenth of the exponentials on the FMA pipe for non-causal batches and none
 * for causal ones), ATTN_SCHED_EXP2_NONE (every exponential on the
 * MUFU unit), ATTN_SCHED_EXP2_POLY or ATTN_SCHED_EXP2_EIGHTHS(k), k = 1..4: k of
 * every 8 of each softmax thread's exponentials (a quarter for
 * ATTN_SCHED_EXP2_POLY alone) are evaluated on the FMA pipe by range reduction
 * and a cubic (relative error <= 1.1e-4, below the e4m3 rounding of P) instead
 * of by the MUFU unit.  Other values return ATTN_ERR_INVALID_ARG.  Arguments,
 * layout and errors as attn_fwd_fp8.
 * Source: "FlashAttention-3: Hopper Asynchrony and FP8 Attention", section
 * "Why This Exists" (FP8 doubles the matrix-multiply rate but not the rate of
 * exponentials).
 */
attn_status_t attn_fwd_fp8_schedule(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                                    const float* q_descale, const float* k_descale,
                                    const float* v_descale, void* o, float* lse, int B, int H,
                                    int N, int d, int causal, float softmax_scale, int schedule,
                                    cudaStream_t stream);

/*
 * attn_selftest_exp2 -- diagnostic: evaluates, for n float32 inputs x, the
 * FMA-pipe exponential of ATTN_SCHED_EXP2_POLY (y_poly) and the MUFU
 * approximation the kernels otherwise use (y_mufu), both 2^x.  x, y_poly and
 * y_mufu are device arrays of n floats; the call is asynchronous on `stream`.
 * Defined for x <= 126; x <= -127 (and -inf) give exactly 0 in y_poly.  The
 * pages give no such routine; it exists so the approximation can be checked
 * against the exact function on the GPU.
 */
attn_status_t attn_selftest_exp2(const float* x, float* y_poly, float* y_mufu, long long n,
                                 cudaStream_t stream);

/*
 * attn_fwd_fp8_varlen -- FP8 forward on a packed batch (the output of
 * attn_fp8_quantize_varlen), grouped-query heads allowed.
 *   q8 : [total, H, d];  k8, v8 : [total, H_kv, d] e4m3;  descales as
 *   attn_fp8_quantize_varlen writes them;  o : [total, H, d] bfloat16;
 *   lse : [H, total] float32;  other arguments and errors as attn_fwd_varlen.
 * Source: the FP8 forward of "FlashAttention-3: Hopper Asynchrony and FP8
 * Attention" over the variable-length batches that "FlashAttention 3 Hardware
 * Acceleration: ...", section "GPU Compatibility and Enablement Matrix", lists
 * as forthcoming (as attn_fwd_varlen).
 */
attn_status_t attn_fwd_fp8_varlen(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                                  const float* q_descale, const float* k_descale,
                                  const float* v_descale, void* o, float* lse,
                                  const int* cu_seqlens, int B, int max_seqlen, int total, int H,
                                  int H_kv, int d, int causal, float softmax_scale,
                                  cudaStream_t stream);

/*
 * attn_fwd_fp8_gqa -- attn_fwd_fp8 with grouped-query heads: query head h of
 * batch b reads key/value head h / (H / H_kv) and its block descales.
 *   q8 : [B, H, N, d] with q_descale [B, H, ceil(N/128)];
 *   k8, v8 : [B, H_kv, N, d] with k_descale, v_descale [B, H_kv, ceil(N/128)]
 *   (the output of attn_fp8_quantize_gqa);  o, lse as attn_fwd_fp8.
 * attn_fwd_fp8 is this call with H_kv = H.  Source: the FP8 forward of
 * "FlashAttention-3: Hopper Asynchrony and FP8 Attention" with the head sharing
 * of "FlashAttention 3 Hardware Acceleration: ...", section "GPU Compatibility
 * and Enablement Matrix".
 */
attn_status_t attn_fwd_fp8_gqa(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8,
                               const float* q_descale, const float* k_descale,
                               const float* v_descale, void* o, float* lse, int B, int H,
                               int H_kv, int N, int d, int causal, float softmax_scale,
                               cudaStream_t stream);

/*
 * attn_get_device_status -- synchronises `stream`, then reads and clears the
 * current device's status word.  ATTN_OK, ATTN_ERR_TIMEOUT (a kernel gave up
 * on an internal wait; attn_last_error() names the role), ATTN_ERR_INVALID_ARG
 * (a packed or paged call met offsets, lengths or pages out of range and
 * skipped them), ATTN_ERR_ARCH, or ATTN_ERR_CUDA.
 * Source: the pages list failure modes ("FlashAttention-3: Hopper Asynchrony
 * and FP8 Attention", section "Where It Breaks") and ask that problems be
 * reported as explicit errors rather than silently degraded ("FlashAttention 3
 * Hardware Acceleration: ...", section "Unsupported GPU Architecture"); this
 * device-side report is the library's own way of doing so for errors found
 * while kernels run.
 */
attn_status_t attn_get_device_status(cudaStream_t stream);

/*
 * attn_selftest_wait_timeout -- diagnostic for the failure path every kernel
 * shares.  Launches one thread that waits, through the kernels' bounded
 * barrier wait, on a barrier nothing ever arrives on; after limit_us
 * microseconds (1 .. 1000000) the wait gives up and records a timeout in the
 * status word, and the kernel returns normally.  A following
 * attn_get_device_status() then returns ATTN_ERR_TIMEOUT (role "self-test")
 * and clears the word; the CUDA context stays usable.  Section "Where It
 * Breaks" of "FlashAttention-3: Hopper Asynchrony and FP8 Attention" lists
 * failure modes but no recovery mechanism; this is the library's own.
 */
attn_status_t attn_selftest_wait_timeout(unsigned limit_us, cudaStream_t stream);

/* Static description of a status code (a string literal; never NULL).  The
 * codes are the library's own explicit errors, in the sense of "FlashAttention
 * 3 Hardware Acceleration: ...", section "Unsupported GPU Architecture"
 * (explicit errors rather than silent degradation). */
const char* attn_status_string(attn_status_t s);

/* Detail of the last error returned on this host thread ("" if none). */
const char* attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
