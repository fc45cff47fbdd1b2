// FP8 (e4m3) path on sm_103a: the quantisation pre-pass and the FP8 forward.
//
// Method: "FlashAttention-3: Hopper Asynchrony and FP8 Attention", section "FP8
// accuracy controls": block quantisation keeps one scale per Q, K or V block,
// and incoherent processing multiplies Q and K by the same orthogonal matrix
// M = diag(s) H_d / sqrt(d) before quantisation, so (QM)(KM)^T = QK^T and the
// forward kernel needs no knowledge of M.
//
// Pre-pass (d = 128): one CTA per (128-row block, head, tensor).  A warp holds
// a row as 32 lanes x 4 values; the Walsh-Hadamard butterfly runs two stages
// inside each lane and five across lanes with xor shuffles.  The block amax
// gives descale = amax / 448 and codes = e4m3_rn_satfinite(x / descale).
// Per-tensor mode (the comparator) runs amax, reduce and quantise kernels.
//
// Forward (d = 128): the BF16 forward's structure (two softmax warps per row)
// with tcgen05.mma kind::f8f6f4 (32-element K steps).  Scores use c_j = scale * log2(e) * dq_i *
// dk_j, folded into the single FMA before exp2.  The per-block V descales are
// folded into the exponent as log2(dv_j / dv_max) (dv_max = largest V descale
// of the head), so P dv_j / dv_max is what is rounded to e4m3 for the P V
// product; the row sum l accumulates the unscaled P, and the epilogue
// multiplies O by dv_max / l.  The page's FP8 layout steps ("FP8 layout
// conformance": V transpose, accumulator byte permutation) are not needed:
// V is read as an MN-major operand and P goes through tensor memory.
#include <cmath>

#include "common.h"
#include "sm103_prims.cuh"

namespace attn {
namespace {

constexpr int kSmemLimit = 232448;
constexpr float kE4m3Max = 448.f;

// ============================================================== pre-pass ====
// Walsh-Hadamard butterfly (unnormalised) of a 128-value row held by a warp as
// 32 lanes x 4 values, packed as (columns 4 lane, 4 lane + 1) and (4 lane + 2,
// 4 lane + 3): the stages of span 1 and 2 inside the lane, then those of span
// 4 .. 64 across lanes (lane distance 1 .. 16), where the lane with bit m set
// takes partner - own and the other own + partner, both as one fused
// multiply-add by +-1 (exactly the add or the subtract).
__device__ __forceinline__ void wht128_row(uint64_t& p01, uint64_t& p23, int lane) {
  const float a = lo2(p01) + hi2(p01), b = lo2(p01) - hi2(p01);
  const float c = lo2(p23) + hi2(p23), e = lo2(p23) - hi2(p23);
  p01 = pack2(a + c, b + e);
  p23 = pack2(a - c, b - e);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float ox = __shfl_xor_sync(0xffffffffu, lo2(p01), m);
    const float oy = __shfl_xor_sync(0xffffffffu, hi2(p01), m);
    const float oz = __shfl_xor_sync(0xffffffffu, lo2(p23), m);
    const float ow = __shfl_xor_sync(0xffffffffu, hi2(p23), m);
    const float sg = (lane & m) ? -1.f : 1.f;
    const uint64_t sg2 = pack2(sg, sg);
    p01 = ffma2(sg2, p01, pack2(ox, oy));
    p23 = ffma2(sg2, p23, pack2(oz, ow));
  }
}

// code = e4m3(x / descale) for four values (two packed pairs), each quotient
// rounded as an IEEE division would: q0 = x y with y = 1 / descale, then
// q0 + (x - descale q0) y (the steps of div_by_recip on packed pairs).
__device__ __forceinline__ uint32_t quantise4(uint64_t x01, uint64_t x23, uint64_t y2, uint64_t nb2) {
  const uint64_t q01 = fmul2(x01, y2), q23 = fmul2(x23, y2);
  const uint64_t c01 = ffma2(ffma2(nb2, q01, x01), y2, q01);
  const uint64_t c23 = ffma2(ffma2(nb2, q23, x23), y2, q23);
  return cvt_pack_e4m3x4(lo2(c01), hi2(c01), lo2(c23), hi2(c23));
}

// Mode: 0 = fused block mode (amax + quantise), 1 = block amax only (into
// descale), 2 = quantise with the descale already in place.  PACKED (mode 0):
// sequences packed back to back, [total, heads, d]; N is the longest sequence
// and a block is 128 rows of one sequence and head (descale [B, heads,
// ceil(N / 128)], 1 for blocks past the sequence's end).
// BF16IN: the inputs are bfloat16 (widened exactly to float32 on load).
// ROPE (mode 0): Q and K rows are rotated first, from caller tables rope_cos,
// rope_sin [N, d/2] indexed by the row's position in its sequence: the pair
// (x_i, x_{i+d/2}) becomes (x_i c - x_{i+d/2} s, x_{i+d/2} c + x_i s).  A lane
// holds columns 4 lane .. 4 lane + 3, so lanes l and l ^ 16 hold partners.
template <int MODE, bool PACKED = false, bool BF16IN = false, bool ROPE = false>
__global__ void __launch_bounds__(256)
    fp8_quant_kernel(const void* __restrict__ src0, const void* __restrict__ src1,
                     const void* __restrict__ src2, uint8_t* __restrict__ dst0,
                     uint8_t* __restrict__ dst1, uint8_t* __restrict__ dst2,
                     float* __restrict__ desc0, float* __restrict__ desc1,
                     float* __restrict__ desc2, const float* __restrict__ signs, int N,
                     int nblk, int kv_planes, const int* __restrict__ cu_seqlens = nullptr,
                     int total = 0, int heads_q = 0, int heads_kv = 0, int* status = nullptr,
                     const float* __restrict__ rope_cos = nullptr,
                     const float* __restrict__ rope_sin = nullptr) {
  constexpr int D = 128;
  const int which = blockIdx.z;
  if (which > 0 && static_cast<int>(blockIdx.y) >= kv_planes) return;   // K, V: B * H_kv planes
  const void* src = which == 0 ? src0 : (which == 1 ? src1 : src2);
  uint8_t* dst = which == 0 ? dst0 : (which == 1 ? dst1 : dst2);
  float* desc = which == 0 ? desc0 : (which == 1 ? desc1 : desc2);
  const bool hadamard = signs != nullptr && which < 2;
  const bool rotate = ROPE && which < 2;
  const int blk = blockIdx.x;
  const int bh = blockIdx.y;
  // row r of this (b, h) lies at element row0 + r * rstride; rows r < nrows exist
  size_t row0 = static_cast<size_t>(bh) * N * D;
  size_t rstride = D;
  int nrows = N;
  if constexpr (PACKED) {
    const int heads = which == 0 ? heads_q : heads_kv;
    const int b = bh / heads;
    const int s0 = cu_seqlens[b];
    const int end = cu_seqlens[b + 1];
    if (s0 < 0 || end < s0 || end > total || end - s0 > N) {
      if (threadIdx.x == 0) atomicCAS(status, 0, kDevBadSeqlens);
      return;
    }
    row0 = (static_cast<size_t>(s0) * heads + bh % heads) * D;
    rstride = static_cast<size_t>(heads) * D;
    nrows = end - s0;
    if (blk * 128 >= nrows) {
      if (threadIdx.x == 0) desc[static_cast<size_t>(bh) * nblk + blk] = 1.f;
      return;
    }
  }
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  __shared__ float warp_max[8];

  // 16 rows per warp, 4 columns per lane, as two packed float32 pairs
  // (columns 4 lane, 4 lane + 1 and 4 lane + 2, 4 lane + 3)
  uint64_t x01[16], x23[16];
  float amax = 0.f;
  float4 s4 = make_float4(1.f, 1.f, 1.f, 1.f);
  if (hadamard) s4 = reinterpret_cast<const float4*>(signs)[lane];
  const float inv_sqrt_d = 0.08838834764831845f;   // 1 / sqrt(128)
  const uint64_t isd2 = pack2(inv_sqrt_d, inv_sqrt_d);
  // bfloat16 rows are small enough (8 bytes per lane) to have all 16 of the
  // warp's loads in flight before the first transform
  uint2 raw[BF16IN ? 16 : 1];
  if constexpr (BF16IN) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int row = blk * 128 + warp * 16 + r;
      raw[r] = row < nrows ? __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(src) + row0 +
                                                                 row * rstride) + lane)
                           : make_uint2(0u, 0u);
    }
  }
  // The sign diagonal of M on bfloat16 inputs: multiplying by -1 flips the
  // sign bit, done while widening.
  const uint32_t sgx = (!ROPE && BF16IN && s4.x < 0.f) ? 0x80000000u : 0u;
  const uint32_t sgy = (!ROPE && BF16IN && s4.y < 0.f) ? 0x80000000u : 0u;
  const uint32_t sgz = (!ROPE && BF16IN && s4.z < 0.f) ? 0x80000000u : 0u;
  const uint32_t sgw = (!ROPE && BF16IN && s4.w < 0.f) ? 0x80000000u : 0u;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int row = blk * 128 + warp * 16 + r;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row < nrows) {
      if constexpr (BF16IN) {
        // four bfloat16 values; each is the upper half of its float32
        const uint2 w = raw[r];
        v = make_float4(__uint_as_float((w.x << 16) ^ sgx), __uint_as_float((w.x & 0xffff0000u) ^ sgy),
                        __uint_as_float((w.y << 16) ^ sgz), __uint_as_float((w.y & 0xffff0000u) ^ sgw));
      } else {
        v = reinterpret_cast<const float4*>(static_cast<const float*>(src) + row0 + row * rstride)[lane];
      }
    }
    if (rotate) {
      // position = row index in the sequence (rows past the end are zero and
      // stay zero; their table row is clamped so every load is in bounds and
      // can be issued early)
      const float ox = __shfl_xor_sync(0xffffffffu, v.x, 16);
      const float oy = __shfl_xor_sync(0xffffffffu, v.y, 16);
      const float oz = __shfl_xor_sync(0xffffffffu, v.z, 16);
      const float ow = __shfl_xor_sync(0xffffffffu, v.w, 16);
      const size_t tix = static_cast<size_t>(min(row, nrows - 1)) * (D / 2) + 4 * (lane & 15);
      const float4 c4 = __ldg(reinterpret_cast<const float4*>(rope_cos + tix));
      const float4 sn = __ldg(reinterpret_cast<const float4*>(rope_sin + tix));
      const float sg = (lane < 16) ? -1.f : 1.f;   // first half: x c - partner s
      v = make_float4(fmaf(sg * ox, sn.x, v.x * c4.x), fmaf(sg * oy, sn.y, v.y * c4.y),
                      fmaf(sg * oz, sn.z, v.z * c4.z), fmaf(sg * ow, sn.w, v.w * c4.w));
    }
    uint64_t p01 = pack2(v.x, v.y), p23 = pack2(v.z, v.w);
    if (hadamard) {
      if (ROPE || !BF16IN) {
        p01 = fmul2(p01, pack2(s4.x, s4.y));
        p23 = fmul2(p23, pack2(s4.z, s4.w));
      }
      wht128_row(p01, p23, lane);
      p01 = fmul2(p01, isd2);
      p23 = fmul2(p23, isd2);
    }
    x01[r] = p01;
    x23[r] = p23;
    amax = fmax3(amax, fmax3(fabsf(lo2(p01)), fabsf(hi2(p01)), fabsf(lo2(p23))), fabsf(hi2(p23)));
  }

  float descale;
  if (MODE == 2) {
    descale = desc[static_cast<size_t>(bh) * nblk + blk];
  } else {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    float bmax = warp_max[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) bmax = fmaxf(bmax, warp_max[w]);
    if (MODE == 1) {
      if (threadIdx.x == 0) desc[static_cast<size_t>(bh) * nblk + blk] = bmax;
      return;
    }
    descale = bmax > 0.f ? __fdiv_rn(bmax, kE4m3Max) : 1.f;
    if (threadIdx.x == 0) desc[static_cast<size_t>(bh) * nblk + blk] = descale;
  }
  const float rdesc = __fdiv_rn(1.f, descale);
  const uint64_t y2 = pack2(rdesc, rdesc);
  const uint64_t nb2 = pack2(-descale, -descale);
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int row = blk * 128 + warp * 16 + r;
    if (row < nrows)
      reinterpret_cast<uint32_t*>(dst + row0 + row * rstride)[lane] = quantise4(x01[r], x23[r], y2, nb2);
  }
}

// Rotary variant (block mode): rotary embedding of Q and K rows first, from
// caller tables rope_cos, rope_sin [N, d/2]: the pair (x_i, x_{i+d/2}) of the row
// at position n becomes (x_i c - x_{i+d/2} s, x_{i+d/2} c + x_i s), c, s =
// table[n][i] ("FlashAttention-3: Hopper Asynchrony and FP8 Attention", section
// "FP8 accuracy controls": the Hadamard transform can be fused with the rotary
// embedding).  Holding a rotated block in registers costs too many registers
// for good occupancy, so this kernel stages the block's rows (contiguous, 64 KB
// of float32) in shared memory with one bulk copy per warp's 16 rows; the warps
// transform rows in place, the block amax gives the descale, and the codes are
// written from shared memory.  (For the plain pre-pass the register-staged
// kernel above measured faster, 4.6 vs 3.8 TB/s.)
constexpr int QROWS = 128;
constexpr int QSMEM = QROWS * 128 * 4;   // one block of float32 rows at d = 128

template <int MODE, bool ROPE>
__global__ void __launch_bounds__(256)
    fp8_quant_staged_kernel(const float* __restrict__ src0, const float* __restrict__ src1,
                     const float* __restrict__ src2, uint8_t* __restrict__ dst0,
                     uint8_t* __restrict__ dst1, uint8_t* __restrict__ dst2,
                     float* __restrict__ desc0, float* __restrict__ desc1,
                     float* __restrict__ desc2, const float* __restrict__ signs, int N,
                     int nblk, int kv_planes, int* status, const float* __restrict__ rope_cos = nullptr,
                     const float* __restrict__ rope_sin = nullptr) {
  constexpr int D = 128;
  if (blockIdx.z > 0 && static_cast<int>(blockIdx.y) >= kv_planes) return;   // K, V: B * H_kv planes
  extern __shared__ __align__(128) float sblk[];   // [QROWS][D]
  __shared__ __align__(8) uint64_t full_bar[8];    // one per warp's 16 rows
  __shared__ int abort_sh;
  __shared__ float warp_max[8];
  const int which = blockIdx.z;
  const float* src = which == 0 ? src0 : (which == 1 ? src1 : src2);
  uint8_t* dst = which == 0 ? dst0 : (which == 1 ? dst1 : dst2);
  float* desc = which == 0 ? desc0 : (which == 1 ? desc1 : desc2);
  const bool hadamard = signs != nullptr && which < 2;
  const bool rotate = ROPE && which < 2;
  const int blk = blockIdx.x;
  const int bh = blockIdx.y;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rows = min(QROWS, N - blk * QROWS);          // valid rows of this block (>= 1)

  if (threadIdx.x == 0) {
    for (int w = 0; w < 8; ++w) mbar_init(&full_bar[w], 1);
    abort_sh = 0;
    fence_mbar_init();
    // one bulk copy per warp's 16 rows, so a warp starts on its rows as soon
    // as they land
    const float* base = src + (static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * QROWS) * D;
    for (int w = 0; w < 8 && 16 * w < rows; ++w) {
      const uint32_t bytes = static_cast<uint32_t>(min(16, rows - 16 * w)) * D * 4;
      mbar_arrive_expect_tx(&full_bar[w], bytes);
      bulk_load(sblk + 16 * w * D, base + 16 * w * D, bytes, &full_bar[w]);
    }
  }
  __syncthreads();
  const Abort ab{&abort_sh, status};
  if (16 * warp < rows && !mbar_wait(&full_bar[warp], 0, ab, kDevTimeoutLoad)) {
    if (lane == 0) mbar_wait_drain(&full_bar[warp], 0);   // the copy may still land
    return;
  }

  float amax = 0.f;
  if (MODE != 2) {
    float4 s4 = make_float4(1.f, 1.f, 1.f, 1.f);
    if (hadamard) s4 = reinterpret_cast<const float4*>(signs)[lane];
    const float inv_sqrt_d = 0.08838834764831845f;   // 1 / sqrt(128)
#pragma unroll 4
    for (int r = 0; r < 16; ++r) {
      const int lr = warp * 16 + r;
      if (lr >= rows) break;                          // warp-uniform
      float4* row4 = reinterpret_cast<float4*>(sblk + lr * D);
      float4 v = row4[lane];
      if (rotate) {
        // lanes 0..15 hold columns 0..63, lanes 16..31 their partners 64..127
        const float4 o = row4[lane ^ 16];
        const size_t t = static_cast<size_t>(blk * QROWS + lr) * (D / 2) + 4 * (lane & 15);
        const float4 c = *reinterpret_cast<const float4*>(rope_cos + t);
        const float4 sn = *reinterpret_cast<const float4*>(rope_sin + t);
        const float sg = (lane < 16) ? -1.f : 1.f;   // first half: x c - partner s
        v = make_float4(fmaf(sg * o.x, sn.x, v.x * c.x), fmaf(sg * o.y, sn.y, v.y * c.y),
                        fmaf(sg * o.z, sn.z, v.z * c.z), fmaf(sg * o.w, sn.w, v.w * c.w));
      }
      if (hadamard) {
        uint64_t p01 = fmul2(pack2(v.x, v.y), pack2(s4.x, s4.y));
        uint64_t p23 = fmul2(pack2(v.z, v.w), pack2(s4.z, s4.w));
        wht128_row(p01, p23, lane);
        const uint64_t isd2 = pack2(inv_sqrt_d, inv_sqrt_d);
        p01 = fmul2(p01, isd2);
        p23 = fmul2(p23, isd2);
        v = make_float4(lo2(p01), hi2(p01), lo2(p23), hi2(p23));
      }
      if (rotate || hadamard) {
        __syncwarp();                                 // partners read before the write-back
        row4[lane] = v;
      }
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
  }

  float descale;
  if (MODE == 2) {
    descale = desc[static_cast<size_t>(bh) * nblk + blk];
  } else {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    float bmax = warp_max[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) bmax = fmaxf(bmax, warp_max[w]);
    if (MODE == 1) {
      if (threadIdx.x == 0) desc[static_cast<size_t>(bh) * nblk + blk] = bmax;
      return;
    }
    descale = bmax > 0.f ? __fdiv_rn(bmax, kE4m3Max) : 1.f;
    if (threadIdx.x == 0) desc[static_cast<size_t>(bh) * nblk + blk] = descale;
  }
  const float rdesc = __fdiv_rn(1.f, descale);
  const uint64_t y2 = pack2(rdesc, rdesc);
  const uint64_t nb2 = pack2(-descale, -descale);
#pragma unroll 4
  for (int r = 0; r < 16; ++r) {
    const int lr = warp * 16 + r;
    if (lr >= rows) break;
    const float4 v = reinterpret_cast<const float4*>(sblk + lr * D)[lane];
    reinterpret_cast<uint32_t*>(dst + (static_cast<size_t>(bh) * N + blk * QROWS + lr) * D)[lane] =
        quantise4(pack2(v.x, v.y), pack2(v.z, v.w), y2, nb2);
  }
}

// Per-tensor mode: one CTA per tensor reduces the block amaxes and writes the
// single descale into every entry.
__global__ void __launch_bounds__(256)
    fp8_tensor_scale_kernel(float* __restrict__ desc0, float* __restrict__ desc1,
                            float* __restrict__ desc2, long long q_count, long long kv_count) {
  float* desc = blockIdx.x == 0 ? desc0 : (blockIdx.x == 1 ? desc1 : desc2);
  const long long count = blockIdx.x == 0 ? q_count : kv_count;
  __shared__ float warp_max[8];
  float m = 0.f;
  for (long long i = threadIdx.x; i < count; i += blockDim.x) m = fmaxf(m, desc[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x / 32] = m;
  __syncthreads();
  float gmax = warp_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) gmax = fmaxf(gmax, warp_max[w]);
  const float descale = gmax > 0.f ? __fdiv_rn(gmax, kE4m3Max) : 1.f;
  __syncthreads();
  for (long long i = threadIdx.x; i < count; i += blockDim.x) desc[i] = descale;
}

// =============================================================== forward ====
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int D8 = 128;
constexpr int NQ8 = 2;
constexpr int TILE8 = BM * D8;            // 16 KB: one 128-byte row per token
constexpr int NSLOT8 = 8;
constexpr int SMEM8 = 1024 + NQ8 * TILE8 + NSLOT8 * TILE8;
// Two softmax warpgroups per query tile: each row of S is split between two
// warps (key columns [0, 64) and [64, 128)).
constexpr int THREADS8 = (8 * NQ8 + 2) * 32;
constexpr int LOAD_WARP8 = 8 * NQ8;
constexpr int MMA_WARP8 = 8 * NQ8 + 1;
__host__ __device__ constexpr uint32_t s_col8(int t) { return 128u * t; }
__host__ __device__ constexpr uint32_t o_col8(int t) { return 256u + 128u * t; }
// TMEM column of the packed e4m3 P for keys [32 kk, 32 kk + 32): each half of
// the row writes its P inside its own score columns
__host__ __device__ constexpr uint32_t p_col8(int kk) {
  return 64u * static_cast<uint32_t>(kk / 2) + 8u * static_cast<uint32_t>(kk % 2);
}
static_assert(SMEM8 <= kSmemLimit - 512, "shared memory");

struct Fp8KParams {
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  void* o;
  float* lse;
  int* status;
  int N;
  int H;
  int nblk;
  float scale_log2;
  int H_kv;   // key/value heads; query head h reads key/value head h / (H / H_kv)
  const int* cu_seqlens;   // packed batch: device [B + 1] token offsets, else nullptr
  int total;               // packed batch: tokens (cu_seqlens[B])
};

__device__ __forceinline__ float lg2_approx8(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// PACKED: a batch of sequences packed back to back -- codes [total, heads, d],
// descales [B, heads, ceil(max_seqlen / 128)] per sequence's 128-row blocks, O
// [total, H, d], LSE [H, total]; kp.N is the longest sequence; query and key
// tiles are read at the sequence's first token by 4-D tensor maps.
// POLY (0..8): of the sixteen 4-key groups of a softmax thread's step, POLY
// (spread out: group g when g POLY mod 16 < POLY) are evaluated by exp2_poly2 on
// the FMA pipe instead of the MUFU unit.  One sixteenth measured a little faster
// than none or one eighth on non-causal batches and is the library's choice
// there; three sixteenths or more measured slower (each emulated exponential
// takes several issue slots, and the softmax is bound by instruction issue, not
// by the MUFU rate).
template <bool CAUSAL, bool PACKED, int POLY = 0>
__global__ void __launch_bounds__(THREADS8, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const Fp8KParams kp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + NQ8 * TILE8;

  __shared__ __align__(8) uint64_t q_full[NQ8];
  __shared__ __align__(8) uint64_t kv_full[NSLOT8];
  __shared__ __align__(8) uint64_t kv_empty[NSLOT8];
  __shared__ __align__(8) uint64_t s_full[NQ8];
  __shared__ __align__(8) uint64_t p_full[NQ8];
  __shared__ __align__(8) uint64_t o_full[NQ8];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int load_items_sh;
  __shared__ float xch[2][NQ8][2][128];   // [step parity][tile][half][row]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // Causal: a 1-D grid ordered by work, heaviest query-tile groups (largest
  // g, which visit the most key tiles) of every head first, so the last wave
  // holds the short ones.  Non-causal: (group, head, batch) keeps a head's
  // CTAs together for K/V reuse in L2.
  const int npairs = (kp.N + BM * NQ8 - 1) / (BM * NQ8);
  const int g = CAUSAL ? npairs - 1 - static_cast<int>(blockIdx.x / (gridDim.x / npairs))
                       : static_cast<int>(blockIdx.x);
  const int bh = CAUSAL ? static_cast<int>(blockIdx.x % (gridDim.x / npairs))
                        : static_cast<int>(blockIdx.z * kp.H + blockIdx.y);
  // key/value plane (and descale row) of this query head
  const int kvp = (bh / kp.H) * kp.H_kv + (bh % kp.H) / (kp.H / kp.H_kv);
  int N = kp.N;      // this sequence's length
  int seq0 = 0;      // packed: its first token
  if constexpr (PACKED) {
    const int b = bh / kp.H;
    const int s0 = kp.cu_seqlens[b];
    const int end = kp.cu_seqlens[b + 1];
    if (s0 < 0 || end < s0 || end > kp.total || end - s0 > kp.N) {
      if (threadIdx.x == 0) atomicCAS(kp.status, 0, kDevBadSeqlens);
      return;
    }
    seq0 = s0;
    N = end - s0;
    if (g * NQ8 * BM >= N) return;   // the sequence ends before this CTA's query tiles
  }
  const int nKtot = (N + BN - 1) / BN;
  int nK[NQ8];
  int nKmax = 0;
#pragma unroll
  for (int t = 0; t < NQ8; ++t) {
    const int qt = g * NQ8 + t;
    nK[t] = (qt * BM < N) ? (CAUSAL ? min(nKtot, qt + 1) : nKtot) : 0;
    nKmax = max(nKmax, nK[t]);
  }
  const int total_items = 2 * nKmax;
  // The last query tile with work runs every key tile; when its S(j) completes,
  // all MMAs reading K_j and V_{j-1} have completed, so its softmax warpgroup
  // hands those ring slots back to the producer.
  const int t_rel = (nK[NQ8 - 1] == nKmax) ? NQ8 - 1 : 0;

  if (threadIdx.x == 0) {
    for (int t = 0; t < NQ8; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 256);
      mbar_init(&o_full[t], 1);
    }
    for (int s = 0; s < NSLOT8; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    load_items_sh = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP8) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const Abort ab{&abort_sh, kp.status};

  if (warp == LOAD_WARP8) {
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
#pragma unroll
      for (int t = 0; t < NQ8; ++t) {
        if (nK[t] == 0) continue;
        mbar_arrive_expect_tx(&q_full[t], TILE8);
        if constexpr (PACKED)
          tma_load_4d(sQ + t * TILE8, &tmQ, &q_full[t], 0, seq0 + (g * NQ8 + t) * BM, bh % kp.H, 0);
        else
          tma_load_3d(sQ + t * TILE8, &tmQ, &q_full[t], 0, (g * NQ8 + t) * BM, bh);
      }
      int it = 0;
      bool ok = true;
      for (int j = 0; j < nKmax && ok; ++j) {
        for (int kv = 0; kv < 2; ++kv) {
          const int slot = it % NSLOT8;
          const int use = it / NSLOT8;
          if (use >= 1 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, ab, kDevTimeoutLoad)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&kv_full[slot], TILE8);
          if constexpr (PACKED)
            tma_load_4d(sKV + slot * TILE8, kv ? &tmV : &tmK, &kv_full[slot], 0, seq0 + j * BN,
                        kvp % kp.H_kv, 0);
          else
            tma_load_3d(sKV + slot * TILE8, kv ? &tmV : &tmK, &kv_full[slot], 0, j * BN, kvp);
          ++it;
        }
      }
      load_items_sh = it;
    }
  } else if (warp == MMA_WARP8) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_e4m3(128, BN, false, false);
      constexpr uint32_t idPV = idesc_e4m3(128, D8, false, true);
      const uint64_t qdesc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);     // K-major Q
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(sKV), 16, 1024);    // K-major K
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(sKV), TILE8, 1024); // MN-major V
      bool ok = true;
#pragma unroll
      for (int t = 0; t < NQ8; ++t)
        if (ok && nK[t] > 0) ok = mbar_wait(&q_full[t], 0, ab, kDevTimeoutMma);
      for (int j = 0; j <= nKmax && ok; ++j) {
        const int itK = 2 * j;          // ring item of K_j
        const int itV = 2 * j - 1;      // ring item of V_{j-1}
        const int slotK = itK % NSLOT8;
        const int slotV = (itV + NSLOT8) % NSLOT8;
        bool haveK = false, haveV = false;
        uint64_t kdesc = 0, vdesc = 0;
#pragma unroll
        for (int t = 0; t < NQ8; ++t) {
          if (j >= 1 && j - 1 < nK[t]) {
            // O_t += P_t(j-1) V_{j-1}
            if (!haveV) {
              if (!(ok = mbar_wait(&kv_full[slotV], (itV / NSLOT8) & 1, ab, kDevTimeoutMma))) break;
              vdesc = opaque(sdesc_add(vdesc0, slotV * TILE8));
              haveV = true;
            }
            if (!(ok = mbar_wait(&p_full[t], (j - 1) & 1, ab, kDevTimeoutMma))) break;
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < BN / 32; ++kk)
              mma_f8_ts(tmem + o_col8(t), tmem + s_col8(t) + p_col8(kk), sdesc_add(vdesc, kk * 32 * 128),
                        idPV, (j - 1 > 0 || kk > 0) ? 1u : 0u);
            if (j - 1 == nK[t] - 1) mma_commit(&o_full[t]);
          }
          if (j < nK[t]) {
            // S_t(j) = Q_t K_j^T
            if (!haveK) {
              if (!(ok = mbar_wait(&kv_full[slotK], (itK / NSLOT8) & 1, ab, kDevTimeoutMma))) break;
              tc_fence_after_sync();
              kdesc = opaque(sdesc_add(kdesc0, slotK * TILE8));
              haveK = true;
            }
            const uint64_t qdesc = sdesc_add(qdesc0, t * TILE8);
#pragma unroll
            for (int kk = 0; kk < D8 / 32; ++kk)
              mma_f8_ss(tmem + s_col8(t), sdesc_add(qdesc, kk * 32), sdesc_add(kdesc, kk * 32), idS,
                        kk > 0 ? 1u : 0u);
            mma_commit(&s_full[t]);
          }
        }
        if (!ok) break;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w: query tile t = w / 8, key half h = (w / 4) % 2, rows of its TMEM
    // lane quarter.  The two warps of a row exchange their partial row max
    // once per step through shared memory (named barrier per warp pair).
    const int t = warp / 8;
    const int h = (warp / 4) & 1;
    const int quarter = warp % 4;
    const int r = quarter * 32 + lane;
    const uint32_t pair_bar = 1 + t * 4 + quarter;
    const int qt = g * NQ8 + t;
    const int my_nK = (qt * BM < N) ? (CAUSAL ? min(nKtot, qt + 1) : nKtot) : 0;
    const int row_g = qt * BM + r;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_addr + s_col8(t) + 64 * h;       // this half's scores
    const uint32_t tO = tmem + lane_addr + o_col8(t) + (D8 / 2) * h;  // this half's O columns
    const float* kdesc = kp.k_descale + static_cast<size_t>(kvp) * kp.nblk;
    const float* vdesc = kp.v_descale + static_cast<size_t>(kvp) * kp.nblk;
    float dv_max = 0.f;
    for (int b = 0; b < (N + BN - 1) / BN; ++b) dv_max = fmaxf(dv_max, vdesc[b]);
    const float inv_dv_max = 1.f / dv_max;
    const float c_q = (my_nK > 0) ? kp.scale_log2 * kp.q_descale[static_cast<size_t>(bh) * kp.nblk + qt] : 0.f;
    float m_ref = -INFINITY;   // in log2 units of the scaled scores
    float l = 0.f;             // this half's share of the row sum
    bool ok = true;
    for (int j = 0; j < my_nK; ++j) {
      const float cj = c_q * kdesc[j];
      const float ratio = vdesc[j] * inv_dv_max;          // in (0, 1]
      const float lg_ratio = lg2_approx8(ratio);
      float inv_ratio;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv_ratio) : "f"(ratio));
      // A warp that gives up (decided for the whole warp: the TMEM loads below
      // are warp-collective) still arrives at this step's pair barrier, where
      // its partner may be waiting; the partner then fails its next wait too,
      // since this warp never signals p_full again.
      if (__any_sync(0xffffffffu, !mbar_wait(&s_full[t], j & 1, ab, kDevTimeoutSoftmax))) {
        named_bar_arrive(pair_bar, 64);
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (t == t_rel && h == 0 && r == 0) {
        if (2 * j + NSLOT8 < total_items) mbar_arrive(&kv_empty[(2 * j) % NSLOT8]);
        if (j >= 1 && 2 * j - 1 + NSLOT8 < total_items) mbar_arrive(&kv_empty[(2 * j - 1) % NSLOT8]);
      }
      uint32_t sr[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld_wait();
      const int kbase = j * BN + 64 * h;
      if ((CAUSAL && j == qt) || kbase + 64 > N) {
        const int lim = (CAUSAL ? min(N, row_g + 1) : N) - kbase;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        mx[u] = fmax3(__uint_as_float(sr[8 * u]), __uint_as_float(sr[8 * u + 1]),
                      fmax3(__uint_as_float(sr[8 * u + 2]), __uint_as_float(sr[8 * u + 3]),
                            fmax3(__uint_as_float(sr[8 * u + 4]), __uint_as_float(sr[8 * u + 5]),
                                  fmaxf(__uint_as_float(sr[8 * u + 6]), __uint_as_float(sr[8 * u + 7])))));
      const float m_half = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                 fmaxf(mx[6], mx[7])) * cj;
      xch[j & 1][t][h][r] = m_half;
      named_bar_sync(pair_bar, 64);
      const float m_new = fmaxf(m_ref, fmaxf(m_half, xch[j & 1][t][h ^ 1][r]));
      // both halves of a row take the same decision
      const bool need = (m_new - m_ref) > 8.f;
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx(m_ref - m_new);
        l *= alpha;
        m_ref = m_new;
      }
      // exponent offset: -m_ref (the running reference) + log2(dv_j / dv_max)
      const float off = ((m_ref == -INFINITY) ? 0.f : -m_ref) + lg_ratio;
      const uint64_t cc = pack2(cj, cj);
      const uint64_t nn = pack2(off, off);
      uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
      for (int c0 = 0; c0 < 2; ++c0) {
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = c0 * 32 + 4 * i;
          const uint64_t y0 = ffma2(pack2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), cc, nn);
          const uint64_t y1 = ffma2(pack2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), cc, nn);
          float p0, p1, p2, p3;
          if (POLY > 0 && (((c0 * 8 + i) * POLY) % 16) < POLY) {
            const uint64_t e0 = exp2_poly2(lo2(y0), hi2(y0));
            const uint64_t e1 = exp2_poly2(lo2(y1), hi2(y1));
            p0 = lo2(e0);
            p1 = hi2(e0);
            p2 = lo2(e1);
            p3 = hi2(e1);
          } else {
            p0 = ex2_approx(lo2(y0));
            p1 = ex2_approx(hi2(y0));
            p2 = ex2_approx(lo2(y1));
            p3 = ex2_approx(hi2(y1));
          }
          acc0 = fadd2(acc0, pack2(p0, p1));
          acc1 = fadd2(acc1, pack2(p2, p3));
          pk[i] = cvt_pack_e4m3x4(p0, p1, p2, p3);
        }
        // packed P of keys [64 h + 32 c0, +32) -> columns [64 h + 8 c0, +8)
        tmem_st_x8(tS + c0 * 8, pk);
      }
      const uint64_t acc = fadd2(acc0, acc1);
      l = fmaf(lo2(acc) + hi2(acc), inv_ratio, l);          // sum of the unscaled P
      // Rescale this half's columns of O (this step's P V product is issued
      // only after the arrive below; the previous one finished before S_t(j)).
      if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c0 = 0; c0 < D8 / 64; ++c0) {
          uint32_t o[32];
          tmem_ld32(tO + c0 * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + c0 * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&p_full[t]);
    }
    bool out_ok = ok && my_nK > 0;
    if (out_ok && __any_sync(0xffffffffu, !mbar_wait(&o_full[t], 0, ab, kDevTimeoutEpilogue))) {
      named_bar_arrive(pair_bar, 64);   // release the partner at the barrier below
      out_ok = false;
    }
    if (out_ok) {
      tc_fence_after_sync();
      // row sum = both halves' shares (buffer of parity my_nK & 1 is free: its
      // last readers passed this pair's barrier of step my_nK - 1)
      xch[my_nK & 1][t][h][r] = l;
      named_bar_sync(pair_bar, 64);
      const float l_row = l + xch[my_nK & 1][t][h ^ 1][r];
      const float mul = dv_max / l_row;
      const size_t orow_idx = PACKED ? static_cast<size_t>(seq0 + row_g) * kp.H + bh % kp.H
                                     : static_cast<size_t>(bh) * N + row_g;
      uint16_t* orow = static_cast<uint16_t*>(kp.o) + orow_idx * D8 + (D8 / 2) * h;
#pragma unroll 1
      for (int c0 = 0; c0 < D8 / 64; ++c0) {
        uint32_t o[32];
        tmem_ld32(tO + c0 * 32, o);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = cvt_pack_bf16(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
        if (row_g < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (h == 0 && row_g < N)
        kp.lse[PACKED ? static_cast<size_t>(bh % kp.H) * kp.total + seq0 + row_g
                      : static_cast<size_t>(bh) * N + row_g] =
            (m_ref + lg2_approx8(l_row)) * 0.69314718055994530942f;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (abort_sh) {
    if (warp == LOAD_WARP8 && lane == 0) {
#pragma unroll
      for (int t = 0; t < NQ8; ++t)
        if (nK[t] > 0) mbar_wait_drain(&q_full[t], 0);
      const int issued = load_items_sh;
      for (int s = 0; s < NSLOT8 && s < issued; ++s)
        mbar_wait_drain(&kv_full[s], ((issued - 1 - s) / NSLOT8) & 1);
    }
    if (warp == MMA_WARP8 && lane == 0) {
      mma_commit(&drain_bar);
      mbar_wait_drain(&drain_bar, 0);
    }
    __syncthreads();
  }
  if (warp == MMA_WARP8) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// Evaluates exp2_poly2 and ex2.approx on the same inputs (diagnostic entry
// point attn_selftest_exp2).
__global__ void exp2_selftest_kernel(const float* __restrict__ x, float* __restrict__ y_poly,
                                     float* __restrict__ y_mufu, long long n) {
  const long long i = 2 * (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float a = x[i];
  const float b = (i + 1 < n) ? x[i + 1] : 0.f;
  const uint64_t e = exp2_poly2(a, b);
  y_poly[i] = lo2(e);
  y_mufu[i] = ex2_approx(a);
  if (i + 1 < n) {
    y_poly[i + 1] = hi2(e);
    y_mufu[i + 1] = ex2_approx(b);
  }
}

// Block mode, or the per-tensor comparator (block amaxes, one reduction, codes).
template <bool BF16IN>
void launch_quant_modes(const Fp8QuantParams& p, dim3 grid, int nblk, int kv_planes,
                        cudaStream_t stream) {
  if (!p.per_tensor) {
    fp8_quant_kernel<0, false, BF16IN><<<grid, 256, 0, stream>>>(
        p.src[0], p.src[1], p.src[2], p.dst[0], p.dst[1], p.dst[2], p.descale[0], p.descale[1],
        p.descale[2], p.signs, p.N, nblk, kv_planes);
    return;
  }
  fp8_quant_kernel<1, false, BF16IN><<<grid, 256, 0, stream>>>(
      p.src[0], p.src[1], p.src[2], p.dst[0], p.dst[1], p.dst[2], p.descale[0], p.descale[1],
      p.descale[2], nullptr, p.N, nblk, kv_planes);
  fp8_tensor_scale_kernel<<<3, 256, 0, stream>>>(p.descale[0], p.descale[1], p.descale[2],
                                                 static_cast<long long>(p.B) * p.H * nblk,
                                                 static_cast<long long>(kv_planes) * nblk);
  fp8_quant_kernel<2, false, BF16IN><<<grid, 256, 0, stream>>>(
      p.src[0], p.src[1], p.src[2], p.dst[0], p.dst[1], p.dst[2], p.descale[0], p.descale[1],
      p.descale[2], nullptr, p.N, nblk, kv_planes);
}

}  // namespace

attn_status_t launch_exp2_selftest(const float* x, float* y_poly, float* y_mufu, long long n,
                                   cudaStream_t stream) {
  const long long pairs = (n + 1) / 2;
  exp2_selftest_kernel<<<static_cast<unsigned>((pairs + 255) / 256), 256, 0, stream>>>(x, y_poly,
                                                                                        y_mufu, n);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "exp2 self-test launch");
  return ATTN_OK;
}

attn_status_t launch_fp8_quantize(const Fp8QuantParams& p, cudaStream_t stream) {
  if (p.d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 path supports d = 128");
  const int nblk = (p.N + 127) / 128;
  if (p.B * p.H > 65535 || nblk > 2147483647 / 128)
    return fail(ATTN_ERR_UNSUPPORTED, "grid dimension limit exceeded");
  const int H_kv = p.H_kv > 0 ? p.H_kv : p.H;
  const int kv_planes = p.B * H_kv;
  dim3 grid(nblk, p.B * p.H, 3);
  const bool rope = p.rope_cos != nullptr;
  if (rope && p.per_tensor) return fail(ATTN_ERR_UNSUPPORTED, "rotation takes the block pre-pass only");
  if (p.cu_seqlens && p.per_tensor)
    return fail(ATTN_ERR_UNSUPPORTED, "packed batches take the block pre-pass only");
  if (p.cu_seqlens || rope) {
    int* status = device_status_word();
    if (!status) return fail(ATTN_ERR_CUDA, "status word unavailable");
    if (rope && !p.cu_seqlens && !p.in_bf16) {
      // float32 rows staged in shared memory by bulk copies (measured faster
      // than holding a rotated block in registers)
      auto kern = fp8_quant_staged_kernel<0, true>;
      attn_status_t s = set_smem(reinterpret_cast<const void*>(kern), QSMEM);
      if (s != ATTN_OK) return s;
      kern<<<grid, 256, QSMEM, stream>>>(static_cast<const float*>(p.src[0]),
                                         static_cast<const float*>(p.src[1]),
                                         static_cast<const float*>(p.src[2]), p.dst[0], p.dst[1],
                                         p.dst[2], p.descale[0], p.descale[1], p.descale[2], p.signs,
                                         p.N, nblk, kv_planes, status, p.rope_cos, p.rope_sin);
    } else {
      // register-staged block pre-pass: {packed, bfloat16 input, rotation}
      auto kern = fp8_quant_kernel<0, false, false, false>;
      const int sel = (p.cu_seqlens ? 4 : 0) | (p.in_bf16 ? 2 : 0) | (rope ? 1 : 0);
      switch (sel) {
        case 1: kern = fp8_quant_kernel<0, false, false, true>; break;
        case 2: kern = fp8_quant_kernel<0, false, true, false>; break;
        case 3: kern = fp8_quant_kernel<0, false, true, true>; break;
        case 4: kern = fp8_quant_kernel<0, true, false, false>; break;
        case 5: kern = fp8_quant_kernel<0, true, false, true>; break;
        case 6: kern = fp8_quant_kernel<0, true, true, false>; break;
        case 7: kern = fp8_quant_kernel<0, true, true, true>; break;
        default: break;
      }
      kern<<<grid, 256, 0, stream>>>(p.src[0], p.src[1], p.src[2], p.dst[0], p.dst[1], p.dst[2],
                                     p.descale[0], p.descale[1], p.descale[2], p.signs, p.N, nblk,
                                     kv_planes, p.cu_seqlens, p.total, p.H, H_kv, status,
                                     p.rope_cos, p.rope_sin);
    }
  } else if (p.in_bf16) {
    launch_quant_modes<true>(p, grid, nblk, kv_planes, stream);
  } else {
    launch_quant_modes<false>(p, grid, nblk, kv_planes, stream);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "FP8 pre-pass launch");
  return ATTN_OK;
}

template <bool CAUSAL, bool PACKED, int POLY = 0>
attn_status_t launch_fwd_fp8_t(const Fp8FwdParams& p, cudaStream_t stream) {
  auto kern = fwd_fp8_kernel<CAUSAL, PACKED, POLY>;
  attn_status_t s = set_smem(reinterpret_cast<const void*>(kern), SMEM8);
  if (s != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
  if constexpr (PACKED) {
    // {d, total tokens, heads, 1}: token stride heads * d bytes, head stride d
    const uint64_t T = static_cast<uint64_t>(p.total);
    if ((s = make_tmap_4d(&tq, p.q8, 1, D8, T, p.H, 1, 1ull * p.H * D8, D8, T * p.H * D8, 128,
                          BM)) != ATTN_OK)
      return s;
    if ((s = make_tmap_4d(&tk, p.k8, 1, D8, T, p.H_kv, 1, 1ull * p.H_kv * D8, D8, T * p.H_kv * D8,
                          128, BN)) != ATTN_OK)
      return s;
    if ((s = make_tmap_4d(&tv, p.v8, 1, D8, T, p.H_kv, 1, 1ull * p.H_kv * D8, D8, T * p.H_kv * D8,
                          128, BN)) != ATTN_OK)
      return s;
  } else {
    const uint64_t planes = static_cast<uint64_t>(p.B) * p.H;
    const uint64_t kv_planes = static_cast<uint64_t>(p.B) * p.H_kv;
    if ((s = make_tmap_3d(&tq, p.q8, 1, D8, p.N, planes, 128, BM)) != ATTN_OK) return s;
    if ((s = make_tmap_3d(&tk, p.k8, 1, D8, p.N, kv_planes, 128, BN)) != ATTN_OK) return s;
    if ((s = make_tmap_3d(&tv, p.v8, 1, D8, p.N, kv_planes, 128, BN)) != ATTN_OK) return s;
  }
  int* status = device_status_word();
  if (!status) return fail(ATTN_ERR_CUDA, "status word unavailable");
  Fp8KParams kp{p.q_descale, p.k_descale, p.v_descale, p.o, p.lse, status, p.N, p.H,
                (p.N + 127) / 128, p.scale * 1.4426950408889634f, p.H_kv, p.cu_seqlens, p.total};
  const unsigned npairs = static_cast<unsigned>((p.N + BM * NQ8 - 1) / (BM * NQ8));
  const dim3 grid = CAUSAL ? dim3(npairs * p.H * p.B, 1, 1) : dim3(npairs, p.H, p.B);
  kern<<<grid, THREADS8, SMEM8, stream>>>(tq, tk, tv, kp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "FP8 forward launch");
  return ATTN_OK;
}

attn_status_t launch_fwd_fp8(const Fp8FwdParams& p, cudaStream_t stream) {
  if (p.d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 path supports d = 128");
  if (p.N > 65535 * 256 || p.H > 65535 || p.B > 65535)
    return fail(ATTN_ERR_UNSUPPORTED, "grid dimension limit exceeded");
  // The library's share of exponentials on the FMA pipe (in sixteenths): one
  // sixteenth for non-causal batches (at B = 2, H = 16, N = 8192: 1732 TFLOP/s
  // with none, 1765 with one eighth, 1777 with one sixteenth; causal unchanged;
  // three sixteenths or more slower), none for causal ones.  Packed batches take
  // the same choice, so one packed sequence gives the bits of the fixed-length call.
  const int poly = p.exp2_poly >= 0 ? p.exp2_poly : (p.causal ? 0 : 1);
  if (p.cu_seqlens) {
    if (poly == 0)
      return p.causal ? launch_fwd_fp8_t<true, true>(p, stream) : launch_fwd_fp8_t<false, true>(p, stream);
    if (poly == 1 && !p.causal) return launch_fwd_fp8_t<false, true, 1>(p, stream);
    return fail(ATTN_ERR_UNSUPPORTED, "packed batches take the library's exponential split");
  }
  switch (poly) {
    case 0: break;
    case 1: return p.causal ? launch_fwd_fp8_t<true, false, 1>(p, stream) : launch_fwd_fp8_t<false, false, 1>(p, stream);
    case 2: return p.causal ? launch_fwd_fp8_t<true, false, 2>(p, stream) : launch_fwd_fp8_t<false, false, 2>(p, stream);
    case 4: return p.causal ? launch_fwd_fp8_t<true, false, 4>(p, stream) : launch_fwd_fp8_t<false, false, 4>(p, stream);
    case 6: return p.causal ? launch_fwd_fp8_t<true, false, 6>(p, stream) : launch_fwd_fp8_t<false, false, 6>(p, stream);
    case 8: return p.causal ? launch_fwd_fp8_t<true, false, 8>(p, stream) : launch_fwd_fp8_t<false, false, 8>(p, stream);
    default: return fail(ATTN_ERR_INVALID_ARG, "exp2 share must be 0, 1, 2, 4, 6 or 8 sixteenths");
  }
  return p.causal ? launch_fwd_fp8_t<true, false>(p, stream) : launch_fwd_fp8_t<false, false>(p, stream);
}

}  // namespace attn
