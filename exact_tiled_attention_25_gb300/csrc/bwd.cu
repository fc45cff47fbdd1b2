// BF16/FP16 attention backward on sm_103a.
//
// Method: "FlashAttention-3: Hopper Asynchrony and FP8 Attention", section
// "Backward warp specialization": producers load K_j and V_j, then stream Q_i
// and dO_i; consumers recompute S and P from the stored L_i, form dP, dS, dV
// and dK; a separate writer adds each local dQ tile into global dQ.  The
// gradient formulas are the chain rule through softmax:
//   P = exp(scale * Q K^T - L),  dV = P^T dO,  dP = dO V^T,
//   dS = P * (dP - D) with D_i = rowsum(dO_i * O_i),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Three kernels:
//  1. prep: -D = -rowsum(dO * O) and -L * log2(e) into 128-row padded arrays
//     (padding: 0 and -inf, so padded query rows get P = 0), and the float32
//     dQ accumulator is zeroed.
//  2. main: one CTA per (key/value tile j, head, batch).  K_j and V_j stay in
//     shared memory; dK_j and dV_j accumulate in tensor memory.  Per query tile
//     i (causal: i >= j) the MMA thread issues, on tcgen05,
//        dP^T = V_j dO_i^T  (it needs nothing from this step's softmax),
//     while the compute warpgroups (thread = key row) form P^T from S^T = K_j
//     Q_i^T (issued the step before) and write it back to tensor memory; then
//        dV += P^T dO_i,   S^T(next) = K_j Q_{i+1}^T,
//     while the same warpgroups form dS^T = P^T (dP^T - D) (into tensor memory
//     for dK, into shared memory for dQ); then
//        dK += dS^T Q_i,   dQ_i = dS K_j  (into tensor memory, one query per lane).
//     The dQ-writer warps (two reduce warpgroups) copy dQ_i out of tensor
//     memory, stage it in 4 KB boxes in shared memory and add each box into
//     the float32 accumulator with a TMA reduce-add, so the reduction runs in
//     the TMA unit and L2 instead of as per-thread atomics.
//  3. convert: dQ = scale * accumulator, rounded to the 16-bit type.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "common.h"
#include "sm103_prims.cuh"

namespace attn {
namespace {

constexpr int kSmemLimit = 232448;
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int D>
struct BwdCfg {
  static constexpr int BM = 128;                 // query rows per step
  static constexpr int BN = 128;                 // keys per CTA
  static constexpr int CH = D / 64;              // 128-byte chunks per row
  static constexpr int CHUNK = 128 * 128;        // one 128-row x 128-byte chunk
  static constexpr int TILE = 128 * D * 2;       // a K, V, Q or dO tile
  // Q_i (with its row vectors) and dO_i have rings of their own: Q_i is read
  // by S^T(i) early and dK late, dO_i only by dP^T(i) and dV.  At d = 128 one
  // dO slot is all that fits next to the dQ staging buffers.
  static constexpr int NQS = 2;                  // Q ring slots
  static constexpr int NDS = (D == 128) ? 1 : 2; // dO ring slots
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;
  static constexpr int OFF_DO = OFF_Q + NQS * TILE;
  static constexpr int OFF_DS = OFF_DO + NDS * TILE;      // dS^T, 128 keys x 128 queries
  // dQ staging: one 32-query x 32-column float32 box (4 KB, 128-byte swizzle)
  // per reduce warp, handed to a TMA reduce-add into the float32 accumulator
  static constexpr int STG_BOX = 32 * 32 * 4;
  static constexpr int OFF_STG = OFF_DS + 2 * CHUNK;
  static constexpr int OFF_LD = OFF_STG + 8 * STG_BOX;    // per Q slot: L*log2e[128], D[128]
  static constexpr int OFF_BAR = OFF_LD + NQS * 1024;
  static constexpr int NEED = OFF_BAR + 256;
  static constexpr int SMEM_BYTES = cmin(kSmemLimit, NEED + 1024);
  static constexpr int SLACK = SMEM_BYTES - NEED;   // room to align the base to 1024
  // TMEM columns: S^T/P^T [0,128), dP^T/dS^T [128,256), dV, dK.  At d = 128
  // there is no room left, so dQ reuses the dP^T columns (after dK has read
  // dS^T there); at d = 64 dQ has its own columns.  dQ is stored with one
  // query per TMEM lane.
  static constexpr bool DQ_IN_DP = (D == 128);
  static constexpr uint32_t S_COL = 0;
  static constexpr uint32_t DP_COL = 128;
  static constexpr uint32_t DV_COL = 256;
  static constexpr uint32_t DK_COL = 256 + D;
  static constexpr uint32_t DQ_COL = DQ_IN_DP ? DP_COL : 256 + 2 * D;
  // Warps 0-7: two compute warpgroups (one per half of the 128 query columns);
  // warps 8-15: two reduce warpgroups (one per half of dQ's columns);
  // warp 16: TMA producer; warp 17: MMA issuer.
  static constexpr int THREADS = 576;
  static constexpr int LOAD_WARP = 16;
  static constexpr int MMA_WARP = 17;
  // Packed 16-bit P^T / dS^T of query half h sit in columns [64 h, 64 h + 32) of
  // the S^T / dP^T region, inside the half's own fp32 columns, so each
  // warpgroup overwrites only scores it has already read.
  __host__ __device__ static constexpr uint32_t half_col(int kk) {
    return 64u * static_cast<uint32_t>(kk / 4) + 8u * static_cast<uint32_t>(kk % 4);
  }
  static_assert(DQ_COL + D <= 512 && DK_COL + D <= 512, "TMEM overflow");
  static_assert(SLACK >= 0, "shared memory overflow");
  static_assert(OFF_STG % 1024 == 0, "staging boxes need 1024-byte alignment (swizzle atoms)");
};

struct Bars {
  uint64_t kv_full;
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t do_full[2];
  uint64_t do_empty[2];
  uint64_t s_full;
  uint64_t dp_full;
  uint64_t p_ready;
  uint64_t ds_ready;
  uint64_t dq_full;
  uint64_t dq_free;
  uint64_t dkv_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int q_items;     // Q slots the producer filled (for draining after an abort)
  int do_items;    // dO slots the producer filled
};

struct BwdKParams {
  void* dk;
  void* dv;
  float* dq_acc;        // same layout as dQ
  const float* lse2;    // -L * log2(e), [B*H][Npad], -inf padding
  const float* delta;   // -rowsum(dO * O), [B*H][Npad], 0 padding
  int* status;
  const int* cu_seqlens;   // packed batch offsets [B + 1], else nullptr
  int N;                   // sequence length, or the longest sequence of a packed batch
  int Npad;
  int total;               // tokens of a packed batch
  int H;
  int H_kv;
  int group;               // query heads per key/value head
  float scale;
  float scale_log2;
};

// Sequence b of a packed batch: first token and length, or false when its
// offsets do not fit (outside [0, total], decreasing, or longer than max_len).
__device__ __forceinline__ bool packed_seq(const int* cu, int b, int total, int max_len, int& s0,
                                           int& len) {
  s0 = cu[b];
  const int e = cu[b + 1];
  if (s0 < 0 || e < s0 || e > total || e - s0 > max_len) return false;
  len = e - s0;
  return true;
}

// ------------------------------------------------------------------ prep ----
// One group of D/8 lanes per row; each lane holds 8 consecutive elements.
// Rows of O, dO and dQ are [B, H, N, d] or, for a packed batch (PACKED),
// [total, H, d] with LSE [H, total].
template <int D, bool FP16, bool PACKED>
__global__ void __launch_bounds__(256)
    bwd_prep_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                    const float* __restrict__ lse, float* __restrict__ lse2,
                    float* __restrict__ delta, float* __restrict__ dq_acc, int N, int Npad,
                    long long total_rows_pad, int H, const int* __restrict__ cu_seqlens,
                    int total) {
  constexpr int L = D / 8;
  constexpr int ROWS_PER_WARP = 32 / L;
  const int lane = threadIdx.x & 31;
  const int sub = lane / L;
  const int li = lane % L;
  const long long warp_global = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const long long prow = warp_global * ROWS_PER_WARP + sub;   // padded row index
  if (prow >= total_rows_pad) return;
  const long long bh = prow / Npad;
  const int n = static_cast<int>(prow - bh * Npad);
  int len = N;
  long long row, lrow;     // row of O / dO / dQ, index into LSE
  if constexpr (PACKED) {
    const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
    int s0 = 0;
    if (!packed_seq(cu_seqlens, b, total, N, s0, len)) len = 0;   // reported by the main kernel
    row = (static_cast<long long>(s0) + n) * H + h;
    lrow = static_cast<long long>(h) * total + s0 + n;
  } else {
    row = bh * N + n;
    lrow = row;
  }
  float acc = 0.f;
  if (n < len) {
    const uint4 a = reinterpret_cast<const uint4*>(o + row * D)[li];
    const uint4 b = reinterpret_cast<const uint4*>(dout + row * D)[li];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 fa, fb;
      if (FP16) {
        fa = __half22float2(*reinterpret_cast<const __half2*>(&av[e]));
        fb = __half22float2(*reinterpret_cast<const __half2*>(&bv[e]));
      } else {
        fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
        fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bv[e]));
      }
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + row * D) + 2 * li;
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = L / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (li == 0) {
    // stored negated so the main kernel adds them with packed f32x2 FMAs
    delta[prow] = (n < len) ? -acc : 0.f;
    lse2[prow] = (n < len) ? -lse[lrow] * kLog2e : -INFINITY;
  }
}

// --------------------------------------------------------------- convert ----
template <bool FP16>
__global__ void __launch_bounds__(256)
    bwd_convert_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq, float scale,
                       long long n8) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 r;
    if (FP16) {
      r.x = cvt_pack_f16(a.x * scale, a.y * scale);
      r.y = cvt_pack_f16(a.z * scale, a.w * scale);
      r.z = cvt_pack_f16(b.x * scale, b.y * scale);
      r.w = cvt_pack_f16(b.z * scale, b.w * scale);
    } else {
      r.x = cvt_pack_bf16(a.x * scale, a.y * scale);
      r.y = cvt_pack_bf16(a.z * scale, a.w * scale);
      r.z = cvt_pack_bf16(b.x * scale, b.y * scale);
      r.w = cvt_pack_bf16(b.z * scale, b.w * scale);
    }
    reinterpret_cast<uint4*>(dq)[i] = r;
  }
}

// ------------------------------------------------------------------ main ----
template <int D, bool CAUSAL, bool FP16, bool PACKED>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdKParams kp) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  if (pad > static_cast<uint32_t>(C::SLACK)) {
    // Cannot place the swizzled tiles: report and leave before touching anything.
    if (threadIdx.x == 0) atomicCAS(kp.status, 0, kDevSmemMisaligned);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  Bars& bars = *reinterpret_cast<Bars*>(smem + C::OFF_BAR);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // One CTA per (key tile j, key/value head hk, batch b).  Causal: a 1-D grid
  // ordered by work, key tile 0 (which meets every query tile) of every head
  // first.  Non-causal: (tile, head, batch).
  const int ntiles = (kp.N + C::BN - 1) / C::BN;
  const int j = CAUSAL ? static_cast<int>(blockIdx.x / (gridDim.x / ntiles)) : static_cast<int>(blockIdx.x);
  const int bhk = CAUSAL ? static_cast<int>(blockIdx.x % (gridDim.x / ntiles))
                         : static_cast<int>(blockIdx.z * kp.H_kv + blockIdx.y);
  const int b = bhk / kp.H_kv;
  const int hk = bhk - b * kp.H_kv;
  int seq0 = 0, N = kp.N;
  if constexpr (PACKED) {
    // this sequence's first token and length; key tiles past its end have no
    // work (the whole CTA leaves before touching any resource)
    if (!packed_seq(kp.cu_seqlens, b, kp.total, kp.N, seq0, N)) {
      if (threadIdx.x == 0 && j == 0) atomicCAS(kp.status, 0, kDevBadSeqlens);
      return;
    }
    if (j * C::BN >= N) return;
  }
  const int nQ = (N + C::BM - 1) / C::BM;
  const int i0 = CAUSAL ? j : 0;
  // Steps walk query tiles i0 .. nQ-1 of the group's first query head, then of
  // the next one: dK_j, dV_j accumulate over every query head sharing K_j, V_j.
  const int nsteps = kp.group * (nQ - i0);
  const int h0 = hk * kp.group;          // first query head of the group

  if (threadIdx.x == 0) {
    mbar_init(&bars.kv_full, 1);
    for (int s = 0; s < C::NQS; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.q_empty[s], 1);
    }
    for (int s = 0; s < C::NDS; ++s) {
      mbar_init(&bars.do_full[s], 1);
      mbar_init(&bars.do_empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.p_ready, 256);
    mbar_init(&bars.ds_ready, 256);
    mbar_init(&bars.dq_full, 1);
    mbar_init(&bars.dq_free, 256);
    mbar_init(&bars.dkv_full, 1);
    mbar_init(&bars.drain, 1);
    bars.abort_flag = 0;
    bars.q_items = 0;
    bars.do_items = 0;
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars.tmem_base;
  const Abort ab{&bars.abort_flag, kp.status};

  if (warp == C::LOAD_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmDO);
      mbar_arrive_expect_tx(&bars.kv_full, 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) {
        // coordinates {c, token, head, 0} for a packed batch, else {c, row, plane}
        if constexpr (PACKED) {
          tma_load_4d(smem + C::OFF_K + c * C::CHUNK, &tmK, &bars.kv_full, c * 64, seq0 + j * C::BN, hk, 0);
          tma_load_4d(smem + C::OFF_V + c * C::CHUNK, &tmV, &bars.kv_full, c * 64, seq0 + j * C::BN, hk, 0);
        } else {
          tma_load_3d(smem + C::OFF_K + c * C::CHUNK, &tmK, &bars.kv_full, c * 64, j * C::BN, bhk);
          tma_load_3d(smem + C::OFF_V + c * C::CHUNK, &tmV, &bars.kv_full, c * 64, j * C::BN, bhk);
        }
      }
      int nq = 0, nd = 0;                  // Q and dO loads issued
      int i = i0, h = h0;                  // query tile and query head of step n
      for (int n = 0; n < nsteps; ++n, (++i == nQ) ? (i = i0, ++h) : 0) {
        // Q_i with its row vectors -L*log2(e) and -D into Q slot n % NQS, freed
        // by dK of step n - NQS
        {
          const int st = n % C::NQS;
          const int use = n / C::NQS;
          if (use >= 1 && !mbar_wait(&bars.q_empty[st], (use - 1) & 1, ab, kDevTimeoutLoad)) break;
          uint8_t* sq = smem + C::OFF_Q + st * C::TILE;
          float* sld = reinterpret_cast<float*>(smem + C::OFF_LD + st * 1024);
          mbar_arrive_expect_tx(&bars.q_full[st], C::TILE + 1024);
#pragma unroll
          for (int c = 0; c < C::CH; ++c) {
            if constexpr (PACKED)
              tma_load_4d(sq + c * C::CHUNK, &tmQ, &bars.q_full[st], c * 64, seq0 + i * C::BM, h, 0);
            else
              tma_load_3d(sq + c * C::CHUNK, &tmQ, &bars.q_full[st], c * 64, i * C::BM, b * kp.H + h);
          }
          const size_t roff = (static_cast<size_t>(b) * kp.H + h) * kp.Npad + static_cast<size_t>(i) * C::BM;
          bulk_load(sld, kp.lse2 + roff, 512, &bars.q_full[st]);
          bulk_load(sld + 128, kp.delta + roff, 512, &bars.q_full[st]);
          ++nq;
        }
        // dO_i into dO slot n % NDS, freed once dP^T and dV of step n - NDS completed
        {
          const int st = n % C::NDS;
          const int use = n / C::NDS;
          if (use >= 1 && !mbar_wait(&bars.do_empty[st], (use - 1) & 1, ab, kDevTimeoutLoad)) break;
          uint8_t* sdo = smem + C::OFF_DO + st * C::TILE;
          mbar_arrive_expect_tx(&bars.do_full[st], C::TILE);
#pragma unroll
          for (int c = 0; c < C::CH; ++c) {
            if constexpr (PACKED)
              tma_load_4d(sdo + c * C::CHUNK, &tmDO, &bars.do_full[st], c * 64, seq0 + i * C::BM, h, 0);
            else
              tma_load_3d(sdo + c * C::CHUNK, &tmDO, &bars.do_full[st], c * 64, i * C::BM, b * kp.H + h);
          }
          ++nd;
        }
      }
      bars.q_items = nq;
      bars.do_items = nd;
    }
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr Elt E = FP16 ? Elt::F16 : Elt::BF16;
      constexpr uint32_t idSP = idesc_f16(E, 128, 128, false, false);   // S^T and dP^T
      constexpr uint32_t idKV = idesc_f16(E, 128, D, false, true);      // dV and dK (A in TMEM)
      // dQ_i = dS K_j: rows = queries; A = dS (the dS^T buffer read MN-major),
      // B = K_j MN-major
      constexpr uint32_t idQ = idesc_f16(E, 128, D, true, true);
      const uint32_t sK = smem_u32(smem + C::OFF_K);
      const uint32_t sV = smem_u32(smem + C::OFF_V);
      const uint32_t sDS = smem_u32(smem + C::OFF_DS);
      const uint64_t mK = opaque(sdesc_sw128(sK, C::CHUNK, 1024));
      const uint64_t mDS = opaque(sdesc_sw128(sDS, C::CHUNK, 1024));
      // S^T(i) = K_j Q_i^T into the S^T columns
      auto issue_s = [&](uint32_t sQ) {
        const uint64_t kK = opaque(sdesc_sw128(sK, 16, 1024));
        const uint64_t kQ = opaque(sdesc_sw128(sQ, 16, 1024));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::CHUNK + (kk % 4) * 32;
          mma_f16_ss(tmem + C::S_COL, sdesc_add(kK, off), sdesc_add(kQ, off), idSP,
                     kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.s_full);
      };
      // dP^T(i) = V_j dO_i^T into the dP^T columns
      auto issue_dp = [&](uint32_t sDO) {
        const uint64_t kV = opaque(sdesc_sw128(sV, 16, 1024));
        const uint64_t kDO = opaque(sdesc_sw128(sDO, 16, 1024));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::CHUNK + (kk % 4) * 32;
          mma_f16_ss(tmem + C::DP_COL, sdesc_add(kV, off), sdesc_add(kDO, off), idSP,
                     kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.dp_full);
      };
      auto slot_q = [&](int n) { return smem_u32(smem + C::OFF_Q + (n % C::NQS) * C::TILE); };
      auto slot_do = [&](int n) { return smem_u32(smem + C::OFF_DO + (n % C::NDS) * C::TILE); };
      auto wait_q = [&](int n) {
        return mbar_wait(&bars.q_full[n % C::NQS], (n / C::NQS) & 1, ab, kDevTimeoutMma);
      };
      auto wait_do = [&](int n) {
        return mbar_wait(&bars.do_full[n % C::NDS], (n / C::NDS) & 1, ab, kDevTimeoutMma);
      };
      // Issue order per step n (each MMA waits only for what it reads):
      //   dP^T(n) [dO_n loaded; at d = 128 after dQ(n-1) was read out of the
      //   shared columns]   dV(n) [P^T(n) ready]   S^T(n+1) [Q_{n+1} loaded]
      //   dK(n) [dS(n) ready]   dQ(n)
      // dP^T(n) needs nothing from step n's softmax, so it runs while the compute
      // warpgroups form P^T(n), and their dS phase starts as soon as P^T(n) is
      // written; the P phase of step n+1 overlaps dK(n), dQ(n).
      bool ok = mbar_wait(&bars.kv_full, 0, ab, kDevTimeoutMma) && wait_q(0);
      if (ok) {
        tc_fence_after_sync();
        issue_s(slot_q(0));
      }
      for (int n = 0; n < nsteps && ok; ++n) {
        const uint32_t sQ = slot_q(n);
        const uint32_t sDO = slot_do(n);
        // dP^T(n); its completion also means dQ(n-1) has finished reading the
        // dS^T buffer, which the dS phase of step n overwrites
        if (C::DQ_IN_DP && n > 0) {
          if (!(ok = mbar_wait(&bars.dq_free, (n - 1) & 1, ab, kDevTimeoutMma))) break;
        }
        if (!(ok = wait_do(n))) break;
        tc_fence_after_sync();
        issue_dp(sDO);
        // dV += P^T dO_i  (A = P^T from tensor memory); dO_i is free after it
        if (!(ok = mbar_wait(&bars.p_ready, n & 1, ab, kDevTimeoutMma))) break;
        tc_fence_after_sync();
        const uint64_t mDO = opaque(sdesc_sw128(sDO, C::CHUNK, 1024));
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          mma_f16_ts(tmem + C::DV_COL, tmem + C::S_COL + C::half_col(kk), sdesc_add(mDO, kk * 16 * 128),
                     idKV, (n > 0 || kk > 0) ? 1u : 0u);
        if (n + C::NDS < nsteps) mma_commit(&bars.do_empty[n % C::NDS]);
        // S^T of the next step (its columns now only hold P^T(n), read by dV above)
        if (n + 1 < nsteps) {
          if (!(ok = wait_q(n + 1))) break;
          tc_fence_after_sync();
          issue_s(slot_q(n + 1));
        }
        // dK += dS^T Q_i  (A = dS^T from tensor memory); the Q slot is free after it
        if (!(ok = mbar_wait(&bars.ds_ready, n & 1, ab, kDevTimeoutMma))) break;
        tc_fence_after_sync();
        const uint64_t mQ = opaque(sdesc_sw128(sQ, C::CHUNK, 1024));
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          mma_f16_ts(tmem + C::DK_COL, tmem + C::DP_COL + C::half_col(kk), sdesc_add(mQ, kk * 16 * 128),
                     idKV, (n > 0 || kk > 0) ? 1u : 0u);
        if (n + C::NQS < nsteps) mma_commit(&bars.q_empty[n % C::NQS]);
        // dQ_i = dS K_j into its columns (at d = 64 once dQ(n-1) was read out)
        if (!C::DQ_IN_DP && n > 0) {
          if (!(ok = mbar_wait(&bars.dq_free, (n - 1) & 1, ab, kDevTimeoutMma))) break;
          tc_fence_after_sync();
        }
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          mma_f16_ss(tmem + C::DQ_COL, sdesc_add(mDS, kk * 16 * 128), sdesc_add(mK, kk * 16 * 128),
                     idQ, kk > 0 ? 1u : 0u);
        mma_commit(&bars.dq_full);
      }
      if (ok) mma_commit(&bars.dkv_full);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute WGs
    const int h = warp >> 2;                         // query half: columns [64 h, 64 h + 64)
    const int quarter = warp & 3;
    const int k = quarter * 32 + lane;               // key row of the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int key_g = j * C::BN + k;
    const bool key_ok = key_g < N;
    const float c2 = kp.scale_log2;
    const uint32_t sDSrow = smem_u32(smem + C::OFF_DS) + h * C::CHUNK + k * 128;
    bool ok = true;
    int i = i0;                                      // query tile of step n
    for (int n = 0; n < nsteps; ++n, i = (i + 1 == nQ) ? i0 : i + 1) {
      const int st = n % C::NQS;
      const float4* nlse4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + st * 1024);  // -L log2 e
      const float4* ndvec4 = nlse4 + 32;                                                  // -D
      const bool diag = CAUSAL && i == j;
      // phase A: P^T = exp2(S^T c - L log2 e), written back as 16-bit
      if (!(ok = mbar_wait(&bars.s_full, n & 1, ab, kDevTimeoutSoftmax))) break;
      tc_fence_after_sync();
      uint32_t pb[32];                               // this half's P^T, packed pairs
      const uint64_t cc = pack2(c2, c2);
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {               // queries [64 h + 32 c2, +32): one load, one wait
        uint32_t svv[32];
        tmem_ld32(tmem + lane_addr + C::S_COL + 64 * h + 32 * c2, svv);
        tmem_ld_wait();
#pragma unroll
      for (int c = 2 * c2; c < 2 * c2 + 2; ++c) {    // queries [64 h + 16 c, +16)
        const int qb = 64 * h + 16 * c;
        const uint32_t* sv = svv + 16 * (c - 2 * c2);
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const int q0 = qb + e;
          const float4 l4 = nlse4[q0 / 4];
          const uint64_t y0 = ffma2(pack2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), cc,
                                    pack2(l4.x, l4.y));
          const uint64_t y1 = ffma2(pack2(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])), cc,
                                    pack2(l4.z, l4.w));
          float p[4] = {ex2_approx(lo2(y0)), ex2_approx(hi2(y0)), ex2_approx(lo2(y1)), ex2_approx(hi2(y1))};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (diag && k > q0 + u) p[u] = 0.f;
            if (!key_ok) p[u] = 0.f;
          }
          pb[(16 * c + e) / 2] = FP16 ? cvt_pack_f16(p[0], p[1]) : cvt_pack_bf16(p[0], p[1]);
          pb[(16 * c + e) / 2 + 1] = FP16 ? cvt_pack_f16(p[2], p[3]) : cvt_pack_bf16(p[2], p[3]);
        }
        // packed P^T of queries [qb, qb + 16) -> columns [64 h + 8 c, +8)
        tmem_st_x8(tmem + lane_addr + C::S_COL + 64 * h + 8 * c,
                   *reinterpret_cast<const uint32_t(*)[8]>(&pb[8 * c]));
      }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars.p_ready);
      // phase B: dS^T = P^T (dP^T - D), from the 16-bit P^T kept in registers,
      // into tensor memory (for dK) and the shared dS^T buffer (for dQ).  dP^T(n)
      // is issued after dQ(n-1), so its completion also means dQ(n-1) has
      // finished reading the buffer this phase overwrites
      if (!(ok = mbar_wait(&bars.dp_full, n & 1, ab, kDevTimeoutSoftmax))) break;
      tc_fence_after_sync();
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {               // queries [64 h + 32 c2, +32): one load, one wait
        uint32_t dpvv[32];
        tmem_ld32(tmem + lane_addr + C::DP_COL + 64 * h + 32 * c2, dpvv);
        tmem_ld_wait();
#pragma unroll
      for (int c = 2 * c2; c < 2 * c2 + 2; ++c) {    // queries [64 h + 16 c, +16)
        const int qb = 64 * h + 16 * c;
        const uint32_t* dpv = dpvv + 16 * (c - 2 * c2);
        uint32_t dd[8];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const int q0 = qb + e;
          const float4 d4 = ndvec4[q0 / 4];
          // unpack here, not earlier: keeps packed registers live instead of floats
          const uint32_t pw0 = opaque32(pb[(16 * c + e) / 2]);
          const uint32_t pw1 = opaque32(pb[(16 * c + e) / 2 + 1]);
          uint64_t pa, pc;
          if (FP16) {
            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&pw0));
            const float2 fc = __half22float2(*reinterpret_cast<const __half2*>(&pw1));
            pa = pack2(fa.x, fa.y);
            pc = pack2(fc.x, fc.y);
          } else {
            // a bf16 value is the upper half of the float32 with the same bits
            pa = pack2(__uint_as_float(pw0 << 16), __uint_as_float(pw0 & 0xffff0000u));
            pc = pack2(__uint_as_float(pw1 << 16), __uint_as_float(pw1 & 0xffff0000u));
          }
          const uint64_t dsa = fmul2(pa, fadd2(pack2(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])),
                                               pack2(d4.x, d4.y)));
          const uint64_t dsc = fmul2(pc, fadd2(pack2(__uint_as_float(dpv[e + 2]), __uint_as_float(dpv[e + 3])),
                                               pack2(d4.z, d4.w)));
          dd[e / 2] = FP16 ? cvt_pack_f16(lo2(dsa), hi2(dsa)) : cvt_pack_bf16(lo2(dsa), hi2(dsa));
          dd[e / 2 + 1] = FP16 ? cvt_pack_f16(lo2(dsc), hi2(dsc)) : cvt_pack_bf16(lo2(dsc), hi2(dsc));
        }
        tmem_st_x8(tmem + lane_addr + C::DP_COL + 64 * h + 8 * c, dd);
        // dS^T row k, queries [qb, qb + 16) = 16-byte pieces 2c and 2c + 1 of
        // chunk h, placed with the 128-byte swizzle
#pragma unroll
        for (int pc = 0; pc < 2; ++pc) {
          const uint32_t piece = static_cast<uint32_t>(2 * c + pc);
          st_shared_v4(sDSrow + ((piece ^ (k & 7)) * 16), dd[4 * pc], dd[4 * pc + 1],
                       dd[4 * pc + 2], dd[4 * pc + 3]);
        }
      }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&bars.ds_ready);
    }
    // ------------------------------------------------------------ epilogue
    // half 0 stores dV, half 1 stores dK (scaled by softmax_scale)
    if (ok && mbar_wait(&bars.dkv_full, 0, ab, kDevTimeoutEpilogue)) {
      tc_fence_after_sync();
      const uint32_t col = h ? C::DK_COL : C::DV_COL;
      const float mul = h ? kp.scale : 1.f;
      // [B, H_kv, N, d], or [total, H_kv, d] for a packed batch
      const size_t krow = PACKED ? static_cast<size_t>(seq0 + key_g) * kp.H_kv + hk
                                 : static_cast<size_t>(bhk) * N + key_g;
      uint16_t* dst_row = static_cast<uint16_t*>(h ? kp.dk : kp.dv) + krow * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_addr + col + c0 * 32, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float a = __uint_as_float(v[2 * e]) * mul;
          const float b = __uint_as_float(v[2 * e + 1]) * mul;
          pk[e] = FP16 ? cvt_pack_f16(a, b) : cvt_pack_bf16(a, b);
        }
        if (key_ok) {
          uint4* dst = reinterpret_cast<uint4*>(dst_row + c0 * 32);
#pragma unroll
          for (int x = 0; x < 4; ++x)
            dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ reduce WGs
    // TMEM lane = query row of the tile; reduce warpgroup g takes dQ columns
    // [g HC, g HC + HC).  Each warp copies its 32 rows x HC columns out of
    // tensor memory, hands the columns back, then moves them 32 columns at a
    // time through its 4 KB staging box (128-byte swizzle: row r's 16-byte piece
    // c sits at piece c ^ (r % 8)) and adds the box into the float32
    // accumulator with a TMA reduce-add, which skips rows outside the tensor.
    const int g = (warp - 8) >> 2;
    const int quarter = warp & 3;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr int HC = D / 2;                        // columns per reduce warpgroup
    uint8_t* const stg = smem + C::OFF_STG + (warp - 8) * C::STG_BOX;
    const uint32_t stg_row = smem_u32(stg) + lane * 128;
    int i = i0, hq = h0;                             // query tile and head of step n
    bool pending = false;                            // a reduce from `stg` may be reading it
    for (int n = 0; n < nsteps; ++n, (++i == nQ) ? (i = i0, ++hq) : 0) {
      if (!mbar_wait(&bars.dq_full, n & 1, ab, kDevTimeoutReduce)) break;
      tc_fence_after_sync();
      uint32_t v[HC];
#pragma unroll
      for (int c0 = 0; c0 < HC / 32; ++c0)
        tmem_ld32(tmem + lane_addr + C::DQ_COL + g * HC + c0 * 32,
                  *reinterpret_cast<uint32_t(*)[32]>(&v[c0 * 32]));
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars.dq_free);
      const int row0 = i * C::BM + quarter * 32;     // first query row of this warp's box
#pragma unroll
      for (int bx = 0; bx < HC / 32; ++bx) {
        if (pending) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
        }
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(stg_row + ((c ^ (lane & 7)) * 16), v[32 * bx + 4 * c], v[32 * bx + 4 * c + 1],
                       v[32 * bx + 4 * c + 2], v[32 * bx + 4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int col = g * HC + 32 * bx;
          if constexpr (PACKED)
            tma_reduce_add_4d(&tmDQ, stg, col, seq0 + row0, hq, 0);
          else
            tma_reduce_add_3d(&tmDQ, stg, col, row0, b * kp.H + hq);
          bulk_commit_group();
        }
        pending = true;
      }
    }
    // every reduce this warp issued has finished before the CTA ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (bars.abort_flag) {
    if (warp == C::LOAD_WARP && lane == 0) {
      mbar_wait_drain(&bars.kv_full, 0);
      const int nq = bars.q_items;
      for (int s = 0; s < C::NQS && s < nq; ++s)
        mbar_wait_drain(&bars.q_full[s], ((nq - 1 - s) / C::NQS) & 1);
      const int nd = bars.do_items;
      for (int s = 0; s < C::NDS && s < nd; ++s)
        mbar_wait_drain(&bars.do_full[s], ((nd - 1 - s) / C::NDS) & 1);
    }
    if (warp == C::MMA_WARP && lane == 0) {
      mma_commit(&bars.drain);
      mbar_wait_drain(&bars.drain, 0);
    }
    __syncthreads();
  }
  if (warp == C::MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool FP16, bool PACKED>
attn_status_t launch_bwd_t(const BwdParams& p, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const int Npad = (p.N + 127) / 128 * 128;
  const long long rows_pad = static_cast<long long>(p.B) * p.H * Npad;
  // 1. prep
  {
    constexpr int rows_per_block = 8 * (32 / (D / 8));
    const long long blocks = (rows_pad + rows_per_block - 1) / rows_per_block;
    bwd_prep_kernel<D, FP16, PACKED><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(p.o), static_cast<const uint16_t*>(p.dout), p.lse, p.lse2,
        p.delta, p.dq_acc, p.N, Npad, rows_pad, p.H, p.cu_seqlens, p.total);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e, "backward prep launch");
  }
  // 2. main
  {
    auto kern = bwd_main_kernel<D, CAUSAL, FP16, PACKED>;
    attn_status_t s = set_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
    if (s != ATTN_OK) return s;
    CUtensorMap tq, tk, tv, tdo, tdq;
    if constexpr (PACKED) {
      // {d, total tokens, heads, 1}: token stride heads * d, head stride d
      const uint64_t T = static_cast<uint64_t>(p.total);
      const uint64_t qr = 2ull * p.H * D, kvr = 2ull * p.H_kv * D;
      if ((s = make_tmap_4d(&tq, p.q, 2, D, T, p.H, 1, qr, 2ull * D, T * qr, 64, 128)) != ATTN_OK) return s;
      if ((s = make_tmap_4d(&tdo, p.dout, 2, D, T, p.H, 1, qr, 2ull * D, T * qr, 64, 128)) != ATTN_OK)
        return s;
      if ((s = make_tmap_4d(&tk, p.k, 2, D, T, p.H_kv, 1, kvr, 2ull * D, T * kvr, 64, 128)) != ATTN_OK)
        return s;
      if ((s = make_tmap_4d(&tv, p.v, 2, D, T, p.H_kv, 1, kvr, 2ull * D, T * kvr, 64, 128)) != ATTN_OK)
        return s;
      // float32 dQ accumulator [total, H, d]: reduce boxes of 32 rows x 32 columns
      const uint64_t ar = 4ull * p.H * D;
      if ((s = make_tmap_4d(&tdq, p.dq_acc, 4, D, T, p.H, 1, ar, 4ull * D, T * ar, 32, 32)) != ATTN_OK)
        return s;
    } else {
      // {d, N, B * heads}
      const uint64_t pq = static_cast<uint64_t>(p.B) * p.H, pkv = static_cast<uint64_t>(p.B) * p.H_kv;
      if ((s = make_tmap_3d(&tq, p.q, 2, D, p.N, pq, 64, 128)) != ATTN_OK) return s;
      if ((s = make_tmap_3d(&tdo, p.dout, 2, D, p.N, pq, 64, 128)) != ATTN_OK) return s;
      if ((s = make_tmap_3d(&tk, p.k, 2, D, p.N, pkv, 64, 128)) != ATTN_OK) return s;
      if ((s = make_tmap_3d(&tv, p.v, 2, D, p.N, pkv, 64, 128)) != ATTN_OK) return s;
      // float32 dQ accumulator [B * H, N, d]: reduce boxes of 32 rows x 32 columns
      if ((s = make_tmap_3d(&tdq, p.dq_acc, 4, D, p.N, pq, 32, 32)) != ATTN_OK) return s;
    }
    int* status = device_status_word();
    if (!status) return fail(ATTN_ERR_CUDA, "status word unavailable");
    BwdKParams kp{p.dk,  p.dv,    p.dq_acc, p.lse2, p.delta, status,        p.cu_seqlens,
                  p.N,   Npad,    p.total,  p.H,    p.H_kv,  p.H / p.H_kv,  p.scale,
                  p.scale * kLog2e};
    const unsigned ntiles = static_cast<unsigned>((p.N + 127) / 128);
    const dim3 grid = CAUSAL ? dim3(ntiles * p.H_kv * p.B, 1, 1) : dim3(ntiles, p.H_kv, p.B);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, tdq, kp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e, "backward main launch");
  }
  // 3. convert
  {
    const long long elems = PACKED ? static_cast<long long>(p.total) * p.H * D
                                   : static_cast<long long>(p.B) * p.H * p.N * D;
    const long long n8 = elems / 8;
    const long long want = (n8 + 255) / 256;
    const unsigned blocks = static_cast<unsigned>(want < 152 * 16 ? want : 152 * 16);
    bwd_convert_kernel<FP16><<<blocks, 256, 0, stream>>>(p.dq_acc, static_cast<uint16_t*>(p.dq),
                                                         p.scale, n8);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e, "backward convert launch");
  }
  return ATTN_OK;
}

template <int D, bool PACKED>
attn_status_t launch_bwd_dp(const BwdParams& p, cudaStream_t stream) {
  if (p.causal)
    return p.fp16 ? launch_bwd_t<D, true, true, PACKED>(p, stream)
                  : launch_bwd_t<D, true, false, PACKED>(p, stream);
  return p.fp16 ? launch_bwd_t<D, false, true, PACKED>(p, stream)
                : launch_bwd_t<D, false, false, PACKED>(p, stream);
}

template <int D>
attn_status_t launch_bwd_d(const BwdParams& p, cudaStream_t stream) {
  return p.cu_seqlens ? launch_bwd_dp<D, true>(p, stream) : launch_bwd_dp<D, false>(p, stream);
}

}  // namespace

attn_status_t launch_bwd(const BwdParams& p, cudaStream_t stream) {
  if (p.N > 65535 * 128 || p.H > 65535 || p.B > 65535 ||
      static_cast<long long>((p.N + 127) / 128) * p.H_kv * p.B > 2147483647LL)
    return fail(ATTN_ERR_UNSUPPORTED, "grid dimension limit exceeded");
  switch (p.d) {
    case 64: return launch_bwd_d<64>(p, stream);
    case 128: return launch_bwd_d<128>(p, stream);
  }
  return fail(ATTN_ERR_UNSUPPORTED, "the backward pass supports d = 64 and 128");
}

}  // namespace attn
