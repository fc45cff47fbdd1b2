// BF16/FP16 attention forward on sm_103a.
//
// Method: "FlashAttention-3: Hopper Asynchrony and FP8 Attention" -- the query
// tile stays on chip while key/value tiles stream through a ring of
// shared-memory stages ("Producer-consumer asynchrony"), the running row max
// m and sum l are updated per tile and the output numerator is rescaled when
// m grows ("Symbol Map"; "Putting It Together", steps 4-5), and the epilogue
// divides by l and stores L = m + log(l) ("Putting It Together", step 7).
//
// GB300 design (not the page's Hopper design):
//  * One CTA owns NQ query tiles of 128 rows (NQ = 2 for d <= 128, 1 for
//    d = 256).  Scores S_t and output accumulators O_t live in tensor memory
//    (TMEM); the probabilities P_t are written back over S_t as 16-bit values
//    and fed to the P V product straight from TMEM.  At d = 256 the query tile
//    sits in TMEM too (the A operand of S), which leaves shared memory for a
//    third K/V stage.
//  * Warp roles: one TMA producer warp, one MMA warp whose elected thread
//    issues every tcgen05.mma, and two softmax warpgroups per query tile: a
//    warp owns 32 rows (one TMEM lane quarter) and one half of the key
//    columns, so each row is split across two warps that swap partial maxima
//    once per step and add their row-sum shares at the end.  The MMA thread
//    alternates between the tiles, so while one tile's softmax runs its
//    exponentials the tensor core works on the other tile -- the same overlap
//    the page's "Ping-pong scheduling" gets from two Hopper warpgroups.
//  * Rescaling is lazy: the exponent reference m_ref moves only when the row
//    max exceeds it by more than 8 (log2 units), so P <= 2^8 and most tiles
//    skip the TMEM read-modify-write of O.  In exact arithmetic the result is
//    the same as rescaling on every tile.
//  * Causal: query tile i visits key tiles 0..i only and masks the diagonal
//    tile; CTAs are launched longest-first.
#include <cmath>

#include "common.h"
#include "sm103_prims.cuh"

namespace attn {
namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // keys per tile
constexpr int kSmemLimit = 232448;

// Schedule variants of the forward kernel, kept for measurement (the pages'
// pipeline ablation): the default alternates two query tiles per CTA and
// rescales lazily.
enum : int {
  kSchedOneTile = 1,   // one query tile per CTA: no second tile to fill the softmax window
  kSchedEager = 2,     // rescale O whenever the row max grows (no 2^8 slack)
};

template <int D, int NQ_ = (D <= 128) ? 2 : 1>
struct FwdCfg {
  static constexpr int NQ = NQ_;
  static constexpr int CH = D / 64;                  // 128-byte column chunks per row
  static constexpr int CHUNK_BYTES = BM * 128;       // one 128-row x 128-byte chunk
  static constexpr int TILE_BYTES = BM * D * 2;      // a Q, K or V tile
  // row-statistics exchange between the two warps of a row (static shared memory)
  static constexpr int XCH_BYTES = 2 * NQ * 2 * 128 * 4;
  // d = 256: S (128 columns) and O (256) leave 128 TMEM columns, enough for the
  // query tile (128 rows x 256 bf16) as the A operand of S.  Q then needs no
  // shared memory of its own (it is staged once through the last ring stage),
  // and the ring gets a third 64 KB stage.
  static constexpr bool Q_IN_TMEM = (D == 256 && NQ == 1);
  static constexpr uint32_t Q_COL = 128;
  static constexpr int Q_SMEM = Q_IN_TMEM ? 0 : NQ * TILE_BYTES;
  static constexpr int NSLOT_FIT = (kSmemLimit - 2048 - XCH_BYTES - Q_SMEM) / TILE_BYTES;
  static constexpr int NSLOT = NSLOT_FIT > 6 ? 6 : NSLOT_FIT;
  static constexpr int SMEM_BYTES = 1024 + Q_SMEM + NSLOT * TILE_BYTES;
  // Two softmax warpgroups per query tile: each row of S is split between two
  // warps (key columns [0, 64) and [64, 128)).
  static constexpr int NUM_SOFTMAX_WARPS = 8 * NQ;
  static constexpr int LOAD_WARP = NUM_SOFTMAX_WARPS;
  static constexpr int MMA_WARP = NUM_SOFTMAX_WARPS + 1;
  static constexpr int THREADS = (NUM_SOFTMAX_WARPS + 2) * 32;
  __host__ __device__ static constexpr uint32_t S_COL(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t O_COL(int t) { return 256u + static_cast<uint32_t>(D) * t; }
  // TMEM column of the packed 16-bit P for keys [16 kk, 16 kk + 16): each half
  // of the row writes its P inside its own score columns
  __host__ __device__ static constexpr uint32_t P_COL(int kk) {
    return 64u * static_cast<uint32_t>(kk / 4) + 8u * static_cast<uint32_t>(kk % 4);
  }
  // With a ring of two stages (d = 256: 64 KB tiles) the next K or V tile can
  // load only into the stage just read, so the MMA thread hands each stage back
  // by a commit right after the products that read it; with deeper rings the
  // softmax does it when it sees S(j) complete, which keeps commits off the
  // MMA thread.
  static constexpr bool COMMIT_RELEASE = (TILE_BYTES >= 65536);
  static_assert(NSLOT >= 2, "need at least two ring stages");
  static_assert(!Q_IN_TMEM || (S_COL(0) + 128 <= Q_COL && Q_COL + D / 2 <= O_COL(0)), "TMEM overflow (Q)");
  static_assert(O_COL(NQ - 1) + D <= 512, "TMEM overflow");
  static_assert(S_COL(NQ - 1) + 128 <= 256, "S region overflow");
};

struct FwdKParams {
  void* o;
  float* lse;
  int* status;
  const int* cu_seqlens;   // packed batch: sequence b is tokens [cu[b], cu[b+1]); else nullptr
  int N;                   // sequence length, or the longest sequence (sizes the grid)
  int total;               // tokens of a packed batch
  int H;
  int group;               // query heads per key/value head
  float scale_log2;   // softmax_scale * log2(e)
};

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// PACKED: a batch of sequences packed back to back ([total, H, d], LSE
// [H, total], offsets cu_seqlens); otherwise [B, H, N, d] and LSE [B, H, N].
// SCHED: 0, or kSchedOneTile / kSchedEager (measurement variants).
template <int D, bool CAUSAL, bool FP16, bool PACKED, int SCHED = 0,
          int NQ_ = ((SCHED & kSchedOneTile) || D > 128) ? 1 : 2>
__global__ void __launch_bounds__(FwdCfg<D, NQ_>::THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdKParams kp) {
  using C = FwdCfg<D, NQ_>;
  constexpr int NQ = C::NQ;
  constexpr int NSLOT = C::NSLOT;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sKV = smem + C::Q_SMEM;
  // Q tiles: their own region, or (Q in tensor memory) staged in the last ring stage
  uint8_t* sQ = C::Q_IN_TMEM ? sKV + (NSLOT - 1) * C::TILE_BYTES : smem;

  __shared__ __align__(8) uint64_t q_full[NQ];
  __shared__ __align__(8) uint64_t kv_full[NSLOT];
  __shared__ __align__(8) uint64_t kv_empty[NSLOT];
  __shared__ __align__(8) uint64_t s_full[NQ];
  __shared__ __align__(8) uint64_t p_full[NQ];
  __shared__ __align__(8) uint64_t o_full[NQ];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t q_moved;   // Q in tensor memory: its staging stage is free
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int load_items_sh;
  __shared__ float xch[2][NQ][2][128];   // [step parity][tile][half][row]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // Causal: a 1-D grid ordered by work, heaviest query-tile groups (largest
  // g, which visit the most key tiles) of every head first, so the last wave
  // holds the short ones.  Non-causal: (group, head, batch) keeps a head's
  // CTAs together for K/V reuse in L2.
  const int npairs = (kp.N + BM * NQ - 1) / (BM * NQ);
  const int g = CAUSAL ? npairs - 1 - static_cast<int>(blockIdx.x / (gridDim.x / npairs))
                       : static_cast<int>(blockIdx.x);
  const int bh = CAUSAL ? static_cast<int>(blockIdx.x % (gridDim.x / npairs))
                        : static_cast<int>(blockIdx.z * kp.H + blockIdx.y);
  // A packed batch: this sequence's first token and length; tiles past its end
  // have nothing to do (the whole CTA leaves before touching any resource).
  int seq0 = 0, N = kp.N;
  if constexpr (PACKED) {
    const int b = bh / kp.H;
    seq0 = kp.cu_seqlens[b];
    const int end = kp.cu_seqlens[b + 1];
    if (seq0 < 0 || end < seq0 || end > kp.total || end - seq0 > kp.N) {
      if (threadIdx.x == 0) atomicCAS(kp.status, 0, kDevBadSeqlens);
      return;
    }
    N = end - seq0;
    if (g * NQ * BM >= N) return;
  }
  const int nKtot = (N + BN - 1) / BN;

  int nK[NQ];
  int nKmax = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int qt = g * NQ + t;
    nK[t] = (qt * BM < N) ? (CAUSAL ? min(nKtot, qt + 1) : nKtot) : 0;
    nKmax = max(nKmax, nK[t]);
  }
  const int total_items = 2 * nKmax;   // K_0, V_0, K_1, V_1, ...
  // The last query tile with work runs every key tile; when its S(j) completes,
  // all MMAs reading K_j and V_{j-1} (of every tile) have completed, so its
  // softmax warpgroup hands those ring slots back to the producer.
  const int t_rel = (nK[NQ - 1] == nKmax) ? NQ - 1 : 0;

  if (threadIdx.x == 0) {
    for (int t = 0; t < NQ; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 256);
      mbar_init(&o_full[t], 1);
    }
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&drain_bar, 1);
    mbar_init(&q_moved, 32 * C::NUM_SOFTMAX_WARPS);
    abort_sh = 0;
    load_items_sh = 0;
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const Abort ab{&abort_sh, kp.status};

  if (warp == C::LOAD_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      // Tensor-map coordinates: {c, row, plane} with plane = b * heads + head
      // for [B, heads, N, d]; {c, token, head, 0} for a packed batch.
      const int b = bh / kp.H;
      const int hq = bh - b * kp.H;            // query head
      const int hkv = hq / kp.group;           // its key/value head
      const int kv_plane = b * (kp.H / kp.group) + hkv;
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        if (nK[t] == 0) continue;
        mbar_arrive_expect_tx(&q_full[t], C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          if constexpr (PACKED)
            tma_load_4d(sQ + t * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ, &q_full[t], c * 64,
                        seq0 + (g * NQ + t) * BM, hq, 0);
          else
            tma_load_3d(sQ + t * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ, &q_full[t], c * 64,
                        (g * NQ + t) * BM, bh);
      }
      int it = 0;
      bool ok = true;
      for (int j = 0; j < nKmax && ok; ++j) {
        for (int kv = 0; kv < 2; ++kv) {
          const int slot = it % NSLOT;
          const int use = it / NSLOT;
          if (use >= 1 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, ab, kDevTimeoutLoad)) {
            ok = false;
            break;
          }
          // the last stage holds Q until the softmax warps have copied it to tensor memory
          if (C::Q_IN_TMEM && it == NSLOT - 1 && !mbar_wait(&q_moved, 0, ab, kDevTimeoutLoad)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&kv_full[slot], C::TILE_BYTES);
          uint8_t* dst = sKV + slot * C::TILE_BYTES;
#pragma unroll
          for (int c = 0; c < C::CH; ++c)
            if constexpr (PACKED)
              tma_load_4d(dst + c * C::CHUNK_BYTES, kv ? &tmV : &tmK, &kv_full[slot], c * 64,
                          seq0 + j * BN, hkv, 0);
            else
              tma_load_3d(dst + c * C::CHUNK_BYTES, kv ? &tmV : &tmK, &kv_full[slot], c * 64,
                          j * BN, kv_plane);
          ++it;
        }
      }
      load_items_sh = it;
    }
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr Elt E = FP16 ? Elt::F16 : Elt::BF16;
      constexpr uint32_t idS = idesc_f16(E, 128, BN, false, false);
      constexpr uint32_t idPV = idesc_f16(E, 128, D, false, true);
      const uint64_t qdesc0 = sdesc_sw128(smem_u32(sQ), 16, 1024);            // K-major Q
      const uint64_t kvdesc0 = sdesc_sw128(smem_u32(sKV), 16, 1024);          // K-major K
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(sKV), C::CHUNK_BYTES, 1024);  // MN-major V
      bool ok = true;
#pragma unroll
      for (int t = 0; t < NQ; ++t)
        if (ok && nK[t] > 0)
          ok = C::Q_IN_TMEM ? mbar_wait(&q_moved, 0, ab, kDevTimeoutMma) : mbar_wait(&q_full[t], 0, ab, kDevTimeoutMma);
      for (int j = 0; j <= nKmax && ok; ++j) {
        const int itK = 2 * j;          // ring item of K_j
        const int itV = 2 * j - 1;      // ring item of V_{j-1}
        const int slotK = itK % NSLOT;
        const int slotV = (itV + NSLOT) % NSLOT;
        bool haveK = false, haveV = false;
        uint64_t kdesc = 0, vdesc = 0;
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (j >= 1 && j - 1 < nK[t]) {
            // O_t += P_t(j-1) V_{j-1}
            if (!haveV) {
              if (!(ok = mbar_wait(&kv_full[slotV], (itV / NSLOT) & 1, ab, kDevTimeoutMma))) break;
              vdesc = opaque(sdesc_add(vdesc0, slotV * C::TILE_BYTES));
              haveV = true;
            }
            if (!(ok = mbar_wait(&p_full[t], (j - 1) & 1, ab, kDevTimeoutMma))) break;
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_f16_ts(tmem + C::O_COL(t), tmem + C::S_COL(t) + C::P_COL(kk),
                         sdesc_add(vdesc, kk * 16 * 128), idPV, (j - 1 > 0 || kk > 0) ? 1u : 0u);
            if (j - 1 == nK[t] - 1) mma_commit(&o_full[t]);
            if (C::COMMIT_RELEASE && t == t_rel && itV + NSLOT < total_items) mma_commit(&kv_empty[slotV]);
          }
          if (j < nK[t]) {
            // S_t(j) = Q_t K_j^T
            if (!haveK) {
              if (!(ok = mbar_wait(&kv_full[slotK], (itK / NSLOT) & 1, ab, kDevTimeoutMma))) break;
              tc_fence_after_sync();
              kdesc = opaque(sdesc_add(kvdesc0, slotK * C::TILE_BYTES));
              haveK = true;
            }
            const uint64_t qdesc = sdesc_add(qdesc0, t * C::TILE_BYTES);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32;
              if constexpr (C::Q_IN_TMEM)
                mma_f16_ts(tmem + C::S_COL(t), tmem + C::Q_COL + 8u * kk, sdesc_add(kdesc, off), idS,
                           kk > 0 ? 1u : 0u);
              else
                mma_f16_ss(tmem + C::S_COL(t), sdesc_add(qdesc, off), sdesc_add(kdesc, off), idS,
                           kk > 0 ? 1u : 0u);
            }
            mma_commit(&s_full[t]);
            if (C::COMMIT_RELEASE && t == t_rel && itK + NSLOT < total_items) mma_commit(&kv_empty[slotK]);
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
    const int qt = g * NQ + t;
    // key tiles of this warpgroup's query tile (a scalar: no runtime-indexed array)
    const int my_nK = (qt * BM < N) ? (CAUSAL ? min(nKtot, qt + 1) : nKtot) : 0;
    const int row_g = qt * BM + r;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::S_COL(t) + 64 * h;     // this half's scores
    const uint32_t tO = tmem + lane_addr + C::O_COL(t) + (D / 2) * h; // this half's O columns
    const float c2 = kp.scale_log2;
    float m_ref = -INFINITY;
    float l = 0.f;                       // this half's share of the row sum
    bool ok = true;
    if constexpr (C::Q_IN_TMEM) {
      // Copy this warp's half of its rows of Q (d in [128 h, 128 h + 128): chunks
      // 2h, 2h + 1 of the 128-byte-swizzled tile) into tensor memory, two bf16 per
      // column, then hand the staging stage back.  Every softmax thread arrives
      // at q_moved (the producer and the MMA thread wait on it).
      if (my_nK > 0) {
        if (__any_sync(0xffffffffu, !mbar_wait(&q_full[t], 0, ab, kDevTimeoutSoftmax))) {
          ok = false;
        } else {
          const uint8_t* qrow = sQ + t * C::TILE_BYTES + r * 128;
          const uint32_t tQ = tmem + lane_addr + C::Q_COL + (D / 4) * h;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const uint8_t* chunk = qrow + (2 * h + cc) * C::CHUNK_BYTES;
            uint32_t w[32];
#pragma unroll
            for (int pc = 0; pc < 8; ++pc) {
              const uint4 v = *reinterpret_cast<const uint4*>(chunk + ((pc ^ (r & 7)) * 16));
              w[4 * pc] = v.x;
              w[4 * pc + 1] = v.y;
              w[4 * pc + 2] = v.z;
              w[4 * pc + 3] = v.w;
            }
            tmem_st32(tQ + 32 * cc, w);
          }
          tmem_st_wait();
        }
      }
      fence_proxy_async_smem();   // the reads above come before the stage's next copy
      tc_fence_before_sync();
      mbar_arrive(&q_moved);
    }
    for (int j = 0; ok && j < my_nK; ++j) {
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
      if (!C::COMMIT_RELEASE && t == t_rel && h == 0 && r == 0) {
        // release only slots the producer refills
        if (2 * j + NSLOT < total_items) mbar_arrive(&kv_empty[(2 * j) % NSLOT]);
        if (j >= 1 && 2 * j - 1 + NSLOT < total_items) mbar_arrive(&kv_empty[(2 * j - 1) % NSLOT]);
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
      // this half's max as a tree of 3-input maxima, then the row max
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        mx[u] = fmax3(__uint_as_float(sr[8 * u]), __uint_as_float(sr[8 * u + 1]),
                      fmax3(__uint_as_float(sr[8 * u + 2]), __uint_as_float(sr[8 * u + 3]),
                            fmax3(__uint_as_float(sr[8 * u + 4]), __uint_as_float(sr[8 * u + 5]),
                                  fmaxf(__uint_as_float(sr[8 * u + 6]), __uint_as_float(sr[8 * u + 7])))));
      const float m_half = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                 fmaxf(mx[6], mx[7]));
      xch[j & 1][t][h][r] = m_half;
      named_bar_sync(pair_bar, 64);
      const float m_new = fmaxf(m_ref, fmaxf(m_half, xch[j & 1][t][h ^ 1][r]));
      // Move the exponent reference only when the max grew by more than 2^8
      // (both halves of a row take the same decision); the eager variant
      // moves it whenever the max grows.
      const bool need = (SCHED & kSchedEager) ? (m_new > m_ref) : (m_new - m_ref) * c2 > 8.f;
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx((m_ref - m_new) * c2);
        l *= alpha;
        m_ref = m_new;
      }
      const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref * c2;
      const uint64_t cc = pack2(c2, c2);
      const uint64_t nn = pack2(neg, neg);
      uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
      for (int c0 = 0; c0 < 2; ++c0) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = c0 * 32 + 2 * i;
          const uint64_t y = ffma2(pack2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), cc, nn);
          const float p0 = ex2_approx(lo2(y));
          const float p1 = ex2_approx(hi2(y));
          if (i & 1) acc1 = fadd2(acc1, pack2(p0, p1));
          else acc0 = fadd2(acc0, pack2(p0, p1));
          pk[i] = FP16 ? cvt_pack_f16(p0, p1) : cvt_pack_bf16(p0, p1);
        }
        // packed P of keys [64 h + 32 c0, +32) -> columns [64 h + 16 c0, +16)
        tmem_st16(tS + c0 * 16, pk);
      }
      const uint64_t acc = fadd2(acc0, acc1);
      l += lo2(acc) + hi2(acc);
      // Rescale this half's columns of O (the P V product of this step is
      // issued only after the arrive below; the previous one finished before
      // S_t(j) did).
      if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c0 = 0; c0 < D / 64; ++c0) {
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
    // ------------------------------------------------------------ epilogue
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
      const float inv_l = 1.f / l_row;
      // O row: [B, H, N, d], or [total, H, d] for a packed batch
      const size_t orow_off = PACKED ? (static_cast<size_t>(seq0 + row_g) * kp.H + bh % kp.H) * D
                                     : (static_cast<size_t>(bh) * N + row_g) * D;
      uint16_t* orow = static_cast<uint16_t*>(kp.o) + orow_off + (D / 2) * h;
#pragma unroll 1
      for (int c0 = 0; c0 < D / 64; ++c0) {
        uint32_t o[32];
        tmem_ld32(tO + c0 * 32, o);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float o0 = __uint_as_float(o[2 * i]) * inv_l;
          const float o1 = __uint_as_float(o[2 * i + 1]) * inv_l;
          pk[i] = FP16 ? cvt_pack_f16(o0, o1) : cvt_pack_bf16(o0, o1);
        }
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
            (m_ref * c2 + lg2_approx(l_row)) * 0.69314718055994530942f;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (abort_sh) {
    // Let every copy and MMA this CTA issued land before the memory goes away.
    if (warp == C::LOAD_WARP && lane == 0) {
#pragma unroll
      for (int t = 0; t < NQ; ++t)
        if (nK[t] > 0) mbar_wait_drain(&q_full[t], 0);
      const int issued = load_items_sh;
      for (int s = 0; s < NSLOT && s < issued; ++s)
        mbar_wait_drain(&kv_full[s], ((issued - 1 - s) / NSLOT) & 1);
    }
    if (warp == C::MMA_WARP && lane == 0) {
      mma_commit(&drain_bar);
      mbar_wait_drain(&drain_bar, 0);
    }
    __syncthreads();
  }
  if (warp == C::MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool FP16, bool PACKED, int SCHED = 0>
attn_status_t launch_fwd_t(const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<D, ((SCHED & kSchedOneTile) || D > 128) ? 1 : 2>;
  auto kern = fwd_kernel<D, CAUSAL, FP16, PACKED, SCHED>;
  attn_status_t s = set_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (s != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
  if constexpr (PACKED) {
    // {d, total tokens, heads, 1}: token stride heads * d, head stride d
    const uint64_t T = static_cast<uint64_t>(p.total);
    if ((s = make_tmap_4d(&tq, p.q, 2, D, T, p.H, 1, 2ull * p.H * D, 2ull * D, 2ull * T * p.H * D,
                          64, BM)) != ATTN_OK)
      return s;
    if ((s = make_tmap_4d(&tk, p.k, 2, D, T, p.H_kv, 1, 2ull * p.H_kv * D, 2ull * D,
                          2ull * T * p.H_kv * D, 64, BN)) != ATTN_OK)
      return s;
    if ((s = make_tmap_4d(&tv, p.v, 2, D, T, p.H_kv, 1, 2ull * p.H_kv * D, 2ull * D,
                          2ull * T * p.H_kv * D, 64, BN)) != ATTN_OK)
      return s;
  } else {
    // {d, N, B * heads}
    if ((s = make_tmap_3d(&tq, p.q, 2, D, p.N, static_cast<uint64_t>(p.B) * p.H, 64, BM)) != ATTN_OK)
      return s;
    if ((s = make_tmap_3d(&tk, p.k, 2, D, p.N, static_cast<uint64_t>(p.B) * p.H_kv, 64, BN)) != ATTN_OK)
      return s;
    if ((s = make_tmap_3d(&tv, p.v, 2, D, p.N, static_cast<uint64_t>(p.B) * p.H_kv, 64, BN)) != ATTN_OK)
      return s;
  }
  int* status = device_status_word();
  if (!status) return fail(ATTN_ERR_CUDA, "status word unavailable");
  FwdKParams kp{p.o,   p.lse, status, p.cu_seqlens,           p.N,
                p.total, p.H,  p.H / p.H_kv, p.scale * 1.4426950408889634f};
  const int rows_per_cta = BM * C::NQ;
  const unsigned npairs = static_cast<unsigned>((p.N + rows_per_cta - 1) / rows_per_cta);
  const dim3 grid = CAUSAL ? dim3(npairs * p.H * p.B, 1, 1) : dim3(npairs, p.H, p.B);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, kp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "forward kernel launch");
  return ATTN_OK;
}

template <int D, bool PACKED>
attn_status_t launch_fwd_dp(const FwdParams& p, cudaStream_t stream) {
  if (p.causal)
    return p.fp16 ? launch_fwd_t<D, true, true, PACKED>(p, stream)
                  : launch_fwd_t<D, true, false, PACKED>(p, stream);
  return p.fp16 ? launch_fwd_t<D, false, true, PACKED>(p, stream)
                : launch_fwd_t<D, false, false, PACKED>(p, stream);
}

template <int D>
attn_status_t launch_fwd_d(const FwdParams& p, cudaStream_t stream) {
  return p.cu_seqlens ? launch_fwd_dp<D, true>(p, stream) : launch_fwd_dp<D, false>(p, stream);
}

}  // namespace

attn_status_t launch_fwd(const FwdParams& p, cudaStream_t stream) {
  if (p.N > 65535 * 256 || p.H > 65535 || p.B > 65535 ||
      static_cast<long long>((p.N + 255) / 128) * p.H * p.B > 2147483647LL)
    return fail(ATTN_ERR_UNSUPPORTED, "grid dimension limit exceeded");
  // packed causal batches: the persistent kernel, which measured faster there
  if (p.cu_seqlens && p.causal) return launch_fwd_persistent(p, stream);
  switch (p.d) {
    case 64: return launch_fwd_d<64>(p, stream);
    case 128: return launch_fwd_d<128>(p, stream);
    case 256: return launch_fwd_d<256>(p, stream);
  }
  return fail(ATTN_ERR_INVALID_ARG, "d must be 64, 128 or 256");
}

// Measurement variants (bfloat16, fixed length, d = 64 or 128).
attn_status_t launch_fwd_sched(const FwdParams& p, int sched, cudaStream_t stream) {
  if (p.fp16 || p.cu_seqlens || p.H_kv != p.H || (p.d != 64 && p.d != 128))
    return fail(ATTN_ERR_UNSUPPORTED,
                "schedule variants: bfloat16, fixed length, H_kv = H, d = 64 or 128");
  if (p.N > 65535 * 128 || p.H > 65535 || p.B > 65535)
    return fail(ATTN_ERR_UNSUPPORTED, "grid dimension limit exceeded");
#define ATTN_SCHED_CASE(S)                                                                   \
  case S:                                                                                    \
    if (p.d == 64)                                                                           \
      return p.causal ? launch_fwd_t<64, true, false, false, S>(p, stream)                   \
                      : launch_fwd_t<64, false, false, false, S>(p, stream);                 \
    return p.causal ? launch_fwd_t<128, true, false, false, S>(p, stream)                    \
                    : launch_fwd_t<128, false, false, false, S>(p, stream);
  switch (sched) {
    ATTN_SCHED_CASE(0)
    ATTN_SCHED_CASE(kSchedOneTile)
    ATTN_SCHED_CASE(kSchedEager)
    ATTN_SCHED_CASE(kSchedOneTile | kSchedEager)
  }
#undef ATTN_SCHED_CASE
  return fail(ATTN_ERR_INVALID_ARG, "schedule must be a combination of ATTN_SCHED_ONE_TILE and ATTN_SCHED_EAGER_RESCALE");
}

}  // namespace attn
