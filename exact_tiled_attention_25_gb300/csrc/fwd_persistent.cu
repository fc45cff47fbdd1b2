// Persistent BF16/FP16 attention forward on sm_103a for packed causal batches.
//
// Method: the forward of "FlashAttention-3: Hopper Asynchrony and FP8 Attention"
// (online softmax over streamed key/value tiles, "Symbol Map" and "Putting It
// Together"), scheduled as "FlashAttention 3 Hardware Acceleration: Hopper GPU
// Strategies for Long-Context Enterprise Inference Optimization" describes for
// Blackwell: section "Tile Scheduler" (tiles assigned to CTAs, only the valid
// causal tiles processed) and section "Blackwell Architecture" (cluster launch
// control hands out work as SMs free up, balancing variable sequence lengths).
//
// The per-tile schedule (warp roles, TMEM layout, split softmax, lazy rescale)
// is the one of fwd.cu.  What differs: a CTA that finishes its tile takes over
// the tile of a CTA not yet launched (clusterlaunchcontrol.try_cancel), so the
// next tile's Q loads and first MMAs overlap the current tile's last softmax
// steps and epilogue.  A 4-entry ring of tile indices, filled by the producer,
// feeds the other roles; Q-empty and O-empty barriers let the next tile start
// while the current one drains; phase counters run across tiles.
//
// Measured on GB300 against fwd.cu (same tests pass on both): faster on packed
// causal batches, where sequences of mixed length leave CTAs with very
// different amounts of work (18154 tokens, H = 16 sharing 4 K/V heads, d = 128:
// 1048-1071 vs 953 TFLOP/s), slower on fixed-length batches at d <= 128 (at 576
// threads the softmax warps are capped at 96 registers and the longer-lived
// loop state spills).  The library therefore routes only packed causal batches
// here.
#include <cmath>

#include "common.h"
#include "sm103_prims.cuh"

namespace attn {
namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // keys per tile
constexpr int kSmemLimit = 232448;

template <int D>
struct FwdCfg {
  static constexpr int NQ = (D <= 128) ? 2 : 1;
  static constexpr int CH = D / 64;                  // 128-byte column chunks per row
  static constexpr int CHUNK_BYTES = BM * 128;       // one 128-row x 128-byte chunk
  static constexpr int TILE_BYTES = BM * D * 2;      // a Q, K or V tile
  // row-statistics exchange between the two warps of a row (static shared memory)
  static constexpr int XCH_BYTES = 2 * NQ * 2 * 128 * 4;
  static constexpr int NSLOT_FIT = (kSmemLimit - 2048 - XCH_BYTES - NQ * TILE_BYTES) / TILE_BYTES;
  static constexpr int NSLOT = NSLOT_FIT > 6 ? 6 : NSLOT_FIT;
  static constexpr int SMEM_BYTES = 1024 + NQ * TILE_BYTES + NSLOT * TILE_BYTES;
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
  static_assert(NSLOT >= 2, "need at least two ring stages");
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

// A tile (work item): one pair (or, at d = 256, one) of query tiles of one
// (batch, head).  Its 1-D index orders the work: causal, heaviest groups of
// every head first; otherwise group fastest, then head, then batch.
template <int NQ>
struct FwdTile {
  int g, bh, seq0, N;
  int nK[NQ];
  int nKmax, t_rel;
};

template <int NQ, bool CAUSAL, bool PACKED>
__device__ __forceinline__ bool fwd_tile(int idx, const FwdKParams& kp, int npairs, int BH,
                                         FwdTile<NQ>& w) {
  w.g = CAUSAL ? npairs - 1 - idx / BH : idx % npairs;
  w.bh = CAUSAL ? idx % BH : idx / npairs;
  w.seq0 = 0;
  w.N = kp.N;
  if constexpr (PACKED) {
    // this sequence's first token and length; groups past its end have no work
    const int b = w.bh / kp.H;
    const int s0 = kp.cu_seqlens[b];
    const int end = kp.cu_seqlens[b + 1];
    if (s0 < 0 || end < s0 || end > kp.total || end - s0 > kp.N) {
      atomicCAS(kp.status, 0, kDevBadSeqlens);
      return false;
    }
    w.seq0 = s0;
    w.N = end - s0;
  }
  const int nKtot = (w.N + BN - 1) / BN;
  w.nKmax = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int qt = w.g * NQ + t;
    w.nK[t] = (qt * BM < w.N) ? (CAUSAL ? min(nKtot, qt + 1) : nKtot) : 0;
    w.nKmax = max(w.nKmax, w.nK[t]);
  }
  // The last query tile with work runs every key tile; when its S(j)
  // completes, every MMA reading K_j and V_{j-1} has completed.
  w.t_rel = (w.nK[NQ - 1] == w.nKmax) ? NQ - 1 : 0;
  return w.nKmax > 0;
}

__device__ __forceinline__ void clc_request(void* resp, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, 16);
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(
          smem_u32(resp)),
      "r"(smem_u32(bar))
      : "memory");
}

// The x index of the CTA whose launch the request cancelled, or -1 if none was
// left to cancel.
__device__ __forceinline__ int clc_result(const void* resp) {
  int x, ok;
  asm volatile(
      "{\n .reg .b128 r;\n .reg .pred p;\n ld.shared.b128 r, [%2];\n"
      " clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n"
      " selp.s32 %1, 1, 0, p;\n"
      " clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %0, r;\n}"
      : "=r"(x), "=r"(ok)
      : "r"(smem_u32(resp))
      : "memory");
  return ok ? x : -1;
}

// Persistent CTAs: a CTA runs its own tile, then keeps taking over the tiles
// of CTAs that have not been launched yet (cluster launch control), so tile
// k+1's loads and first MMAs overlap tile k's last softmax steps and epilogue
// instead of paying a fresh CTA's start-up and drain.  PACKED: a batch of
// sequences packed back to back ([total, H, d], LSE [H, total], offsets
// cu_seqlens); otherwise [B, H, N, d] and LSE [B, H, N].
template <int D, bool CAUSAL, bool FP16, bool PACKED>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    fwd_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdKParams kp) {
  using C = FwdCfg<D>;
  constexpr int NQ = C::NQ;
  constexpr int NSLOT = C::NSLOT;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + NQ * C::TILE_BYTES;

  __shared__ __align__(8) uint64_t q_full[NQ];
  __shared__ __align__(8) uint64_t q_empty[NQ];   // Q_t may be reloaded (all S of a tile done)
  __shared__ __align__(8) uint64_t kv_full[NSLOT];
  __shared__ __align__(8) uint64_t kv_empty[NSLOT];
  __shared__ __align__(8) uint64_t s_full[NQ];
  __shared__ __align__(8) uint64_t p_full[NQ];
  __shared__ __align__(8) uint64_t o_full[NQ];
  __shared__ __align__(8) uint64_t o_empty[NQ];   // O_t read out by the epilogue
  __shared__ __align__(8) uint64_t sched_full[4];
  __shared__ __align__(8) uint64_t clc_bar[2];
  __shared__ __align__(16) uint8_t clc_resp[2][16];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ int sched[4];                         // published tile indices, -1 = no more
  __shared__ int sched_base[4];                    // ring items before each published tile
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int load_items_sh;
  __shared__ int q_loads_sh[NQ];
  __shared__ int clc_pending_sh;                   // a request whose response is outstanding
  __shared__ int clc_req_sh;                       // index of that request
  __shared__ float xch[2][NQ][2][128];             // [step parity][tile][half][row]
  __shared__ float xl[NQ][2][128];                 // epilogue row-sum exchange

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int npairs = (kp.N + BM * NQ - 1) / (BM * NQ);
  const int BH = static_cast<int>(gridDim.x) / npairs;

  if (threadIdx.x == 0) {
    for (int t = 0; t < NQ; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_empty[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 256);
      mbar_init(&o_full[t], 1);
      mbar_init(&o_empty[t], 256);
      q_loads_sh[t] = 0;
    }
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 4; ++s) mbar_init(&sched_full[s], 1);
    mbar_init(&clc_bar[0], 1);
    mbar_init(&clc_bar[1], 1);
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    load_items_sh = 0;
    clc_pending_sh = 0;
    clc_req_sh = 0;
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
    // Also the scheduler: it publishes each tile with work into a 4-entry
    // ring (the consumers run at most two tiles behind it: Q_t is reloaded
    // only after the MMA thread issued every S of the tile before).
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      int it = 0;                   // ring items over all tiles
      int qcnt[NQ];
#pragma unroll
      for (int t = 0; t < NQ; ++t) qcnt[t] = 0;
      int req = 0;                  // CLC requests issued
      bool more = true;             // no request has failed yet
      bool ok = true;
      int pub = 0;
      int idx = static_cast<int>(blockIdx.x);
      FwdTile<NQ> w;
      // the next tile with work at or after `idx` (taking over unlaunched CTAs)
      auto advance = [&](int cand) -> int {
        while (ok) {
          if (cand >= 0 && fwd_tile<NQ, CAUSAL, PACKED>(cand, kp, npairs, BH, w)) return cand;
          if (!more) return -1;
          if (!clc_pending_sh) {
            clc_request(clc_resp[req & 1], &clc_bar[req & 1]);
            clc_req_sh = req;
            clc_pending_sh = 1;
          }
          if (!mbar_wait(&clc_bar[req & 1], (req >> 1) & 1, ab, kDevTimeoutLoad)) {
            ok = false;
            return -1;
          }
          clc_pending_sh = 0;
          cand = clc_result(clc_resp[req & 1]);
          ++req;
          if (cand < 0 || cand >= static_cast<int>(gridDim.x)) {
            more = false;
            cand = -1;
          }
        }
        return -1;
      };
      idx = advance(idx);
      while (true) {
        sched[pub & 3] = idx;
        sched_base[pub & 3] = it;
        mbar_arrive(&sched_full[pub & 3]);
        ++pub;
        if (idx < 0) break;
        // ask for the following tile now, so the answer is back by the end
        if (more && !clc_pending_sh) {
          clc_request(clc_resp[req & 1], &clc_bar[req & 1]);
          clc_req_sh = req;
          clc_pending_sh = 1;
        }
        // Tensor-map coordinates: {c, row, plane} with plane = b * heads + head
        // for [B, heads, N, d]; {c, token, head, 0} for a packed batch.
        const int b = w.bh / kp.H;
        const int hq = w.bh - b * kp.H;            // query head
        const int hkv = hq / kp.group;             // its key/value head
        const int kv_plane = b * (kp.H / kp.group) + hkv;
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (w.nK[t] == 0) continue;
          if (qcnt[t] > 0 && !(ok = mbar_wait(&q_empty[t], (qcnt[t] - 1) & 1, ab, kDevTimeoutLoad)))
            break;
          mbar_arrive_expect_tx(&q_full[t], C::TILE_BYTES);
#pragma unroll
          for (int c = 0; c < C::CH; ++c)
            if constexpr (PACKED)
              tma_load_4d(sQ + t * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ, &q_full[t], c * 64,
                          w.seq0 + (w.g * NQ + t) * BM, hq, 0);
            else
              tma_load_3d(sQ + t * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ, &q_full[t], c * 64,
                          (w.g * NQ + t) * BM, w.bh);
          ++qcnt[t];
          q_loads_sh[t] = qcnt[t];
        }
        for (int j = 0; j < w.nKmax && ok; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            const int slot = it % NSLOT;
            const int use = it / NSLOT;
            if (use >= 1 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, ab, kDevTimeoutLoad)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&kv_full[slot], C::TILE_BYTES);
            uint8_t* dst = sKV + slot * C::TILE_BYTES;
#pragma unroll
            for (int c = 0; c < C::CH; ++c)
              if constexpr (PACKED)
                tma_load_4d(dst + c * C::CHUNK_BYTES, kv ? &tmV : &tmK, &kv_full[slot], c * 64,
                            w.seq0 + j * BN, hkv, 0);
              else
                tma_load_3d(dst + c * C::CHUNK_BYTES, kv ? &tmV : &tmK, &kv_full[slot], c * 64,
                            j * BN, kv_plane);
            ++it;
            load_items_sh = it;
          }
        }
        if (!ok) break;
        idx = advance(-1);
        if (!ok) break;
      }
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
      int pub = 0, base = 0;        // tiles read, ring items of earlier tiles
      int qc[NQ], sc[NQ], oc[NQ];   // per query-tile slot: Q loads, steps, outputs so far
#pragma unroll
      for (int t = 0; t < NQ; ++t) qc[t] = sc[t] = oc[t] = 0;
      FwdTile<NQ> w;
      while (ok) {
        if (!(ok = mbar_wait(&sched_full[pub & 3], (pub >> 2) & 1, ab, kDevTimeoutMma))) break;
        const int idx = sched[pub & 3];
        ++pub;
        if (idx < 0) break;
        fwd_tile<NQ, CAUSAL, PACKED>(idx, kp, npairs, BH, w);
#pragma unroll
        for (int t = 0; t < NQ; ++t)
          if (ok && w.nK[t] > 0) ok = mbar_wait(&q_full[t], qc[t] & 1, ab, kDevTimeoutMma);
        for (int j = 0; j <= w.nKmax && ok; ++j) {
          const int itK = base + 2 * j;          // ring item of K_j
          const int itV = base + 2 * j - 1;      // ring item of V_{j-1}
          const int slotK = itK % NSLOT;
          const int slotV = (itV + NSLOT) % NSLOT;
          bool haveK = false, haveV = false;
          uint64_t kdesc = 0, vdesc = 0;
#pragma unroll
          for (int t = 0; t < NQ; ++t) {
            if (j >= 1 && j - 1 < w.nK[t]) {
              // O_t += P_t(j-1) V_{j-1}
              if (!haveV) {
                if (!(ok = mbar_wait(&kv_full[slotV], (itV / NSLOT) & 1, ab, kDevTimeoutMma))) break;
                vdesc = opaque(sdesc_add(vdesc0, slotV * C::TILE_BYTES));
                haveV = true;
              }
              // the first product overwrites O_t: the last tile's epilogue must
              // have read it out
              if (j == 1 && oc[t] > 0 &&
                  !(ok = mbar_wait(&o_empty[t], (oc[t] - 1) & 1, ab, kDevTimeoutMma)))
                break;
              if (!(ok = mbar_wait(&p_full[t], (sc[t] + j - 1) & 1, ab, kDevTimeoutMma))) break;
              tc_fence_after_sync();
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk)
                mma_f16_ts(tmem + C::O_COL(t), tmem + C::S_COL(t) + C::P_COL(kk),
                           sdesc_add(vdesc, kk * 16 * 128), idPV, (j - 1 > 0 || kk > 0) ? 1u : 0u);
              if (j - 1 == w.nK[t] - 1) mma_commit(&o_full[t]);
            }
            if (j < w.nK[t]) {
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
                mma_f16_ss(tmem + C::S_COL(t), sdesc_add(qdesc, off), sdesc_add(kdesc, off), idS,
                           kk > 0 ? 1u : 0u);
              }
              mma_commit(&s_full[t]);
              if (j == w.nK[t] - 1) mma_commit(&q_empty[t]);   // Q_t may be reloaded
            }
          }
          if (!ok) break;
        }
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (w.nK[t] > 0) {
            ++qc[t];
            ++oc[t];
          }
          sc[t] += w.nK[t];
        }
        base += 2 * w.nKmax;
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
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::S_COL(t) + 64 * h;     // this half's scores
    const uint32_t tO = tmem + lane_addr + C::O_COL(t) + (D / 2) * h; // this half's O columns
    const float c2 = kp.scale_log2;
    // loop-carried state kept small (these warps are at the register limit):
    // tiles read, and the parities of the step and output barriers
    int pub = 0;
    uint32_t spar = 0, opar = 0;
    bool ok = true;
    while (ok) {
      if (__any_sync(0xffffffffu, !mbar_wait(&sched_full[pub & 3], (pub >> 2) & 1, ab,
                                             kDevTimeoutSoftmax)))
        break;
      const int idx = sched[pub & 3];
      ++pub;
      if (idx < 0) break;
      // only scalars stay live through the steps (the tile record is decoded
      // again for the epilogue)
      int qt, my_nK, N, t_rel;
      {
        FwdTile<NQ> w;
        fwd_tile<NQ, CAUSAL, PACKED>(idx, kp, npairs, BH, w);
        qt = w.g * NQ + t;
        my_nK = (t == 0) ? w.nK[0] : w.nK[NQ - 1];
        N = w.N;
        t_rel = w.t_rel;
      }
      const int row_g = qt * BM + r;
      float m_ref = -INFINITY;
      float l = 0.f;                       // this half's share of the row sum
      for (int j = 0; j < my_nK; ++j) {
        // A warp that gives up (decided for the whole warp: the TMEM loads below
        // are warp-collective) still arrives at this step's pair barrier, where
        // its partner may be waiting; the partner then fails its next wait too,
        // since this warp never signals p_full again.
        if (__any_sync(0xffffffffu, !mbar_wait(&s_full[t], spar ^ (j & 1), ab, kDevTimeoutSoftmax))) {
          named_bar_arrive(pair_bar, 64);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (t == t_rel && h == 0 && r == 0) {
          // S(j) complete: every MMA reading K_j and V_{j-1} (the last V of the
          // previous tile when j = 0) has completed
          const int item = sched_base[(pub - 1) & 3] + 2 * j;
          mbar_arrive(&kv_empty[item % NSLOT]);
          if (item >= 1) mbar_arrive(&kv_empty[(item - 1) % NSLOT]);
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
        xch[spar ^ (j & 1)][t][h][r] = m_half;
        named_bar_sync(pair_bar, 64);
        const float m_new = fmaxf(m_ref, fmaxf(m_half, xch[spar ^ (j & 1)][t][h ^ 1][r]));
        // Move the exponent reference only when the max grew by more than 2^8
        // (both halves of a row take the same decision).
        const bool need = (m_new - m_ref) * c2 > 8.f;
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
      if (!ok) break;
      spar ^= static_cast<uint32_t>(my_nK & 1);
      if (my_nK == 0) continue;
      // ---------------------------------------------------------- epilogue
      if (__any_sync(0xffffffffu, !mbar_wait(&o_full[t], opar, ab, kDevTimeoutEpilogue))) {
        named_bar_arrive(pair_bar, 64);   // release the partner at the barrier below
        ok = false;
        break;
      }
      opar ^= 1;
      tc_fence_after_sync();
      // row sum = both halves' shares
      xl[t][h][r] = l;
      named_bar_sync(pair_bar, 64);
      const float l_row = l + xl[t][h ^ 1][r];
      const float inv_l = 1.f / l_row;
      // O row: [B, H, N, d], or [total, H, d] for a packed batch
      FwdTile<NQ> w;
      fwd_tile<NQ, CAUSAL, PACKED>(sched[(pub - 1) & 3], kp, npairs, BH, w);
      const size_t orow_off = PACKED ? (static_cast<size_t>(w.seq0 + row_g) * kp.H + w.bh % kp.H) * D
                                     : (static_cast<size_t>(w.bh) * N + row_g) * D;
      uint16_t* orow = static_cast<uint16_t*>(kp.o) + orow_off + (D / 2) * h;
#pragma unroll 1
      for (int c0 = 0; c0 < D / 64; ++c0) {
        uint32_t o[32];
        tmem_ld32(tO + c0 * 32, o);
        tmem_ld_wait();
        if (c0 == D / 64 - 1) {
          // O_t has been read out: the next tile's products may overwrite it
          tc_fence_before_sync();
          mbar_arrive(&o_empty[t]);
        }
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
        kp.lse[PACKED ? static_cast<size_t>(w.bh % kp.H) * kp.total + w.seq0 + row_g
                      : static_cast<size_t>(w.bh) * N + row_g] =
            (m_ref * c2 + lg2_approx(l_row)) * 0.69314718055994530942f;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (abort_sh) {
    // Let every copy, MMA and launch-control answer this CTA issued land
    // before the memory goes away.
    if (warp == C::LOAD_WARP && lane == 0) {
#pragma unroll
      for (int t = 0; t < NQ; ++t)
        if (q_loads_sh[t] > 0) mbar_wait_drain(&q_full[t], (q_loads_sh[t] - 1) & 1);
      const int issued = load_items_sh;
      for (int s = 0; s < NSLOT && s < issued; ++s)
        mbar_wait_drain(&kv_full[s], ((issued - 1 - s) / NSLOT) & 1);
      if (clc_pending_sh) mbar_wait_drain(&clc_bar[clc_req_sh & 1], (clc_req_sh >> 1) & 1);
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

template <int D, bool FP16>
attn_status_t launch_persistent_t(const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kern = fwd_persistent_kernel<D, true, FP16, true>;
  attn_status_t s = set_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (s != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
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
  int* status = device_status_word();
  if (!status) return fail(ATTN_ERR_CUDA, "status word unavailable");
  FwdKParams kp{p.o,   p.lse, status, p.cu_seqlens,           p.N,
                p.total, p.H,  p.H / p.H_kv, p.scale * 1.4426950408889634f};
  const int rows_per_cta = BM * C::NQ;
  const unsigned npairs = static_cast<unsigned>((p.N + rows_per_cta - 1) / rows_per_cta);
  // 1-D grid of tiles (the kernel decodes the order); CTAs that start take over
  // the tiles of those not yet launched
  const dim3 grid(npairs * p.H * p.B, 1, 1);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, kp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "persistent forward kernel launch");
  return ATTN_OK;
}

template <int D>
attn_status_t launch_persistent_d(const FwdParams& p, cudaStream_t stream) {
  return p.fp16 ? launch_persistent_t<D, true>(p, stream) : launch_persistent_t<D, false>(p, stream);
}

}  // namespace

attn_status_t launch_fwd_persistent(const FwdParams& p, cudaStream_t stream) {
  if (!p.cu_seqlens || !p.causal)
    return fail(ATTN_ERR_UNSUPPORTED, "the persistent forward takes packed causal batches");
  switch (p.d) {
    case 64: return launch_persistent_d<64>(p, stream);
    case 128: return launch_persistent_d<128>(p, stream);
    case 256: return launch_persistent_d<256>(p, stream);
  }
  return fail(ATTN_ERR_INVALID_ARG, "d must be 64, 128 or 256");
}

}  // namespace attn
