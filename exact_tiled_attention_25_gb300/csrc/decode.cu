// Decode attention over a paged key/value cache on sm_103a: BF16/FP16 caches,
// and e4m3 caches with per-page block scaling.
//
// Method: "FlashAttention-3: Hopper Asynchrony and FP8 Attention", section
// "Where It Breaks", leaves a decode-focused inference kernel as open work;
// "FlashAttention 3 Hardware Acceleration: Hopper GPU Strategies for
// Long-Context Enterprise Inference Optimization" describes the key/value
// cache held in fixed-size blocks ("Memory Fragmentation") and separate
// prefill and decode functions ("Production Inference Engines").  The
// arithmetic is the forward pass of exact attention for a few new query
// tokens per sequence.
//
// GB300 design:
//  * One query tile holds the G = H / H_kv query heads that share a key/value
//    head times the n_q new tokens (G * n_q <= 128 rows); in [B, H, n_q, d]
//    these rows are contiguous, so one TMA box per 64 columns loads them.  The
//    key/value head is then read once for all of them: a decode step is bound
//    by HBM bandwidth over the cache, and the tensor cores (S = Q K^T, O += P V
//    through tensor memory, as in the forward) have ample headroom.
//  * Keys and values come from a cache [num_pages, page_size, H_kv, d] through
//    a 4-D tensor map; a 128-key tile is fetched page by page through the
//    block table (one box of min(page_size, 128) rows per page).  Tokens past
//    the sequence end and pages outside the cache are fetched as zeros.
//  * The key range of a sequence is split across CTAs (flash-decoding): each
//    split writes its partial O / l and log-sum-exp per row, and a combine
//    kernel merges the splits by their log-sum-exps.
//  * The score tile is double-buffered in tensor memory, so S(j + 1) is
//    computed while the softmax of tile j runs.
//  * Causal masking is bottom-right aligned: query token t of n_q sits at
//    position len - n_q + t and sees keys 0 .. len - n_q + t.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "common.h"
#include "sm103_prims.cuh"

namespace attn {
namespace {

constexpr int kSmemLimit = 232448;
constexpr int DBM = 128;   // query-tile rows
constexpr int DBN = 128;   // keys per tile

template <int D>
struct DecCfg {
  static constexpr int CH = D / 64;                   // 128-byte column chunks per row
  static constexpr int CHUNK = DBM * 128;             // one 128-row x 128-byte chunk
  static constexpr int TILE = DBM * D * 2;            // a Q, K or V tile
  static constexpr int NSLOT_FIT = (kSmemLimit - 2048 - TILE) / TILE;
  static constexpr int NSLOT = NSLOT_FIT > 8 ? 8 : NSLOT_FIT;
  static constexpr int SMEM = 1024 + TILE + NSLOT * TILE;
  static constexpr int THREADS = 7 * 32;   // 4 softmax warps, key producer, MMA, value producer
  static constexpr int LOAD_WARP = 4;
  static constexpr int MMA_WARP = 5;
  static constexpr int LOAD_V_WARP = 6;
  __host__ __device__ static constexpr uint32_t S_COL(int buf) { return 128u * buf; }
  static constexpr uint32_t O_COL = 256;
  static_assert(NSLOT >= 4, "ring too short");
  static_assert(O_COL + D <= 512, "TMEM overflow");
};

struct DecKParams {
  const int* block_table;   // [B, max_pages]
  const int* seq_lens;      // [B]
  float* o_part;            // [B, H, n_q, splits, D]: O / l of each split
  float* lse_part;          // [B, H, n_q, splits]
  int* status;
  int H, group, n_q, rows_real;
  int max_pages, page_size, box_rows, num_pages;
  int splits, tiles_per_split;
  int causal;
  float scale_log2;
  // e4m3 cache only
  const float* k_descale;   // [num_pages, H_kv]
  const float* v_descale;
  const float* signs;       // d values +-1 of the key transform, or nullptr
  int H_kv, page_shift;
};

__device__ __forceinline__ float lg2_dec(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Producer of one split, run by two warps: one issues the key tiles, the other
// the value tiles (kv = 0 / 1).  A warp stalls on each tensor copy it issues
// until the copy engine has taken it; measured on GB300, one issuing warp
// streamed ~34 GB/s into a CTA's ring whatever the ring depth, two warps ~51.
// Each warp runs the loop over all items and skips the other kind.  The physical pages
// of the split's boxes (one box = min(page_size, 128) rows of one page) are
// read from the block table in windows of 32 boxes, one box per lane, and the
// next window is read while the current one is in use: no table read waits in
// front of a copy.  When a window comes into use its entries are checked; for
// an e4m3 cache each tile's descales are prefetched into L2 with its copy.
// Lane 0 waits for free ring slots; one lane per (box, 64-column chunk) issues
// the tile's copies together; the keys and values of a tile use the same pages.  Item i (K_j = 2j, V_j = 2j + 1)
// goes to ring slot (i + SHIFT) % NSLOT: the first SHIFT slots may start out
// holding other data, released through their empty barrier like a used slot.
// load_items[kv] receives the item count the warp reached (its own items are
// those of parity kv below it).
template <int NSLOT, int CH, int CHUNK, int TILE, int SHIFT>
__device__ __forceinline__ void decode_produce(const CUtensorMap* tmK, const CUtensorMap* tmV,
                                               uint8_t* sKV, uint64_t* kv_full, uint64_t* kv_empty,
                                               const DecKParams& kp, const int* table, int j0,
                                               int nK, int len, int hk, int lane, const Abort& ab,
                                               int kv_own, int* load_items) {
  const int nbox = DBN / kp.box_rows;       // divides 32, so windows start at tile starts
  const int nboxes = nK * nbox;
  // box 32 w + lane lies in the split and the sequence
  auto in_seq = [&](int w) -> bool {
    const int bx = w * 32 + lane;
    return bx < nboxes && (j0 * nbox + bx) * kp.box_rows < len;
  };
  // raw table entry of box 32 w + lane (checked when its window comes into use)
  auto load_window = [&](int w) -> int {
    if (!in_seq(w)) return kp.num_pages;
    return __ldg(table + (((j0 * nbox + w * 32 + lane) * kp.box_rows) >> kp.page_shift));
  };
  // physical page of box 32 w + lane: num_pages (a zero-filled box) past the
  // sequence, or for an entry outside the cache (reported)
  auto take = [&](int pg, int w) -> int {
    if (!in_seq(w)) return kp.num_pages;
    if (pg < 0 || pg >= kp.num_pages) {
      atomicCAS(kp.status, 0, kDevBadSeqlens);
      return kp.num_pages;
    }
    return pg;
  };
  int win = take(load_window(0), 0);
  int win_next = load_window(1);
  int it = 0;
  bool ok = true;
  for (int j = 0; j < nK && ok; ++j) {
    const int wcur = (j * nbox) / 32;
    if (j > 0 && ((j * nbox) & 31) == 0) {
      win = take(win_next, wcur);
      win_next = load_window(wcur + 1);
    }
    for (int kv = 0; kv < 2; ++kv) {
      if (kv != kv_own) {
        ++it;
        continue;
      }
      const int slot = (it + SHIFT) % NSLOT;
      const int use = (it + SHIFT) / NSLOT;
      int go = 1;
      if (lane == 0) {
        if (use >= 1 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, ab, kDevTimeoutLoad)) go = 0;
        else mbar_arrive_expect_tx(&kv_full[slot], TILE);
      }
      if (!__shfl_sync(0xffffffffu, go, 0)) {
        ok = false;
        break;
      }
      // lane x * CH + c issues column chunk c of box x (one instruction for the
      // whole tile; lane 0 registered the expected bytes above, before any lane
      // issues); nbox * CH <= 32
      uint8_t* dst = sKV + slot * TILE;
      const int x = lane / CH, c = lane - x * CH;
      const int phys = __shfl_sync(0xffffffffu, win, (j * nbox + x) & 31);
      if (x < nbox) {
        const int tok = (j0 + j) * DBN + x * kp.box_rows;
        tma_load_4d(dst + c * CHUNK + x * kp.box_rows * 128, kv ? tmV : tmK, &kv_full[slot], c * 64,
                    tok & (kp.page_size - 1), hk, phys);
        if (kp.k_descale && c == 0 && phys < kp.num_pages) {
          // the tile's descales, into L2 a ring's depth before the softmax
          // warps read them (a whole block-table window ahead they were
          // evicted again by the stream of keys and values)
          const size_t at = static_cast<size_t>(phys) * kp.H_kv + hk;
          asm volatile("prefetch.global.L2 [%0];" ::"l"((kv ? kp.v_descale : kp.k_descale) + at));
        }
      }
      ++it;
    }
  }
  if (lane == 0) load_items[kv_own] = it;
}

// After an abort: wait (bounded) for the copies a producer warp still has in
// flight, the last NSLOT items it may have issued.
template <int NSLOT, int SHIFT, typename Parity>
__device__ __forceinline__ void decode_drain_items(uint64_t* kv_full, int issued, int kv_own,
                                                   Parity parity) {
  for (int i = issued - 1; i >= 0 && i >= issued - NSLOT; --i)
    if ((i & 1) == kv_own) mbar_wait_drain(&kv_full[(i + SHIFT) % NSLOT], parity(i));
}

template <int D, bool FP16>
__global__ void __launch_bounds__(DecCfg<D>::THREADS, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecKParams kp) {
  using C = DecCfg<D>;
  constexpr int NSLOT = C::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::TILE;

  __shared__ __align__(8) uint64_t q_full;
  __shared__ __align__(8) uint64_t kv_full[NSLOT];
  __shared__ __align__(8) uint64_t kv_empty[NSLOT];
  __shared__ __align__(8) uint64_t s_full[2];    // per score buffer
  __shared__ __align__(8) uint64_t p_full[2];    // per score buffer
  __shared__ __align__(8) uint64_t pv_done;      // one phase per tile
  __shared__ __align__(8) uint64_t o_full;
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int load_items_sh[2];

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int split = blockIdx.x;
  const int hk = blockIdx.y;
  const int b = blockIdx.z;
  const int len = kp.seq_lens[b];
  if (len < 0 || len > kp.max_pages * kp.page_size) {
    if (threadIdx.x == 0) atomicCAS(kp.status, 0, kDevBadSeqlens);
    return;
  }
  const int ntiles = (len + DBN - 1) / DBN;
  const int j0 = split * kp.tiles_per_split;
  const int nK = max(0, min(ntiles, j0 + kp.tiles_per_split) - j0);
  const int r = warp * 32 + lane;             // query-tile row of a softmax thread
  const int gq = r / kp.n_q, tq = r - gq * kp.n_q;
  const size_t prow = (static_cast<size_t>(b) * kp.H + hk * kp.group + gq) * kp.n_q + tq;
  if (nK == 0) {
    // no keys in this split: it contributes nothing to the merge
    if (warp < 4 && r < kp.rows_real) kp.lse_part[prow * kp.splits + split] = -INFINITY;
    return;
  }
  const int total_items = 2 * nK;              // K_0, V_0, K_1, V_1, ... of this split

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
    }
    mbar_init(&pv_done, 1);
    mbar_init(&o_full, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    load_items_sh[0] = load_items_sh[1] = 0;
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

  if (warp == C::LOAD_WARP || warp == C::LOAD_V_WARP) {
    // ------------------------------------------------------------ producers
    const int kv_own = warp == C::LOAD_WARP ? 0 : 1;
    if (lane == 0 && kv_own == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(&q_full, C::TILE);
#pragma unroll
      for (int c = 0; c < C::CH; ++c)
        tma_load_3d(sQ + c * C::CHUNK, &tmQ, &q_full, c * 64, hk * kp.group * kp.n_q, b);
    }
    decode_produce<NSLOT, C::CH, C::CHUNK, C::TILE, 0>(
        &tmK, &tmV, sKV, kv_full, kv_empty, kp, kp.block_table + static_cast<size_t>(b) * kp.max_pages,
        j0, nK, len, hk, lane, ab, kv_own, load_items_sh);
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr Elt E = FP16 ? Elt::F16 : Elt::BF16;
      constexpr uint32_t idS = idesc_f16(E, 128, DBN, false, false);
      constexpr uint32_t idPV = idesc_f16(E, 128, D, false, true);
      const uint64_t qdesc = sdesc_sw128(smem_u32(sQ), 16, 1024);              // K-major Q
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(sKV), 16, 1024);            // K-major K
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(sKV), C::CHUNK, 1024);      // MN-major V
      bool ok = mbar_wait(&q_full, 0, ab, kDevTimeoutMma);
      // S(jj) = Q K_jj^T into buffer jj % 2
      auto issue_s = [&](int jj) -> bool {
        const int item = 2 * jj;
        const int slot = item % NSLOT;
        if (!mbar_wait(&kv_full[slot], (item / NSLOT) & 1, ab, kDevTimeoutMma)) return false;
        const uint64_t kdesc = opaque(sdesc_add(kdesc0, slot * C::TILE));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::CHUNK + (kk % 4) * 32;
          mma_f16_ss(tmem + C::S_COL(jj & 1), sdesc_add(qdesc, off), sdesc_add(kdesc, off), idS,
                     kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[jj & 1]);
        // the slot of K_jj is free once these products complete
        if (item + NSLOT < total_items) mma_commit(&kv_empty[slot]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && nK > 1) ok = issue_s(1);
      for (int j = 0; j < nK && ok; ++j) {
        // O += P(j) V_j, P(j) packed 16-bit in columns [0, 64) of buffer j % 2
        const int item = 2 * j + 1;
        const int slot = item % NSLOT;
        if (!(ok = mbar_wait(&kv_full[slot], (item / NSLOT) & 1, ab, kDevTimeoutMma))) break;
        const uint64_t vdesc = opaque(sdesc_add(vdesc0, slot * C::TILE));
        if (!(ok = mbar_wait(&p_full[j & 1], (j >> 1) & 1, ab, kDevTimeoutMma))) break;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < DBN / 16; ++kk)
          mma_f16_ts(tmem + C::O_COL, tmem + C::S_COL(j & 1) + 8 * kk,
                     sdesc_add(vdesc, kk * 16 * 128), idPV, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&pv_done);
        if (item + NSLOT < total_items) mma_commit(&kv_empty[slot]);   // V_j's slot
        if (j == nK - 1) mma_commit(&o_full);
        if (j + 2 < nK) ok = issue_s(j + 2);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Thread r owns row r (TMEM lane r) of S and O.
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const float c2 = kp.scale_log2;
    // keys this row may see: all of the sequence, or (causal) up to its position
    const int vis_end = kp.causal ? min(len, len - kp.n_q + tq + 1) : len;
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < nK; ++j) {
      if (__any_sync(0xffffffffu, !mbar_wait(&s_full[j & 1], (j >> 1) & 1, ab, kDevTimeoutSoftmax))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t tS = tmem + lane_addr + C::S_COL(j & 1);
      uint32_t sr[DBN];
#pragma unroll
      for (int c0 = 0; c0 < DBN / 32; ++c0)
        tmem_ld32(tS + c0 * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c0 * 32]));
      tmem_ld_wait();
      const int kbase = (j0 + j) * DBN;
      if (kbase + DBN > vis_end) {
        const int lim = vis_end - kbase;
#pragma unroll
        for (int c = 0; c < DBN; ++c)
          if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx[16];
#pragma unroll
      for (int u = 0; u < 16; ++u)
        mx[u] = fmax3(__uint_as_float(sr[8 * u]), __uint_as_float(sr[8 * u + 1]),
                      fmax3(__uint_as_float(sr[8 * u + 2]), __uint_as_float(sr[8 * u + 3]),
                            fmax3(__uint_as_float(sr[8 * u + 4]), __uint_as_float(sr[8 * u + 5]),
                                  fmaxf(__uint_as_float(sr[8 * u + 6]), __uint_as_float(sr[8 * u + 7])))));
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = fmaxf(mx[u], mx[u + 8]);
      const float m_new = fmaxf(m_ref, fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                             fmaxf(mx[6], mx[7])));
      // lazy rescale: move the exponent reference only when the max grew by
      // more than 2^8
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
      for (int c0 = 0; c0 < DBN / 32; ++c0) {
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
        // packed P of keys [32 c0, +32) -> columns [16 c0, +16)
        tmem_st16(tS + c0 * 16, pk);
      }
      const uint64_t acc = fadd2(acc0, acc1);
      l += lo2(acc) + hi2(acc);
      // Rescale O.  P(j-1) V_{j-1} may still be in flight (it is issued after
      // step j-1 ends), so wait for it; this step's product is issued only
      // after the arrive below.
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        if (__any_sync(0xffffffffu, !mbar_wait(&pv_done, (j - 1) & 1, ab, kDevTimeoutSoftmax))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll 1
        for (int c0 = 0; c0 < D / 32; ++c0) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_addr + C::O_COL + c0 * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_addr + C::O_COL + c0 * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&p_full[j & 1]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && !__any_sync(0xffffffffu, !mbar_wait(&o_full, 0, ab, kDevTimeoutEpilogue))) {
      tc_fence_after_sync();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      float* dst = kp.o_part + (prow * kp.splits + split) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_addr + C::O_COL + c0 * 32, o);
        tmem_ld_wait();
        if (r < kp.rows_real) {
          float4* d4 = reinterpret_cast<float4*>(dst + c0 * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            d4[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
        }
      }
      if (r < kp.rows_real)
        kp.lse_part[prow * kp.splits + split] =
            l > 0.f ? (m_ref * c2 + lg2_dec(l)) * 0.69314718055994530942f : -INFINITY;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (abort_sh) {
    if ((warp == C::LOAD_WARP || warp == C::LOAD_V_WARP) && lane == 0) {
      const int kv_own = warp == C::LOAD_WARP ? 0 : 1;
      if (kv_own == 0) mbar_wait_drain(&q_full, 0);
      decode_drain_items<NSLOT, 0>(kv_full, load_items_sh[kv_own], kv_own,
                                   [](int i) -> uint32_t { return (i / NSLOT) & 1u; });
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

// Merge the splits of every (b, h, t) row: LSE = log sum_s exp(lse_s) and
// O = sum_s exp(lse_s - LSE) O_s.  One warp per row, D / 32 columns per lane.
template <int D, bool FP16>
__global__ void __launch_bounds__(256)
    decode_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                          uint16_t* __restrict__ o, float* __restrict__ lse, long long rows,
                          int splits) {
  constexpr int PER = D / 32;
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* lp = lse_part + row * splits;
  float mx = -INFINITY;
  for (int s = lane; s < splits; s += 32) mx = fmaxf(mx, lp[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float sum = 0.f;
  if (mx != -INFINITY)
    for (int s = lane; s < splits; s += 32) sum += expf(lp[s] - mx);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float total = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const float ls = lp[s];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - total);
      const float* op = o_part + (row * splits + s) * D + lane * PER;
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = fmaf(w, op[i], acc[i]);
    }
  }
  uint16_t* orow = o + row * D + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; i += 2) {
    const uint32_t pk = FP16 ? cvt_pack_f16(acc[i], acc[i + 1]) : cvt_pack_bf16(acc[i], acc[i + 1]);
    *reinterpret_cast<uint32_t*>(orow + i) = pk;
  }
  if (lane == 0) lse[row] = total;
}

// ================================================================ e4m3 cache ====
// The same schedule over a cache of e4m3 codes with one float32 descale per
// (physical page, key/value head), d = 128.  Both products run as kind::f8f6f4:
//  * the query tile arrives in 16-bit; each softmax thread quantises its row
//    to e4m3 in shared memory (optionally after the transform x -> x M, M =
//    diag(signs) H_d / sqrt(d), which the keys were stored with), with one
//    descale dq = amax / 448 per row, by the block quantiser's rule;
//  * a 128-key tile may span several pages (page_size >= 16), so descales are
//    kept per 16-key group: the score coefficient of group g is
//    scale * log2(e) * dq * dk_g, and the value descale enters the exponent:
//    the running maximum is taken over y = s + log2(dv_g), so P' = 2^(y - m)
//    <= 1 multiplies the raw value codes and the row sum adds P' / dv_g.
//    No value-descale pre-scan or extra O rescale is needed.
//  * lanes 0..15 of every softmax warp fetch the descales of a tile two tiles
//    ahead (its block-table entries two tiles before that) and share them by
//    shuffles.
struct Dec8Cfg {
  static constexpr int D = 128;
  static constexpr int CHUNK16 = DBM * 128;          // 64 columns of the 16-bit query tile
  static constexpr int Q16 = 2 * CHUNK16;            // 16-bit query tile, in ring slots 0 and 1
  static constexpr int TILE8 = DBM * D;              // e4m3 query, key or value tile
  static constexpr int NSLOT_FIT = (kSmemLimit - 2048 - TILE8) / TILE8;
  static constexpr int NSLOT = NSLOT_FIT > 14 ? 14 : NSLOT_FIT;
  static constexpr int SHIFT = 2;                    // ring slots the query tile occupies first
  static constexpr int SMEM = 1024 + TILE8 + NSLOT * TILE8;
  static_assert(Q16 == SHIFT * TILE8, "query staging must fill whole ring slots");
  static constexpr int THREADS = 7 * 32;
  static constexpr int LOAD_WARP = 4;      // keys (and the query tile)
  static constexpr int MMA_WARP = 5;
  static constexpr int LOAD_V_WARP = 6;    // values
  __host__ __device__ static constexpr uint32_t S_COL(int buf) { return 128u * buf; }
  static constexpr uint32_t O_COL = 256;
  static_assert(NSLOT >= 6, "ring too short");
};

template <bool FP16>
__global__ void __launch_bounds__(Dec8Cfg::THREADS, 1)
    decode_fp8_split_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const DecKParams kp) {
  using C = Dec8Cfg;
  constexpr int D = C::D;
  constexpr int NSLOT = C::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ8 = smem;                 // e4m3 query tile
  uint8_t* sKV = smem + C::TILE8;      // ring of NSLOT key / value tiles
  uint8_t* sQ = sKV;                   // 16-bit query tile (two 64-column chunks) in slots 0, 1

  __shared__ __align__(8) uint64_t q_full;
  __shared__ __align__(8) uint64_t q8_full;
  __shared__ __align__(8) uint64_t kv_full[NSLOT];
  __shared__ __align__(8) uint64_t kv_empty[NSLOT];
  __shared__ __align__(8) uint64_t s_full[2];
  __shared__ __align__(8) uint64_t p_full[2];
  __shared__ __align__(8) uint64_t pv_done;
  __shared__ __align__(8) uint64_t o_full;
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int load_items_sh[2];

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int split = blockIdx.x;
  const int hk = blockIdx.y;
  const int b = blockIdx.z;
  const int len = kp.seq_lens[b];
  if (len < 0 || len > kp.max_pages * kp.page_size) {
    if (threadIdx.x == 0) atomicCAS(kp.status, 0, kDevBadSeqlens);
    return;
  }
  const int ntiles = (len + DBN - 1) / DBN;
  const int j0 = split * kp.tiles_per_split;
  const int nK = max(0, min(ntiles, j0 + kp.tiles_per_split) - j0);
  const int r = warp * 32 + lane;
  const int gq = r / kp.n_q, tq = r - gq * kp.n_q;
  const size_t prow = (static_cast<size_t>(b) * kp.H + hk * kp.group + gq) * kp.n_q + tq;
  if (nK == 0) {
    if (warp < 4 && r < kp.rows_real) kp.lse_part[prow * kp.splits + split] = -INFINITY;
    return;
  }
  const int total_items = 2 * nK;

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&q8_full, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
    }
    mbar_init(&pv_done, 1);
    mbar_init(&o_full, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    load_items_sh[0] = load_items_sh[1] = 0;
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
  const int* table = kp.block_table + static_cast<size_t>(b) * kp.max_pages;
  // Phase parity of the full barrier of item i's slot: the uses of that slot
  // before it, not counting the query tile that first occupies slots
  // 0 .. SHIFT-1 (it arrives through q_full, not through the slot's barrier).
  auto full_parity = [](int i) -> uint32_t {
    const int slot = (i + C::SHIFT) % NSLOT;
    return static_cast<uint32_t>((i + C::SHIFT) / NSLOT - (slot < C::SHIFT ? 1 : 0)) & 1u;
  };

  if (warp == C::LOAD_WARP || warp == C::LOAD_V_WARP) {
    // ------------------------------------------------------------ producers
    const int kv_own = warp == C::LOAD_WARP ? 0 : 1;
    if (lane == 0 && kv_own == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(&q_full, C::Q16);
#pragma unroll
      for (int c = 0; c < 2; ++c)
        tma_load_3d(sQ + c * C::CHUNK16, &tmQ, &q_full, c * 64, hk * kp.group * kp.n_q, b);
    }
    decode_produce<NSLOT, 1, 0, C::TILE8, C::SHIFT>(&tmK, &tmV, sKV, kv_full, kv_empty, kp, table, j0,
                                                    nK, len, hk, lane, ab, kv_own, load_items_sh);
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idS = idesc_e4m3(128, DBN, false, false);
      constexpr uint32_t idPV = idesc_e4m3(128, D, false, true);
      const uint64_t qdesc = sdesc_sw128(smem_u32(sQ8), 16, 1024);            // K-major Q
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(sKV), 16, 1024);           // K-major K
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(sKV), C::TILE8, 1024);     // MN-major V
      bool ok = mbar_wait(&q8_full, 0, ab, kDevTimeoutMma);
      if (ok) {
        // every softmax thread has read its 16-bit query row: slots 0 and 1
        // are free for keys and values
        for (int sl = 0; sl < C::SHIFT; ++sl) mbar_arrive(&kv_empty[sl]);
      }
      auto issue_s = [&](int jj) -> bool {
        const int item = 2 * jj;
        const int slot = (item + C::SHIFT) % NSLOT;
        if (!mbar_wait(&kv_full[slot], full_parity(item), ab, kDevTimeoutMma)) return false;
        const uint64_t kdesc = opaque(sdesc_add(kdesc0, slot * C::TILE8));
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
          mma_f8_ss(tmem + C::S_COL(jj & 1), sdesc_add(qdesc, kk * 32), sdesc_add(kdesc, kk * 32),
                    idS, kk > 0 ? 1u : 0u);
        mma_commit(&s_full[jj & 1]);
        // the slot of K_jj is free once these products complete
        if (item + NSLOT < total_items) mma_commit(&kv_empty[slot]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && nK > 1) ok = issue_s(1);
      for (int j = 0; j < nK && ok; ++j) {
        // O += P'(j) V_j, P' packed e4m3 in columns [0, 32) of buffer j % 2
        const int item = 2 * j + 1;
        const int slot = (item + C::SHIFT) % NSLOT;
        if (!(ok = mbar_wait(&kv_full[slot], full_parity(item), ab, kDevTimeoutMma))) break;
        const uint64_t vdesc = opaque(sdesc_add(vdesc0, slot * C::TILE8));
        if (!(ok = mbar_wait(&p_full[j & 1], (j >> 1) & 1, ab, kDevTimeoutMma))) break;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < DBN / 32; ++kk)
          mma_f8_ts(tmem + C::O_COL, tmem + C::S_COL(j & 1) + 8 * kk,
                    sdesc_add(vdesc, kk * 32 * 128), idPV, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&pv_done);
        if (item + NSLOT < total_items) mma_commit(&kv_empty[slot]);   // V_j's slot
        if (j == nK - 1) mma_commit(&o_full);
        if (j + 2 < nK) ok = issue_s(j + 2);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    bool ok = true;
    float c_q = 0.f;   // scale * log2(e) * dq of this row
    // ---- quantise this thread's query row
    if (__any_sync(0xffffffffu, !mbar_wait(&q_full, 0, ab, kDevTimeoutSoftmax))) {
      ok = false;
    } else if (r >= kp.rows_real) {
      // padding row: its scores are never used; zero codes
#pragma unroll
      for (int u = 0; u < 8; ++u) st_shared_v4(smem_u32(sQ8 + r * 128 + (u << 4)), 0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
      mbar_arrive(&q8_full);
    } else {
      float x[D];
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 w = *reinterpret_cast<const uint4*>(sQ + c * C::CHUNK16 + r * 128 +
                                                          ((u ^ (r & 7)) << 4));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 f;
            if (FP16) f = __half22float2(*reinterpret_cast<const __half2*>(&ws[e]));
            else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e]));
            x[c * 64 + u * 8 + 2 * e] = f.x;
            x[c * 64 + u * 8 + 2 * e + 1] = f.y;
          }
        }
      if (kp.signs) {
        // x -> (x o signs) H_d / sqrt(d), fast Walsh-Hadamard butterflies
#pragma unroll
        for (int i = 0; i < D; i += 4) {
          const float4 sg = __ldg(reinterpret_cast<const float4*>(kp.signs + i));
          x[i] *= sg.x;
          x[i + 1] *= sg.y;
          x[i + 2] *= sg.z;
          x[i + 3] *= sg.w;
        }
#pragma unroll
        for (int h = 1; h < D; h <<= 1)
#pragma unroll
          for (int i = 0; i < D; ++i)
            if ((i & h) == 0) {
              const float a = x[i], bb = x[i + h];
              x[i] = a + bb;
              x[i + h] = a - bb;
            }
#pragma unroll
        for (int i = 0; i < D; ++i) x[i] *= 0.08838834764831845f;   // 1 / sqrt(128)
      }
      float am[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < D; ++i) am[i & 3] = fmaxf(am[i & 3], fabsf(x[i]));
      const float amax = fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3]));
      // descale = amax / 448 and code = e4m3(x / descale) with x / descale
      // rounded as an IEEE float32 division (the block quantiser's rule): one
      // division for y = RN(1 / dq), then a corrected product per value.
      const float dq = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
      const float y = __fdiv_rn(1.f, dq);
      auto quot = [&](float v) -> float { return div_by_recip(v, dq, y); };
      c_q = kp.scale_log2 * dq;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint32_t wq[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = u * 16 + e * 4;
          wq[e] = cvt_pack_e4m3x4(quot(x[i]), quot(x[i + 1]), quot(x[i + 2]), quot(x[i + 3]));
        }
        st_shared_v4(smem_u32(sQ8 + r * 128 + ((u ^ (r & 7)) << 4)), wq[0], wq[1], wq[2], wq[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&q8_full);
    }
    // ---- descales of the 16-key groups, fetched ahead by lanes 0..15
    const float* dsrc = (lane & 8) ? kp.v_descale : kp.k_descale;
    auto page_of = [&](int jj) -> int {
      const int tok = (j0 + jj) * DBN + 16 * (lane & 7);
      if (lane >= 16 || jj >= nK || tok >= len) return -1;
      return __ldg(table + (tok >> kp.page_shift));   // checked when used, a tile later
    };
    auto desc_of = [&](int ph) -> float {
      return (ph < 0 || ph >= kp.num_pages) ? 1.f
                                             : __ldg(dsrc + static_cast<size_t>(ph) * kp.H_kv + hk);
    };
    // descales two tiles ahead of use, block-table entries two tiles before that
    int ph3 = page_of(3), ph4 = page_of(4);
    float dcur = desc_of(page_of(0));
    float dn1 = desc_of(page_of(1));
    float dn2 = desc_of(page_of(2));

    const int vis_end = kp.causal ? min(len, len - kp.n_q + tq + 1) : len;
    float m_ref = -INFINITY;   // log2 units of y = s + log2(dv)
    float l = 0.f;             // sum of 2^(s - m_ref)
    for (int j = 0; j < nK && ok; ++j) {
      // group coefficients: lanes g < 8 hold dk_g, lanes 8 + g hold dv_g
      const float lgd = lg2_dec(dcur);
      float invd;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(invd) : "f"(dcur));
      float coef[8], lgv[8], ivv[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        coef[g] = c_q * __shfl_sync(0xffffffffu, dcur, g);
        lgv[g] = __shfl_sync(0xffffffffu, lgd, 8 + g);
        ivv[g] = __shfl_sync(0xffffffffu, invd, 8 + g);
      }
      if (__any_sync(0xffffffffu, !mbar_wait(&s_full[j & 1], (j >> 1) & 1, ab, kDevTimeoutSoftmax))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t tS = tmem + lane_addr + C::S_COL(j & 1);
      uint32_t sr[DBN];
#pragma unroll
      for (int c0 = 0; c0 < DBN / 32; ++c0)
        tmem_ld32(tS + c0 * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c0 * 32]));
      tmem_ld_wait();
      const int kbase = (j0 + j) * DBN;
      if (kbase + DBN > vis_end) {
        const int lim = vis_end - kbase;
#pragma unroll
        for (int c = 0; c < DBN; ++c)
          if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
      }
      // max over y: per 16-key group, raw max x coefficient + log2(dv)
      float mt = -INFINITY;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const int c = 16 * g;
        const float m16 = fmaxf(
            fmax3(fmax3(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), __uint_as_float(sr[c + 2])),
                  fmax3(__uint_as_float(sr[c + 3]), __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5])),
                  fmax3(__uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]), __uint_as_float(sr[c + 8]))),
            fmax3(fmax3(__uint_as_float(sr[c + 9]), __uint_as_float(sr[c + 10]), __uint_as_float(sr[c + 11])),
                  fmax3(__uint_as_float(sr[c + 12]), __uint_as_float(sr[c + 13]), __uint_as_float(sr[c + 14])),
                  __uint_as_float(sr[c + 15])));
        mt = fmaxf(mt, fmaf(m16, coef[g], lgv[g]));
      }
      // The reference follows the running maximum exactly (no lazy slack):
      // the largest weight is then exactly 1, which e4m3 holds exactly, and in
      // a peaked row that weight carries most of the sum.  A lagging reference
      // (weights up to 2^8) rounds it too and about doubles the P rounding
      // error; the running maximum of a decode row rises on few tiles, so the
      // extra O rescales cost little.
      const float m_new = fmaxf(m_ref, mt);
      const bool need = m_new > m_ref;
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx(m_ref - m_new);
        l *= alpha;
        m_ref = m_new;
      }
      const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
#pragma unroll
      for (int c0 = 0; c0 < DBN / 32; ++c0) {
        uint32_t pk[8];
#pragma unroll
        for (int hg = 0; hg < 2; ++hg) {
          const int g = 2 * c0 + hg;
          const uint64_t cc = pack2(coef[g], coef[g]);
          const float off = neg + lgv[g];
          const uint64_t nn = pack2(off, off);
          uint64_t acc = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = 16 * g + 4 * i;
            const uint64_t y0 = ffma2(pack2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), cc, nn);
            const uint64_t y1 = ffma2(pack2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), cc, nn);
            const float p0 = ex2_approx(lo2(y0));
            const float p1 = ex2_approx(hi2(y0));
            const float p2 = ex2_approx(lo2(y1));
            const float p3 = ex2_approx(hi2(y1));
            acc = fadd2(acc, fadd2(pack2(p0, p1), pack2(p2, p3)));
            pk[4 * hg + i] = cvt_pack_e4m3x4(p0, p1, p2, p3);
          }
          l = fmaf(lo2(acc) + hi2(acc), ivv[g], l);
        }
        // P' of keys [32 c0, +32) -> columns [8 c0, +8)
        tmem_st_x8(tS + c0 * 8, pk);
      }
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        if (__any_sync(0xffffffffu, !mbar_wait(&pv_done, (j - 1) & 1, ab, kDevTimeoutSoftmax))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll 1
        for (int c0 = 0; c0 < D / 32; ++c0) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_addr + C::O_COL + c0 * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_addr + C::O_COL + c0 * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&p_full[j & 1]);
      // advance the descale pipeline
      dcur = dn1;
      dn1 = dn2;
      dn2 = desc_of(ph3);
      ph3 = ph4;
      ph4 = page_of(j + 5);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && !__any_sync(0xffffffffu, !mbar_wait(&o_full, 0, ab, kDevTimeoutEpilogue))) {
      tc_fence_after_sync();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      float* dst = kp.o_part + (prow * kp.splits + split) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_addr + C::O_COL + c0 * 32, o);
        tmem_ld_wait();
        if (r < kp.rows_real) {
          float4* d4 = reinterpret_cast<float4*>(dst + c0 * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            d4[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
        }
      }
      if (r < kp.rows_real)
        kp.lse_part[prow * kp.splits + split] =
            l > 0.f ? (m_ref + lg2_dec(l)) * 0.69314718055994530942f : -INFINITY;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (abort_sh) {
    if ((warp == C::LOAD_WARP || warp == C::LOAD_V_WARP) && lane == 0) {
      const int kv_own = warp == C::LOAD_WARP ? 0 : 1;
      if (kv_own == 0) mbar_wait_drain(&q_full, 0);
      decode_drain_items<NSLOT, C::SHIFT>(kv_full, load_items_sh[kv_own], kv_own, full_parity);
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

// ============================================ e4m3 cache, keys on M ====
// A decode step has few query rows per key/value head (R = G * n_q).  With
// R <= 16 the products run transposed, the keys of a tile on the MMA's M side
// and the query rows on N = 16:
//     S^T (128 keys x 16) = K_j Q8^T,      O^T (d x 16) += V_j^T P'^T,
// so each softmax thread holds the scores of one key for every query row and
// computes NC (>= R, a power of two <= 16) exponentials per tile, where the
// rows-on-M kernel computes 128 per thread for 128 padded rows (with more than
// 4 rows, CW = 2 softmax warps share a key quarter, each taking half of the
// columns).  The row maximum becomes a reduction over the 128 key threads
// (redux.sync per warp, then the four key quarters' partial maxima through
// shared memory and an mbarrier), the row sums stay per thread until the
// epilogue (one column-transposing warp exchange there), and the weights go
// to shared memory as the B operand of the P V product.  Numerics are those of
// the rows-on-M kernel: the same query quantiser, the exact running maximum of
// y = s + log2(dv) per row, P' = 2^(y - m) in e4m3 against raw value codes,
// and row sums of P' / dv.
template <int CW>   // softmax warps per key quarter (each takes NC / CW query columns)
struct Dec8TCfg {
  static constexpr int D = 128;
  static constexpr int NQ = 16;                  // MMA N: query rows, padded
  static constexpr int TILE8 = DBN * D;          // e4m3 key or value tile, 16 KB
  static constexpr int Q8_OFF = 0;               // e4m3 query rows, 16 x 128 B
  static constexpr int P_OFF = 2048;             // two e4m3 P'^T tiles, 16 x 128 B each
  static constexpr int Q16_OFF = 6144;           // 16-bit query rows: two 64-column chunks
  static constexpr int CHUNK16 = NQ * 128;
  static constexpr int RING_OFF = 10240;
  static constexpr int NSLOT_FIT = (kSmemLimit - 2048 - RING_OFF) / TILE8;
  static constexpr int NSLOT = NSLOT_FIT > 13 ? 13 : NSLOT_FIT;
  static constexpr int SMEM = 1024 + RING_OFF + NSLOT * TILE8;
  static constexpr int SOFTMAX_WARPS = 4 * CW;
  static constexpr int THREADS = (SOFTMAX_WARPS + 4) * 32;
  static constexpr int LOAD_WARP = SOFTMAX_WARPS;         // keys (and the query rows)
  static constexpr int MMA_WARP = SOFTMAX_WARPS + 1;      // P V products (and the TMEM allocation)
  static constexpr int LOAD_V_WARP = SOFTMAX_WARPS + 2;   // values
  static constexpr int MMA_S_WARP = SOFTMAX_WARPS + 3;    // score products
  __host__ __device__ static constexpr uint32_t S_COL(int buf) { return 16u * buf; }
  static constexpr uint32_t O_COL = 32;
  static constexpr uint32_t TMEM_COLS = 64;
  static_assert(NSLOT >= 6, "ring too short");
  static_assert(Q16_OFF + 2 * CHUNK16 <= RING_OFF, "staging overlaps the ring");
};

// One exchange round at lane distance STEP with W columns left (rounds with
// W = 1 combine the single column), then the next round.
template <int NC, int W, int STEP, typename Op>
__device__ __forceinline__ float col_reduce_round(float (&cur)[NC], int lane, Op op, int& c) {
  if constexpr (STEP == 0) {
    return cur[0];
  } else if constexpr (W > 1) {
    constexpr int H = W / 2;
    const bool hi = (lane & STEP) != 0;
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const float send = hi ? cur[i] : cur[i + H];
      const float keep = hi ? cur[i + H] : cur[i];
      cur[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, STEP));
    }
    if (hi) c += H;
    return col_reduce_round<NC, H, STEP / 2>(cur, lane, op, c);
  } else {
    cur[0] = op(cur[0], __shfl_xor_sync(0xffffffffu, cur[0], STEP));
    return col_reduce_round<NC, 1, STEP / 2>(cur, lane, op, c);
  }
}

// Reduce NC per-lane values over the 32 lanes of a warp, column by column.
// While more than one column is left, each exchange round halves the columns a
// lane keeps: it keeps one half, sends the other to its partner and combines
// what it receives; the remaining rounds combine a single column.  Returns the
// warp total of column *col (every lane ends with some column; 32 / NC lanes
// share each).
template <int NC, typename Op>
__device__ __forceinline__ float warp_col_reduce(const float (&v)[NC], int lane, Op op, int* col) {
  float cur[NC];
#pragma unroll
  for (int i = 0; i < NC; ++i) cur[i] = v[i];
  int c = 0;
  const float r = col_reduce_round<NC, NC, 16>(cur, lane, op, c);
  *col = c;
  return r;
}

struct AddOp {
  __device__ float operator()(float a, float b) const { return a + b; }
};

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 16) tmem_ld16(taddr, r);
  else if constexpr (N == 8) tmem_ld8(taddr, r);
  else tmem_ld4(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 16) tmem_st16(taddr, r);
  else if constexpr (N == 8) tmem_st_x8(taddr, r);
  else tmem_st4(taddr, r);
}

__device__ __forceinline__ void st_shared_u8(uint32_t saddr, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(saddr), "r"(v) : "memory");
}

template <bool FP16, int NC, int CW>
__global__ void __launch_bounds__(Dec8TCfg<CW>::THREADS, 1)
    decode_fp8_keys_kernel(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const DecKParams kp) {
  using C = Dec8TCfg<CW>;
  constexpr int D = C::D;
  constexpr int NSLOT = C::NSLOT;
  constexpr int NCW = NC / CW;   // query columns of one softmax thread
  static_assert(NC == 4 || NC == 8 || NC == 16, "query columns");
  static_assert(NCW == 4 || NCW == 8 || NCW == 16, "columns per softmax thread");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ8 = smem + C::Q8_OFF;
  uint8_t* sP = smem + C::P_OFF;
  uint8_t* sQ16 = smem + C::Q16_OFF;
  uint8_t* sKV = smem + C::RING_OFF;

  __shared__ __align__(8) uint64_t q_full;
  __shared__ __align__(8) uint64_t q8_full;
  __shared__ __align__(8) uint64_t kv_full[NSLOT];
  __shared__ __align__(8) uint64_t kv_empty[NSLOT];
  __shared__ __align__(8) uint64_t s_full[2];
  __shared__ __align__(8) uint64_t p_full[2];
  __shared__ __align__(8) uint64_t red_full[2];
  __shared__ __align__(8) uint64_t fin_bar;
  __shared__ __align__(8) uint64_t o_full;
  __shared__ __align__(8) uint64_t drain_bar[2];
  __shared__ __align__(16) float red_sh[2][4 * NC];   // [parity][key quarter][column]: maxima
  __shared__ __align__(16) float fin_sh[4 * NC];      // [key quarter][column]: row sums
  __shared__ float cq_sh[C::NQ];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int load_items_sh[2];

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // softmax threads: key t of a tile and d index t of O^T (the warp's TMEM lane
  // quarter), query columns [cg NCW, (cg + 1) NCW)
  const int t = (warp & 3) * 32 + lane;
  const int cg = warp >> 2;
  const int split = blockIdx.x;
  const int hk = blockIdx.y;
  const int b = blockIdx.z;
  const int len = kp.seq_lens[b];
  if (len < 0 || len > kp.max_pages * kp.page_size) {
    if (threadIdx.x == 0) atomicCAS(kp.status, 0, kDevBadSeqlens);
    return;
  }
  const int ntiles = (len + DBN - 1) / DBN;
  const int j0 = split * kp.tiles_per_split;
  const int nK = max(0, min(ntiles, j0 + kp.tiles_per_split) - j0);
  // the R rows of this key/value head are contiguous in [B, H, n_q]
  const size_t prow0 = (static_cast<size_t>(b) * kp.H + static_cast<size_t>(hk) * kp.group) * kp.n_q;
  if (nK == 0) {
    if (threadIdx.x < kp.rows_real) kp.lse_part[(prow0 + threadIdx.x) * kp.splits + split] = -INFINITY;
    return;
  }
  const int total_items = 2 * nK;

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&q8_full, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 32 * C::SOFTMAX_WARPS);
      mbar_init(&red_full[i], 32 * C::SOFTMAX_WARPS);
    }
    mbar_init(&fin_bar, 32 * C::SOFTMAX_WARPS);
    mbar_init(&o_full, 1);
    for (int sl = 0; sl < NSLOT; ++sl) {
      mbar_init(&kv_full[sl], 1);
      mbar_init(&kv_empty[sl], 1);
    }
    mbar_init(&drain_bar[0], 1);
    mbar_init(&drain_bar[1], 1);
    abort_sh = 0;
    load_items_sh[0] = load_items_sh[1] = 0;
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const Abort ab{&abort_sh, kp.status};
  const int* table = kp.block_table + static_cast<size_t>(b) * kp.max_pages;
  auto full_parity = [](int i) -> uint32_t { return static_cast<uint32_t>(i / NSLOT) & 1u; };

  if (warp == C::LOAD_WARP || warp == C::LOAD_V_WARP) {
    // ------------------------------------------------------------ producers
    const int kv_own = warp == C::LOAD_WARP ? 0 : 1;
    if (lane == 0 && kv_own == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(&q_full, 2 * C::CHUNK16);
#pragma unroll
      for (int c = 0; c < 2; ++c)
        tma_load_3d(sQ16 + c * C::CHUNK16, &tmQ, &q_full, c * 64, hk * kp.rows_real, b);
    }
    decode_produce<NSLOT, 1, 0, C::TILE8, 0>(&tmK, &tmV, sKV, kv_full, kv_empty, kp, table, j0, nK,
                                             len, hk, lane, ab, kv_own, load_items_sh);
  } else if (warp == C::MMA_WARP || warp == C::MMA_S_WARP) {
    // ------------------------------------------------------------ MMA issue
    // Two issuing threads: the score products and the P V products.  Issuing
    // a product or a commit costs the issuing thread tens to a hundred cycles
    // (measured), which with one thread for both bounded the tile rate.
    //  * S(j) waits for K_j and for P V(j - 2) (so the softmax has read S(j - 2)
    //    from the same TMEM buffer and P V(j - 2) has read the P'^T tile that
    //    the softmax of tile j overwrites); one commit on s_full[j % 2].
    //  * P V(j) waits for V_j and the softmax's P'(j); one commit on the value
    //    slot's empty barrier, whose phase also tells the softmax (rescale of
    //    O^T) and the score issuer that P V(j) has landed.  Key slots are
    //    released by the softmax once it has seen S(j).
    auto v_done_parity = [](int jj) -> uint32_t { return static_cast<uint32_t>((2 * jj + 1) / NSLOT) & 1u; };
    if (lane == 0 && warp == C::MMA_S_WARP) {
      constexpr uint32_t idS = idesc_e4m3(128, C::NQ, false, false);
      const uint64_t qdesc = sdesc_sw128(smem_u32(sQ8), 16, 1024);           // B: query rows, K-major
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(sKV), 16, 1024);          // A: keys, K-major
      bool ok = mbar_wait(&q8_full, 0, ab, kDevTimeoutMma);
      for (int jj = 0; jj < nK && ok; ++jj) {
        const int item = 2 * jj;
        const int slot = item % NSLOT;
        if (!(ok = mbar_wait(&kv_full[slot], full_parity(item), ab, kDevTimeoutMma))) break;
        if (jj >= 2 &&
            !(ok = mbar_wait(&kv_empty[(2 * jj - 3) % NSLOT], v_done_parity(jj - 2), ab, kDevTimeoutMma)))
          break;
        tc_fence_after_sync();
        const uint64_t kdesc = opaque(sdesc_add(kdesc0, slot * C::TILE8));
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
          mma_f8_ss(tmem + C::S_COL(jj & 1), sdesc_add(kdesc, kk * 32), sdesc_add(qdesc, kk * 32), idS,
                    kk > 0 ? 1u : 0u);
        mma_commit(&s_full[jj & 1]);
      }
    } else if (lane == 0) {
      constexpr uint32_t idPV = idesc_e4m3(128, C::NQ, true, false);
      const uint64_t pdesc0 = sdesc_sw128(smem_u32(sP), 16, 1024);           // B: P'^T rows, K-major
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(sKV), C::TILE8, 1024);    // A: V^T, MN-major
      bool ok = true;
      for (int j = 0; j < nK && ok; ++j) {
        const int item = 2 * j + 1;
        const int slot = item % NSLOT;
        if (!(ok = mbar_wait(&kv_full[slot], full_parity(item), ab, kDevTimeoutMma))) break;
        const uint64_t vdesc = opaque(sdesc_add(vdesc0, slot * C::TILE8));
        if (!(ok = mbar_wait(&p_full[j & 1], (j >> 1) & 1, ab, kDevTimeoutMma))) break;
        tc_fence_after_sync();
        const uint64_t pdesc = sdesc_add(pdesc0, (j & 1) * C::CHUNK16);
#pragma unroll
        for (int kk = 0; kk < DBN / 32; ++kk)
          mma_f8_ss(tmem + C::O_COL, sdesc_add(vdesc, kk * 32 * 128), sdesc_add(pdesc, kk * 32), idPV,
                    (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&kv_empty[slot]);   // every use of a value slot gets its phase
        if (j == nK - 1) mma_commit(&o_full);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    // ---- quantise the query rows: 8 threads per row, 16 columns each (the
    // first four softmax warps)
    if (cg == 0) {
      const int qn = t >> 3, qp = t & 7;
      if (__any_sync(0xffffffffu, !mbar_wait(&q_full, 0, ab, kDevTimeoutSoftmax))) {
        ok = false;
      } else {
        float x[16];
        const uint8_t* src = sQ16 + (qp >> 2) * C::CHUNK16 + qn * 128;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int unit = 2 * (qp & 3) + u;
          const uint4 w = *reinterpret_cast<const uint4*>(src + ((unit ^ (qn & 7)) << 4));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 f;
            if (FP16) f = __half22float2(*reinterpret_cast<const __half2*>(&ws[e]));
            else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e]));
            x[8 * u + 2 * e] = f.x;
            x[8 * u + 2 * e + 1] = f.y;
          }
        }
        if (kp.signs) {
          // x -> (x o signs) H_d / sqrt(d): butterflies of span 1..8 inside the
          // thread, 16..64 between the lanes t ^ 1, t ^ 2, t ^ 4 of the row
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 sg = __ldg(reinterpret_cast<const float4*>(kp.signs + 16 * qp + i));
            x[i] *= sg.x;
            x[i + 1] *= sg.y;
            x[i + 2] *= sg.z;
            x[i + 3] *= sg.w;
          }
#pragma unroll
          for (int h = 1; h < 16; h <<= 1)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if ((i & h) == 0) {
                const float a = x[i], bb = x[i + h];
                x[i] = a + bb;
                x[i + h] = a - bb;
              }
#pragma unroll
          for (int h = 1; h < 8; h <<= 1) {
            const bool upper = (qp & h) != 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float o = __shfl_xor_sync(0xffffffffu, x[i], h);
              x[i] = upper ? o - x[i] : x[i] + o;
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] *= 0.08838834764831845f;   // 1 / sqrt(128)
        }
        float am = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(x[i]));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
        const bool real = qn < kp.rows_real;
        // descale = amax / 448, code = e4m3(x / descale) with the quotient
        // rounded as an IEEE float32 division (the block quantiser's rule)
        const float dq = (real && am > 0.f) ? __fdiv_rn(am, 448.f) : 1.f;
        const float yq = __fdiv_rn(1.f, dq);
        uint32_t wq[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          wq[e] = real ? cvt_pack_e4m3x4(div_by_recip(x[4 * e], dq, yq), div_by_recip(x[4 * e + 1], dq, yq),
                                         div_by_recip(x[4 * e + 2], dq, yq), div_by_recip(x[4 * e + 3], dq, yq))
                       : 0u;
        st_shared_v4(smem_u32(sQ8 + qn * 128 + ((qp ^ (qn & 7)) << 4)), wq[0], wq[1], wq[2], wq[3]);
        if (qp == 0) cq_sh[qn] = real ? kp.scale_log2 * dq : 0.f;
        // both P'^T tiles start zero: rows at or past NC are never written
        st_shared_v4(smem_u32(sP + t * 32), 0u, 0u, 0u, 0u);
        st_shared_v4(smem_u32(sP + t * 32 + 16), 0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        mbar_arrive(&q8_full);
      }
    }
    float cq[NCW];     // scale * log2(e) * dq of each query row (0: padding)
    int vend[NCW];     // keys [0, vend) visible to each query row (0: padding)
    float m_ref[NCW];  // running maximum of y = s + log2(dv), log2 units
    float lsum[NCW];   // this thread's share of the row sums of 2^(s - m_ref)
    if (ok && __any_sync(0xffffffffu, !mbar_wait(&q8_full, 0, ab, kDevTimeoutSoftmax))) ok = false;
#pragma unroll
    for (int n = 0; n < NCW; ++n) {
      const int nc = cg * NCW + n;
      cq[n] = cq_sh[nc];
      const int tq = nc % kp.n_q;
      vend[n] = nc < kp.rows_real ? (kp.causal ? min(len, len - kp.n_q + tq + 1) : len) : 0;
      m_ref[n] = -INFINITY;
      lsum[n] = 0.f;
    }
    // ---- descales of this thread's key.  U register sets, one per tile
    // residue mod U, with the loop unrolled by U: a tile's descales are loaded
    // U tiles before use and its block-table entry U tiles before that, and no
    // register copy waits on a load in flight (with one set rotated by copies,
    // the copy stalled on the load a tile later).  U = 2 for 16 columns, where
    // three copies of the larger loop body ran slower.
    auto page_of = [&](int jj) -> int {
      const int tok = (j0 + jj) * DBN + t;
      if (jj >= nK || tok >= len) return -1;
      return __ldg(table + (tok >> kp.page_shift));   // range-checked when used
    };
    auto dk_of = [&](int ph) -> float {
      return (ph < 0 || ph >= kp.num_pages) ? 1.f : __ldg(kp.k_descale + static_cast<size_t>(ph) * kp.H_kv + hk);
    };
    auto dv_of = [&](int ph) -> float {
      return (ph < 0 || ph >= kp.num_pages) ? 1.f : __ldg(kp.v_descale + static_cast<size_t>(ph) * kp.H_kv + hk);
    };
    constexpr int U = NCW >= 16 ? 2 : 3;
    float dk0 = dk_of(page_of(0)), dv0 = dv_of(page_of(0));
    float dk1 = dk_of(page_of(1)), dv1 = dv_of(page_of(1));
    float dk2 = U > 2 ? dk_of(page_of(2)) : 1.f, dv2 = U > 2 ? dv_of(page_of(2)) : 1.f;
    int ph0 = page_of(U), ph1 = page_of(U + 1), ph2 = U > 2 ? page_of(U + 2) : -1;

    auto tile_step = [&](const int j, float& dk_cur, float& dv_cur, int& ph_next) -> bool {
      const float lgv = lg2_dec(dv_cur);
      float inv_dv;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv_dv) : "f"(dv_cur));
      float coef[NCW];
#pragma unroll
      for (int n = 0; n < NCW; ++n) coef[n] = cq[n] * dk_cur;
      if (__any_sync(0xffffffffu, !mbar_wait(&s_full[j & 1], (j >> 1) & 1, ab, kDevTimeoutSoftmax))) {
        return false;
      }
      tc_fence_after_sync();
      uint32_t sr[NCW];
      tmem_ld_cols<NCW>(tmem + lane_addr + C::S_COL(j & 1) + cg * NCW, sr);
      // S(j) has completed: K_j's slot is free
      if (threadIdx.x == 0 && 2 * j + NSLOT < total_items) mbar_arrive(&kv_empty[(2 * j) % NSLOT]);
      tmem_ld_wait();
      const int key = (j0 + j) * DBN + t;
      float y[NCW];
#pragma unroll
      for (int n = 0; n < NCW; ++n)
        y[n] = key < vend[n] ? fmaf(__uint_as_float(sr[n]), coef[n], lgv) : -INFINITY;
      // column maxima over the tile's 128 keys: per warp, then across warps
      float wmax[NCW];
#pragma unroll
      for (int n = 0; n < NCW; ++n) asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(wmax[n]) : "f"(y[n]));
      if (lane == 0) {
#pragma unroll
        for (int n = 0; n < NCW; n += 4)
          *reinterpret_cast<float4*>(&red_sh[j & 1][(warp & 3) * NC + cg * NCW + n]) =
              make_float4(wmax[n], wmax[n + 1], wmax[n + 2], wmax[n + 3]);
      }
      mbar_arrive(&red_full[j & 1]);
      if (__any_sync(0xffffffffu, !mbar_wait(&red_full[j & 1], (j >> 1) & 1, ab, kDevTimeoutSoftmax))) {
        return false;
      }
      // The reference follows the running maximum exactly (no lazy slack), so
      // the largest weight of a row is exactly 1, which e4m3 holds exactly.
      float alpha[NCW];
      bool grew = false;
#pragma unroll
      for (int n4 = 0; n4 < NCW; n4 += 4) {
        float4 r4[4];
#pragma unroll
        for (int w = 0; w < 4; ++w)
          r4[w] = *reinterpret_cast<const float4*>(&red_sh[j & 1][w * NC + cg * NCW + n4]);
        const float mt[4] = {fmaxf(fmaxf(r4[0].x, r4[1].x), fmaxf(r4[2].x, r4[3].x)),
                             fmaxf(fmaxf(r4[0].y, r4[1].y), fmaxf(r4[2].y, r4[3].y)),
                             fmaxf(fmaxf(r4[0].z, r4[1].z), fmaxf(r4[2].z, r4[3].z)),
                             fmaxf(fmaxf(r4[0].w, r4[1].w), fmaxf(r4[2].w, r4[3].w))};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = n4 + i;
          alpha[n] = 1.f;
          if (mt[i] > m_ref[n]) {
            alpha[n] = ex2_approx(m_ref[n] - mt[i]);   // 0 while m_ref = -inf
            m_ref[n] = mt[i];
            grew = true;
          }
        }
      }
      // weights P' = 2^(y - m) <= 1, e4m3 codes into row n of P'^T (key t)
      float pw[NCW];
#pragma unroll
      for (int n = 0; n < NCW; ++n) {
        const float off = (m_ref[n] == -INFINITY ? 0.f : -m_ref[n]) + lgv;
        pw[n] = key < vend[n] ? ex2_approx(fmaf(__uint_as_float(sr[n]), coef[n], off)) : 0.f;
        lsum[n] = fmaf(pw[n], inv_dv, lsum[n] * alpha[n]);
      }
      const uint32_t pbase = smem_u32(sP + (j & 1) * C::CHUNK16) + (t & 15);
#pragma unroll
      for (int n = 0; n < NCW; n += 2) {
        const int nc = cg * NCW + n;
        uint16_t pr;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pr) : "f"(pw[n + 1]), "f"(pw[n]));
        st_shared_u8(pbase + nc * 128 + ((((t >> 4) ^ nc) & 7) << 4), pr & 0xFFu);
        st_shared_u8(pbase + (nc + 1) * 128 + ((((t >> 4) ^ (nc + 1)) & 7) << 4), pr >> 8);
      }
      if (j > 0 && __any_sync(0xffffffffu, grew)) {
        // rescale O^T by alpha once P V(j - 1) has landed (the phase of its
        // value slot's empty barrier)
        if (__any_sync(0xffffffffu, !mbar_wait(&kv_empty[(2 * j - 1) % NSLOT],
                                               static_cast<uint32_t>((2 * j - 1) / NSLOT) & 1u, ab,
                                               kDevTimeoutSoftmax))) {
          return false;
        }
        tc_fence_after_sync();
        uint32_t o[NCW];
        tmem_ld_cols<NCW>(tmem + lane_addr + C::O_COL + cg * NCW, o);
        tmem_ld_wait();
#pragma unroll
        for (int n = 0; n < NCW; ++n) o[n] = __float_as_uint(__uint_as_float(o[n]) * alpha[n]);
        tmem_st_cols<NCW>(tmem + lane_addr + C::O_COL + cg * NCW, o);
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&p_full[j & 1]);
      // descales of tile j + U (same register set), block-table entry of tile j + 2 U
      dk_cur = dk_of(ph_next);
      dv_cur = dv_of(ph_next);
      ph_next = page_of(j + 2 * U);
      return true;
    };
    for (int j = 0; j < nK && ok; j += U) {
      if (!(ok = tile_step(j, dk0, dv0, ph0)) || j + 1 >= nK) break;
      if constexpr (U == 2) {
        ok = tile_step(j + 1, dk1, dv1, ph1);
      } else {
        if (!(ok = tile_step(j + 1, dk1, dv1, ph1)) || j + 2 >= nK) break;
        ok = tile_step(j + 2, dk2, dv2, ph2);
      }
    }
    // ------------------------------------------------------------ epilogue
    if (ok && !__any_sync(0xffffffffu, !mbar_wait(&o_full, 0, ab, kDevTimeoutEpilogue))) {
      tc_fence_after_sync();
      uint32_t o[NCW];
      tmem_ld_cols<NCW>(tmem + lane_addr + C::O_COL + cg * NCW, o);
      tmem_ld_wait();
      int col;
      const float wsum = warp_col_reduce<NCW>(lsum, lane, AddOp{}, &col);
      fin_sh[(warp & 3) * NC + cg * NCW + col] = wsum;
      mbar_arrive(&fin_bar);
      if (!__any_sync(0xffffffffu, !mbar_wait(&fin_bar, 0, ab, kDevTimeoutEpilogue))) {
#pragma unroll
        for (int n = 0; n < NCW; ++n) {
          const int nc = cg * NCW + n;
          if (nc >= kp.rows_real) break;
          const float l = ((fin_sh[nc] + fin_sh[NC + nc]) + fin_sh[2 * NC + nc]) + fin_sh[3 * NC + nc];
          const float inv_l = l > 0.f ? 1.f / l : 0.f;
          const size_t pr = (prow0 + nc) * kp.splits + split;
          kp.o_part[pr * D + t] = __uint_as_float(o[n]) * inv_l;
          if (t == 0) kp.lse_part[pr] = l > 0.f ? (m_ref[n] + lg2_dec(l)) * 0.69314718055994530942f : -INFINITY;
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (abort_sh) {
    if ((warp == C::LOAD_WARP || warp == C::LOAD_V_WARP) && lane == 0) {
      const int kv_own = warp == C::LOAD_WARP ? 0 : 1;
      if (kv_own == 0) mbar_wait_drain(&q_full, 0);
      decode_drain_items<NSLOT, 0>(kv_full, load_items_sh[kv_own], kv_own, full_parity);
    }
    if ((warp == C::MMA_WARP || warp == C::MMA_S_WARP) && lane == 0) {
      uint64_t* bar = &drain_bar[warp == C::MMA_WARP ? 0 : 1];
      mma_commit(bar);
      mbar_wait_drain(bar, 0);
    }
    __syncthreads();
  }
  if (warp == C::MMA_WARP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <bool FP16, int NC, int CW>
attn_status_t launch_decode_fp8_keys(const DecodeParams& p, const DecKParams& kp, const DecodeSplits& sp,
                                     const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  using C = Dec8TCfg<CW>;
  auto kern = decode_fp8_keys_kernel<FP16, NC, CW>;
  attn_status_t s = set_smem(reinterpret_cast<const void*>(kern), C::SMEM);
  if (s != ATTN_OK) return s;
  CUtensorMap tq;
  // Q: {d, H * n_q rows, B}, boxes of 16 rows: the R rows of head hk from row hk * R
  if ((s = make_tmap_3d(&tq, p.q, 2, C::D, static_cast<uint64_t>(p.H) * p.n_q, p.B, 64, C::NQ)) != ATTN_OK)
    return s;
  kern<<<dim3(sp.splits, p.H_kv, p.B), C::THREADS, C::SMEM, stream>>>(tq, tk, tv, kp);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "FP8 decode split kernel launch");
  return ATTN_OK;
}

template <bool FP16>
attn_status_t launch_decode_fp8_t(const DecodeParams& p, cudaStream_t stream) {
  using C = Dec8Cfg;
  auto kern = decode_fp8_split_kernel<FP16>;
  attn_status_t s = set_smem(reinterpret_cast<const void*>(kern), C::SMEM);
  if (s != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
  if ((s = make_tmap_3d(&tq, p.q, 2, C::D, static_cast<uint64_t>(p.H) * p.n_q, p.B, 64, DBM)) != ATTN_OK)
    return s;
  // e4m3 cache: {d, page_size, H_kv, num_pages}, one 128-byte row per token
  const int box_rows = p.page_size < DBN ? p.page_size : DBN;
  const uint64_t tok_b = static_cast<uint64_t>(p.H_kv) * C::D, head_b = C::D, page_b = tok_b * p.page_size;
  if ((s = make_tmap_4d(&tk, p.k_cache, 1, C::D, p.page_size, p.H_kv, p.num_pages, tok_b, head_b, page_b,
                        C::D, box_rows)) != ATTN_OK)
    return s;
  if ((s = make_tmap_4d(&tv, p.v_cache, 1, C::D, p.page_size, p.H_kv, p.num_pages, tok_b, head_b, page_b,
                        C::D, box_rows)) != ATTN_OK)
    return s;
  int* status = device_status_word();
  if (!status) return fail(ATTN_ERR_CUDA, "status word unavailable");
  const DecodeSplits sp = decode_splits(p.B, p.H_kv, p.max_seqlen);
  int shift = 0;
  while ((1 << shift) < p.page_size) ++shift;
  DecKParams kp{p.block_table, p.seq_lens, p.o_part,  p.lse_part,  status,
                p.H,           p.H / p.H_kv, p.n_q,   (p.H / p.H_kv) * p.n_q,
                p.max_pages,   p.page_size, box_rows, p.num_pages,
                sp.splits,     sp.tiles_per_split, p.causal, p.scale * 1.4426950408889634f,
                p.k_descale,   p.v_descale, p.signs, p.H_kv, shift};
  const int rows_real = (p.H / p.H_kv) * p.n_q;
  if (rows_real <= Dec8TCfg<1>::NQ) {
    // up to 4 query rows: one softmax warp per key quarter; more: two, each
    // taking half of the query columns
    s = rows_real <= 4   ? launch_decode_fp8_keys<FP16, 4, 1>(p, kp, sp, tk, tv, stream)
        : rows_real <= 8 ? launch_decode_fp8_keys<FP16, 8, 2>(p, kp, sp, tk, tv, stream)
                         : launch_decode_fp8_keys<FP16, 16, 2>(p, kp, sp, tk, tv, stream);
    if (s != ATTN_OK) return s;
  } else {
    kern<<<dim3(sp.splits, p.H_kv, p.B), C::THREADS, C::SMEM, stream>>>(tq, tk, tv, kp);
    const cudaError_t e0 = cudaGetLastError();
    if (e0 != cudaSuccess) return fail_cuda(e0, "FP8 decode split kernel launch");
  }
  cudaError_t e = cudaSuccess;
  const long long rows = static_cast<long long>(p.B) * p.H * p.n_q;
  decode_combine_kernel<128, FP16><<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, stream>>>(
      p.o_part, p.lse_part, static_cast<uint16_t*>(p.o), p.lse, rows, sp.splits);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "decode combine kernel launch");
  return ATTN_OK;
}

template <int D, bool FP16>
attn_status_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  using C = DecCfg<D>;
  auto kern = decode_split_kernel<D, FP16>;
  attn_status_t s = set_smem(reinterpret_cast<const void*>(kern), C::SMEM);
  if (s != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
  // Q: {d, H * n_q rows, B}: the query tile of key/value head hk starts at row
  // hk * G * n_q
  if ((s = make_tmap_3d(&tq, p.q, 2, D, static_cast<uint64_t>(p.H) * p.n_q, p.B, 64, DBM)) != ATTN_OK)
    return s;
  // cache: {d, page_size, H_kv, num_pages}, one box per page (or per 128 rows)
  const int box_rows = p.page_size < DBN ? p.page_size : DBN;
  const uint64_t tok_b = 2ull * p.H_kv * D, head_b = 2ull * D, page_b = tok_b * p.page_size;
  if ((s = make_tmap_4d(&tk, p.k_cache, 2, D, p.page_size, p.H_kv, p.num_pages, tok_b, head_b, page_b, 64,
                        box_rows)) != ATTN_OK)
    return s;
  if ((s = make_tmap_4d(&tv, p.v_cache, 2, D, p.page_size, p.H_kv, p.num_pages, tok_b, head_b, page_b, 64,
                        box_rows)) != ATTN_OK)
    return s;
  int* status = device_status_word();
  if (!status) return fail(ATTN_ERR_CUDA, "status word unavailable");
  const DecodeSplits sp = decode_splits(p.B, p.H_kv, p.max_seqlen);
  int shift = 0;
  while ((1 << shift) < p.page_size) ++shift;
  DecKParams kp{p.block_table, p.seq_lens, p.o_part,  p.lse_part,  status,
                p.H,           p.H / p.H_kv, p.n_q,   (p.H / p.H_kv) * p.n_q,
                p.max_pages,   p.page_size, box_rows, p.num_pages,
                sp.splits,     sp.tiles_per_split, p.causal, p.scale * 1.4426950408889634f,
                nullptr,       nullptr,     nullptr, p.H_kv, shift};
  kern<<<dim3(sp.splits, p.H_kv, p.B), C::THREADS, C::SMEM, stream>>>(tq, tk, tv, kp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "decode split kernel launch");
  const long long rows = static_cast<long long>(p.B) * p.H * p.n_q;
  decode_combine_kernel<D, FP16><<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, stream>>>(
      p.o_part, p.lse_part, static_cast<uint16_t*>(p.o), p.lse, rows, sp.splits);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "decode combine kernel launch");
  return ATTN_OK;
}

}  // namespace

attn_status_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.B > 65535 || p.H_kv > 65535) return fail(ATTN_ERR_UNSUPPORTED, "grid dimension limit exceeded");
  if (p.fp8) {
    if (p.d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 decode supports d = 128");
    return p.fp16 ? launch_decode_fp8_t<true>(p, stream) : launch_decode_fp8_t<false>(p, stream);
  }
  switch (p.d) {
    case 64: return p.fp16 ? launch_decode_t<64, true>(p, stream) : launch_decode_t<64, false>(p, stream);
    case 128: return p.fp16 ? launch_decode_t<128, true>(p, stream) : launch_decode_t<128, false>(p, stream);
  }
  return fail(ATTN_ERR_UNSUPPORTED, "decode supports d = 64 and 128");
}

}  // namespace attn
