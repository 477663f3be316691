// gated_attention_pair.cu — K6, causal grouped-query attention with the
// sigmoid output gate of the Qwen3-Next / Qwen3.5 global-attention layer
// (head_dim 256), on pairs of CTAs sharing one tcgen05 MMA stream.
//
// For every query row (b, i, h), with the normalised, partially rotated qhat
// and keys khat_j of group h / g:
//   z = sigmoid(gate[b, i, h, :]) * sum_{j <= i} softmax_j(qhat . khat_j / 16) v_j
// ("Chapter 20, Qwen3 and Qwen3.5" §20.4: the attention output is multiplied
// elementwise by the sigmoid of the gate half of the query projection before
// the output projection; "14. The Qwen family", Qwen3-Next section.)
//
// Why pairs. With d = 256 a 128-row Q tile is 64 KB of shared memory and its
// fp32 O tile 256 of the 512 TMEM columns, so a CTA holds one Q tile, and a
// lone CTA's QK^T runs as small-N MMAs whose cost is dominated by the
// per-instruction operand reads. A cluster of two CTAs issues M = 256 MMAs
// (tcgen05.mma.cta_group::2): each CTA holds its own 128 query rows (A) and
// half of every K/V tile (B), so QK^T runs as N = 128 steps and PV as N = 256
// steps, each CTA loads half the K/V bytes, and a 128-key tile costs each CTA
// 64 KB of its ring.
//
// Tiling. The pair owns 256 query rows: two 128-row tiles of the g heads of one
// KV group for floor(128/g) consecutive tokens each, packed row r = (token r/g,
// head kv*g + r%g) by a 4-D TMA box; the even CTA holds the first tile. When g
// does not divide 128 (g = 6, 12) the last 128 - g*floor(128/g) rows of a
// tile are padding: computed on stale shared memory, never stored. KV tiles are
// 128 keys. CTA c holds keys 64c..64c+63 of each K tile (four 8 KB blocks of
// 64 dims) and dims 128c..128c+127 of each V tile (two 16 KB blocks of 64
// dims), in a ring of four 32 KB slots, loaded in the order the MMAs read them
// (K_0, K_1, V_0, K_2, V_1, ...).
//
// Persistence. The plain prefill runs one pair per two SMs, each walking its
// work items (a 256-row pair tile of one KV group, longest first) in rounds
// of the number of pairs, in snake order. The MMA stream runs on across
// items: the next item's Q tiles load once the item's last QK^T has completed
// ("Q free", committed to both CTAs), the ring, the S buffers and every
// barrier phase continue, and the next item's first PV waits only for every
// softmax warp of the pair to have read O ("O free"). A chunk against the
// caches runs the same way.
//
// Roles (640 threads per CTA):
//   WG 0..3  softmax + epilogue of the CTA's own 128 rows. Warp w serves TMEM
//            lanes 32(w%4).. and the key quarter c = w/4 of every S tile (32
//            keys), and O columns 64c..64c+63 in the epilogue;
//   warp 16  TMA producer of the CTA's Q tile and ring;
//   warp 17  (even CTA) the MMA issuer of the pair;
//   warp 18  (odd CTA) forwards its ring's "tile landed" events to the even
//            CTA, whose MMA issuer waits for both halves;
//   warp 19  hands ring slots back to the producer as soon as the MMAs that
//            read them complete: K_j's when S_j completes, V_j's when PV_j
//            does (an arrive on "PV done" follows every PV).
// TMEM per CTA: S0 | S1 (128 fp32 columns each, double-buffered) | O (256).
// "P ready" and "O free" are the even CTA's barriers: its own softmax warps
// arrive with CTA scope, the odd CTA's with cluster scope, all relaxed (the
// payload is tensor memory the warp has finished with, so nothing needs
// releasing, and a release would make each warp wait for its earlier global
// stores: the odd CTA's on every tile, both CTAs' after the epilogue).
// P goes back as bf16 pairs over the first half of each thread's own S
// columns and PV reads it from there. MMA stream: S_0, S_1, then per KV tile
// j: PV_j, S_{j+2}. Commits arrive on the barriers of both CTAs.
//
// Softmax: fixed shift from the norm's logit bound (16 max|1 + w_q|
// max|1 + w_k|, written by the prologue), or above its limit an online max
// exchanged between the four key quarters of a row, with O rescaled in TMEM
// after the previous PV has completed.
//
// A chunk against the caches ("Chapter 20, Qwen3 and Qwen3.5" §20.3: cached
// keys followed by the chunk's own, a causal mask that starts at the chunk's
// first position) is the same kernel with K and V read from the head-major
// caches and a per-sequence start position p0: token t sees keys 0..p0 + t.
// Rows of the last V tile past p0 + T hold whatever the cache holds there (a
// NaN there would turn a zero weight into a NaN in PV), so each CTA's producer
// warp clears them in its own V half once that tile has landed; the odd CTA
// then forwards "tail cleared" instead of "tile landed" for that load, and the
// MMA issuer waits for the even CTA's own "tail cleared".
//
// Every mbarrier wait is bounded; a timeout sets the error word and every
// role unwinds; the MMA issuer drains its MMAs and both CTAs meet at a cluster
// barrier before freeing tensor memory.
#include <type_traits>

#include "q3a_internal.h"
#include "q3a_pair.cuh"

namespace q3a {

namespace {

constexpr int BM = 128;  // query rows per CTA (256 per pair)
constexpr int BN = 128;  // keys per KV tile
constexpr int D = kGatedD;
constexpr int kSoftmaxWGs = 4;
constexpr int kThreads = (kSoftmaxWGs + 1) * 128;
constexpr int kSlots = 4;
constexpr uint32_t kQBlock = 16384;  // 128 rows x 128 bytes: 64 dims of the Q tile
constexpr uint32_t kKBlock = 8192;   // 64 keys x 128 bytes: 64 dims of a K half tile
constexpr uint32_t kVBlock = 16384;  // 128 keys x 128 bytes: 64 dims of a V half tile
constexpr uint32_t kSlotBytes = 32768;
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = OFF_Q + 4 * kQBlock;
constexpr uint32_t OFF_BAR = OFF_RING + kSlots * kSlotBytes;
// tile maxima [2 parities][4 quarters][128] fp32, then partial sums
// [2 item parities][4 quarters][128]
constexpr uint32_t OFF_XCHG = OFF_BAR + 512;
constexpr uint32_t kSmemBytes = OFF_XCHG + (2 * 4 * 128 + 2 * 4 * 128) * 4 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;
constexpr float kScaleLog2 = 0.09016844005556021f;  // log2(e) / sqrt(256)
constexpr float kRescaleThreshold = 8.0f;
constexpr float kFixedMaxLimit = 60.0f;
constexpr unsigned kFull = 0xffffffffu;

struct Bars {
  uint64_t q_full, q_peer;
  uint64_t q_empty;  // the Q tile is free again: the item's last QK^T completed
  uint64_t slot_full[kSlots], slot_peer[kSlots], slot_empty[kSlots];
  uint64_t s_full[2];
  uint64_t p_full[2];  // even CTA: all 32 softmax warps of the pair
  uint64_t pv_done;    // PV_j complete (one phase per KV tile)
  uint64_t xmax_full;  // online-max path: the CTA's four quarters posted their tile max
  uint64_t o_final;
  uint64_t o_free;   // even CTA: every softmax warp of the pair has read O
  uint64_t drain;
  uint64_t vtail;      // chunk: the last V half tile's rows past the valid keys cleared
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

__device__ __forceinline__ uint32_t slot_of(uint32_t n) { return n % kSlots; }
__device__ __forceinline__ uint32_t use_of(uint32_t n) { return (n / kSlots) & 1u; }

// S = Q K_j^T over the pair: 16 steps of 16 dims, M = 256, N = 128. Q block c
// holds dims 64c..64c+63 (16 KB apart); the K half tile's block c likewise
// (8 KB apart) in ring slot `slot`.
__device__ __forceinline__ void issue_s(uint32_t tmem_s, uint64_t q_desc, uint64_t ring_k,
                                        uint32_t slot) {
  constexpr uint32_t idesc = idesc_bf16_f32(256, BN, 0, 0);
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) {
    const int c = kk >> 2;
    const uint64_t a = q_desc + (uint64_t)((c * kQBlock + (kk & 3) * 32) >> 4);
    const uint64_t b =
        ring_k + (uint64_t)((slot * kSlotBytes + c * kKBlock + (kk & 3) * 32) >> 4);
    if (kk == 0)
      mma_pair_ss<0>(tmem_s, a, b, idesc);
    else
      mma_pair_ss<1>(tmem_s, a, b, idesc);
  }
}

// O += P_j V_j over the pair: 8 steps of 16 keys, M = 256, N = 256. P for
// keys 32q..32q+31 sits in S columns 32q..32q+15 (bf16 pairs); B = the V half
// tile, MN-major: its two 64-dim blocks 16 KB apart (the leading offset),
// 8-key groups 1 KB apart, 16 keys = 2 KB per step.
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t ring_v,
                                         uint32_t slot, bool accumulate_first) {
  constexpr uint32_t idesc = idesc_bf16_f32(256, 256, 0, 1);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint64_t b = ring_v + (uint64_t)((slot * kSlotBytes + kk * 2048) >> 4);
    mma_pair_ts(tmem_o, tmem_p + 32 * (kk >> 1) + 8 * (kk & 1), b, idesc,
                (accumulate_first || kk > 0) ? 1u : 0u);
  }
}

// The plain prefill and the chunk against the caches are two instantiations,
// so the plain one carries none of the chunk's bookkeeping.
__host__ __device__ __forceinline__ const GatedAttnArgs& base_args(const GatedAttnArgs& a) {
  return a;
}
__host__ __device__ __forceinline__ const GatedAttnArgs& base_args(const GatedAttnChunkArgs& a) {
  return a.base;
}
static GatedAttnArgs& base_args_mut(GatedAttnArgs& a) { return a; }
static GatedAttnArgs& base_args_mut(GatedAttnChunkArgs& a) { return a.base; }
__device__ __forceinline__ int chunk_start(const GatedAttnArgs&, int) { return 0; }
__device__ __forceinline__ int chunk_start(const GatedAttnChunkArgs& a, int b) {
  return a.pos_b[b];
}
__device__ __forceinline__ bool fixed_shift_allowed(const GatedAttnArgs&) { return true; }
__device__ __forceinline__ bool fixed_shift_allowed(const GatedAttnChunkArgs& a) {
  return a.fixed_shift_ok != 0;
}

template <class Args>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gated_attention_pair_kernel(const __grid_constant__ Args args) {
  constexpr bool kChunk = sizeof(Args) != sizeof(GatedAttnArgs);
  const GatedAttnArgs& a = base_args(args);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  float* xchg = reinterpret_cast<float*>(smem + OFF_XCHG);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: the even CTA, which issues the MMAs

  // ---- work items ------------------------------------------------------------
  // Item i (longest first): pair tile pm = n_mtiles - 1 - i / (B * Hkv) of
  // group (b, kv) = i % (B * Hkv); a chunk's as item_index orders them
  // (longest first within each set of groups). A pair takes items in rounds
  // of the number of pairs, in snake order (forward in even rounds, backward
  // in odd ones).
  const int bk_count = a.B * a.Hkv;
  const int n_items = a.n_mtiles * bk_count;
  const int g = a.g;
  const int tile_tok = BM / g;
  const int G = (int)(gridDim.x >> 1), c = (int)(blockIdx.x >> 1);
  auto item_of_round = [&](int r) { return r * G + ((r & 1) ? G - 1 - c : c); };
  struct Item {
    int b, kv, t0_pair, p0, n_tiles, n_keys;
  };
  auto item_at = [&](int i) {
    Item it;
    int pm, bk;
    if (kChunk) {
      // group_sets: a power of two dividing the group count
      const ItemIndex ix = item_index(i, a.n_mtiles, bk_count >> (31 - __clz(a.group_sets)));
      pm = ix.mt;
      bk = ix.bk;
    } else {
      pm = a.n_mtiles - 1 - i / bk_count;
      bk = i % bk_count;
    }
    it.b = bk / a.Hkv;
    it.kv = bk % a.Hkv;
    it.t0_pair = pm * 2 * tile_tok;
    const int t_last = min(it.t0_pair + 2 * tile_tok, a.T) - 1;
    // token t of the sequence sits at position p0 + t (p0 = 0 for a plain
    // prefill) and sees keys 0..p0+t; keys p0+T.. are not valid
    it.p0 = chunk_start(args, it.b);
    it.n_tiles = (it.p0 + t_last) / BN + 1;
    it.n_keys = it.p0 + a.T;
    return it;
  };
  const float bound = *a.logit_bound;
  const bool fixed_max = fixed_shift_allowed(args) && bound >= 0.f && bound <= kFixedMaxLimit;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_peer, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars->slot_full[s], 1);
      mbar_init(&bars->slot_peer[s], 1);
      mbar_init(&bars->slot_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 2 * kSoftmaxWGs * 4);  // one arrive per softmax warp, both CTAs
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->xmax_full, kSoftmaxWGs * 128);
    mbar_init(&bars->o_final, 1);
    mbar_init(&bars->o_free, 2 * kSoftmaxWGs * 4);  // one arrive per softmax warp, both CTAs
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->vtail, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc_pair<kTmemCols>(&bars->tmem_base);
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort_flag;

  // Per item the loads are K_0, K_1, then per KV tile j: V_j, K_{j+2}: load
  // index of K_j is 0, then 2j - 1; of V_j 2j + 2, except the last V at
  // 2n - 1. Indices below are global over the pair's items (item base L).
  if (warp >= kSoftmaxWGs * 4) {
    if (warp == kSoftmaxWGs * 4) {
      // ------------------------------------------------------------ producer
      // Lane 0 issues the loads. Chunk: an item's last V half tile may hold
      // rows past the valid keys; the whole warp clears them in this CTA's
      // half once that tile has landed and publishes it on "V tail" (one phase
      // per item that has such a tail).
      if (lane == 0) {
        tma_prefetch_desc(&a.tm_q);
        tma_prefetch_desc(&a.tm_k);
        tma_prefetch_desc(&a.tm_v);
      }
      uint32_t n = 0;    // half tiles issued (global; every lane keeps the count)
      uint32_t n_q = 0;  // Q tiles issued (lane 0)
      bool ok = kChunk || lane == 0;  // the plain prefill's loop runs on lane 0 only
      for (int r = 0; ok && item_of_round(r) < n_items; ++r) {
        const Item it = item_at(item_of_round(r));
        const int row3 = it.b * a.Hkv + it.kv;
        if (lane == 0) {
          // this CTA's Q tile, once the previous item's last QK^T has completed
          ok = n_q == 0 || mbar_wait(&bars->q_empty, (n_q - 1) & 1, a.err, kDevTimeoutTma, abort);
          if (ok) {
            // g * floor(128/g) rows of 128 bytes per 64-dim block (126 or 120
            // when g does not divide 128)
            mbar_arrive_expect_tx(&bars->q_full, 4u * (uint32_t)(g * tile_tok) * 128u);
            const int t0 = it.t0_pair + (int)rank * tile_tok;
            for (int cc = 0; cc < 4; ++cc)
              tma_load_4d(smem + OFF_Q + cc * kQBlock, &a.tm_q, &bars->q_full, 64 * cc, it.kv * g,
                          t0, it.b);
            ++n_q;  // lane 0's count
          }
        }
        uint32_t n0 = n;  // lane 0 counts its loads from here
        auto load_tile = [&](bool is_k, int j) {
          if (!ok) return;
          const uint32_t s = slot_of(n0);
          if (!mbar_wait(&bars->slot_empty[s], use_of(n0) ^ 1u, a.err, kDevTimeoutTma, abort)) {
            ok = false;
            return;
          }
          mbar_arrive_expect_tx(&bars->slot_full[s], kSlotBytes);
          uint8_t* dst = smem + OFF_RING + s * kSlotBytes;
          if (is_k) {  // keys 64 rank .. of the tile, all 256 dims
            for (int cc = 0; cc < 4; ++cc)
              tma_load_3d(dst + cc * kKBlock, &a.tm_k, &bars->slot_full[s], 64 * cc,
                          j * BN + 64 * (int)rank, row3);
          } else {  // dims 128 rank .. of the tile, all 128 keys
            for (int cc = 0; cc < 2; ++cc) {
              if (a.v_head_major)  // a V cache [B*Hkv, rows, 256]
                tma_load_3d(dst + cc * kVBlock, &a.tm_v, &bars->slot_full[s],
                            128 * (int)rank + 64 * cc, j * BN, row3);
              else  // the projection's V [B, T, Hkv, 256]
                tma_load_4d(dst + cc * kVBlock, &a.tm_v, &bars->slot_full[s],
                            128 * (int)rank + 64 * cc, it.kv, j * BN, it.b);
            }
          }
          ++n0;
        };
        if (lane == 0) {
          load_tile(true, 0);
          if (it.n_tiles > 1) load_tile(true, 1);
          for (int j = 0; ok && j < it.n_tiles; ++j) {
            load_tile(false, j);
            if (j + 2 < it.n_tiles) load_tile(true, j + 2);
          }
        }
        if (kChunk) {  // the whole warp runs the loop (it clears V tails)
          ok = __shfl_sync(kFull, ok, 0);
          n0 = __shfl_sync(kFull, n0, 0);
        }
        if (!ok) {
          n = n0;
          break;
        }
        n = n0;
        if (kChunk && it.n_tiles * BN > it.n_keys) {
          // every load of the item has been issued and none after it, so the
          // slot's barrier is in the phase of the item's last load: wait for
          // it, clear this CTA's rows past the valid keys in both 64-dim
          // blocks (a cleared row is 128 bytes whatever the swizzle), and
          // publish that
          const uint32_t tail_load = n - 1;
          const int tail_first = it.n_keys - (it.n_tiles - 1) * BN;
          ok = __all_sync(kFull, mbar_wait(&bars->slot_full[slot_of(tail_load)],
                                           use_of(tail_load), a.err, kDevTimeoutTma, abort));
          if (!ok) break;
          uint8_t* vt = smem + OFF_RING + slot_of(tail_load) * kSlotBytes;
          const int chunks = (BN - tail_first) * 16;  // 16-byte chunks, both blocks
          for (int ch = lane; ch < chunks; ch += 32) {
            const int row = tail_first + (ch >> 4), blk = (ch >> 3) & 1, q16 = ch & 7;
            *reinterpret_cast<uint4*>(vt + blk * kVBlock + row * 128 + q16 * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();  // the tensor pipe reads these rows next
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->vtail);
        }
      }
      if (lane == 0 && *abort) {
        // let every copy that was issued land before the CTA goes away
        if (n_q > 0) mbar_wait(&bars->q_full, (n_q - 1) & 1, nullptr, 0, nullptr);
        for (uint32_t i = n > (uint32_t)kSlots ? n - kSlots : 0u; i < n; ++i)
          mbar_wait(&bars->slot_full[slot_of(i)], use_of(i), nullptr, 0, nullptr);
      }
    } else if (warp == kSoftmaxWGs * 4 + 2 && lane == 0 && rank == 1) {
      // ----------------------------------------------- forwarder (odd CTA)
      // the even CTA's MMA issuer reads this CTA's Q and ring too: tell it
      // when each of them has landed, in load order
      uint32_t L = 0;
      uint32_t n_tail = 0;  // earlier items with a cleared V tail
      bool ok = true;
      for (int r = 0, k = 0; ok && item_of_round(r) < n_items; ++r, ++k) {
        const Item it = item_at(item_of_round(r));
        const bool v_tail = kChunk && it.n_tiles * BN > it.n_keys;
        const uint32_t n_loads = 2u * (uint32_t)it.n_tiles;
        if (!mbar_wait(&bars->q_full, k & 1, a.err, kDevTimeoutTma, abort)) break;
        mbar_arrive_cluster(peer_smem_addr(&bars->q_peer, 0));
        for (uint32_t t = 0; t < n_loads; ++t) {
          const uint32_t gt = L + t;
          const bool tail = v_tail && t + 1 == n_loads;
          if (!mbar_poll(tail ? &bars->vtail : &bars->slot_full[slot_of(gt)],
                         tail ? (n_tail & 1) : use_of(gt), a.err, kDevTimeoutTma, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(peer_smem_addr(&bars->slot_peer[slot_of(gt)], 0));
        }
        L += n_loads;
        if (v_tail) ++n_tail;
      }
    } else if (warp == kSoftmaxWGs * 4 + 3 && lane == 0) {
      // ------------------------------------------------------------ releaser
      // Completion order on the tensor pipe: per item S_0, then per KV tile j:
      // S_{j+1} (if any), PV_j.
      uint32_t L = 0, S = 0;  // loads and steps of the pair's earlier items
      bool ok = true;
      for (int r = 0; ok && item_of_round(r) < n_items; ++r) {
        const int n = item_at(item_of_round(r)).n_tiles;
        if (!mbar_wait_cluster(&bars->s_full[S & 1], (S >> 1) & 1, a.err, kDevTimeoutSoftmax,
                               abort))
          break;
        mbar_arrive(&bars->slot_empty[slot_of(L)]);
        for (int j = 0; j < n; ++j) {
          const uint32_t s = S + (uint32_t)j;
          if (j + 1 < n) {
            if (!mbar_wait_cluster(&bars->s_full[(s + 1) & 1], ((s + 1) >> 1) & 1, a.err,
                                   kDevTimeoutSoftmax, abort)) {
              ok = false;
              break;
            }
            mbar_arrive(&bars->slot_empty[slot_of(L + (uint32_t)(2 * j + 1))]);
          }
          if (!mbar_wait_cluster(&bars->pv_done, s & 1, a.err, kDevTimeoutSoftmax, abort)) {
            ok = false;
            break;
          }
          mbar_arrive(&bars->slot_empty[slot_of(L + (uint32_t)min(2 * j + 2, 2 * n - 1))]);
        }
        L += 2u * (uint32_t)n;
        S += (uint32_t)n;
      }
    } else if (warp == kSoftmaxWGs * 4 + 1 && lane == 0 && rank == 0) {
      // ------------------------------------------- MMA issuer (even CTA)
      const uint32_t q_addr = smem_u32(smem + OFF_Q);
      const uint32_t ring = smem_u32(smem + OFF_RING);
      const uint64_t q_desc = smem_desc_sw128(q_addr, 16, 1024);
      const uint64_t ring_k = smem_desc_sw128(ring, 16, 1024);        // K-major K halves
      const uint64_t ring_v = smem_desc_sw128(ring, kVBlock, 1024);   // MN-major V halves
      uint32_t L = 0, S = 0;  // loads and steps of the pair's earlier items
      uint32_t n_tail = 0;    // earlier items with a cleared V tail
      bool ok = true;
      for (int r = 0, k = 0; ok && item_of_round(r) < n_items; ++r, ++k) {
        const Item it = item_at(item_of_round(r));
        const int n_tiles = it.n_tiles;
        const bool v_tail = kChunk && n_tiles * BN > it.n_keys;
        const uint32_t last_load = L + 2u * (uint32_t)n_tiles - 1u;
        auto wait_tile = [&](uint32_t t) {  // both CTAs' halves of (global) load t
          const bool tail = v_tail && t == last_load;
          return mbar_wait_cluster(tail ? &bars->vtail : &bars->slot_full[slot_of(t)],
                                   tail ? (n_tail & 1) : use_of(t), a.err, kDevTimeoutMma,
                                   abort) &&
                 mbar_wait_cluster(&bars->slot_peer[slot_of(t)], use_of(t), a.err,
                                   kDevTimeoutMma, abort);
        };
        // An mbarrier wait issued after a tcgen05.commit stalls this thread
        // until the commit resolves. The waits for a PV's inputs (P, V and the
        // K tile after next) are therefore placed after the queued MMAs that
        // keep the tensor pipe busy meanwhile, and before the commit that
        // publishes S_{j+2}: that commit only gates softmax j+2, which cannot
        // start before softmax j+1 has produced P_{j+1} anyway. Before the
        // item's first PV, O must have been read by the previous epilogue.
        auto wait_pv_inputs = [&](int j, uint32_t t) {
          const uint32_t s = S + (uint32_t)j;
          return mbar_wait_cluster(&bars->p_full[s & 1], (s >> 1) & 1, a.err, kDevTimeoutMma,
                                   abort) &&
                 wait_tile(t) &&
                 (j > 0 || k == 0 ||
                  mbar_wait_cluster(&bars->o_free, (k - 1) & 1, a.err, kDevTimeoutMma, abort));
        };
        // load index of K_j: 0, then 2j - 1
        auto k_load = [&](int j) { return L + (j == 0 ? 0u : (uint32_t)(2 * j - 1)); };
        auto s_col = [&](int j) { return tmem + ((S + (uint32_t)j) & 1u) * BN; };
        uint32_t n = L;  // loads consumed
        ok = mbar_wait_cluster(&bars->q_full, k & 1, a.err, kDevTimeoutMma, abort) &&
             mbar_wait_cluster(&bars->q_peer, k & 1, a.err, kDevTimeoutMma, abort) &&
             wait_tile(n);
        if (!ok) break;
        tc_fence_after();
        issue_s(s_col(0), q_desc, ring_k, slot_of(n));
        n += 1;
        if (n_tiles > 1) {
          ok = wait_tile(n);  // K_1
          mma_commit_pair(&bars->s_full[S & 1]);
          if (!ok) break;
          tc_fence_after();
          issue_s(s_col(1), q_desc, ring_k, slot_of(n));
          n += 1;
          ok = wait_pv_inputs(0, n) && (n_tiles <= 2 || wait_tile(k_load(2)));
          mma_commit_pair(&bars->s_full[(S + 1) & 1]);
          if (n_tiles == 2) mma_commit_pair(&bars->q_empty);  // the item's last QK^T
        } else {
          mma_commit_pair(&bars->s_full[S & 1]);
          mma_commit_pair(&bars->q_empty);  // the item's last QK^T
          ok = wait_pv_inputs(0, n);
        }
        for (int j = 0; ok && j < n_tiles; ++j) {
          // P_j, V_j (load n) and K_{j+2} (load n + 1) have been waited for
          tc_fence_after();
          issue_pv(tmem + kTmemO, s_col(j), ring_v, slot_of(n), j > 0);
          n += 1;
          mma_commit_pair(&bars->pv_done);
          const bool next_s = j + 2 < n_tiles;
          if (next_s) {
            issue_s(s_col(j), q_desc, ring_k, slot_of(n));
            n += 1;
          }
          if (j + 1 < n_tiles)  // P_{j+1}, V_{j+1}, K_{j+3}
            ok = wait_pv_inputs(j + 1, n) && (j + 3 >= n_tiles || wait_tile(k_load(j + 3)));
          if (next_s) {
            mma_commit_pair(&bars->s_full[(S + (uint32_t)j) & 1]);
            if (j + 3 == n_tiles) mma_commit_pair(&bars->q_empty);  // the item's last QK^T
          }
        }
        if (ok) mma_commit_pair(&bars->o_final);
        L += 2u * (uint32_t)n_tiles;
        S += (uint32_t)n_tiles;
        if (v_tail) ++n_tail;
      }
      // drain: every MMA issued above has completed once this phase completes
      mma_commit_pair(&bars->drain);
      mbar_wait_cluster(&bars->drain, 0, nullptr, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int lq = warp & 3;   // TMEM lane quarter: rows 32 lq ..
    const int cq = warp >> 2;  // key quarter of each S tile (32 keys); O columns 64 cq ..
    const int r = lq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(lq * 32) << 16;
    const uint32_t p_full_even[2] = {peer_smem_addr(&bars->p_full[0], 0),
                                     peer_smem_addr(&bars->p_full[1], 0)};
    const uint32_t o_free_even = peer_smem_addr(&bars->o_free, 0);
    uint32_t S = 0;  // steps of the pair's earlier items
    // Every thread runs every item of the pair (even after an abort, when each
    // wait returns at once), so the named barrier of the epilogue is reached
    // the same number of times by all softmax threads of the CTA.
    for (int rr = 0, k = 0; item_of_round(rr) < n_items; ++rr, ++k) {
      const int item = item_of_round(rr);
      int n_tiles, tok, key_last;  // what lives through the loop
      {
        const Item it = item_at(item);
        n_tiles = it.n_tiles;
        tok = it.t0_pair + (int)rank * tile_tok + r / g;
        // last key this row sees: padding rows of a chunk stop at the last
        // valid key, so they never read rows past the valid keys either
        key_last = kChunk ? it.p0 + min(tok, a.T - 1) : tok;
        // the row's 64 gate values (one 128-byte line) into L2 now, so that
        // the epilogue, on the item boundary, finds them there
        if (tok < a.T) {
          const long long gate_row = ((long long)it.b * a.T + tok) * a.Hq + (it.kv * g + (r % g));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(a.qg + gate_row * (2 * D) + D + cq * 64));
        }
      }
      float m = fixed_max ? bound * 1.01f + 0.5f : -INFINITY;
      float l = 0.f;
      bool ok = true;
      for (int j = 0; j < n_tiles; ++j) {
        const uint32_t s = S + (uint32_t)j;
        ok = __all_sync(kFull, mbar_wait_cluster(&bars->s_full[s & 1], (s >> 1) & 1, a.err,
                                                 kDevTimeoutSoftmax, abort));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tmem_s = tmem + (s & 1) * BN + cq * 32 + lane_off;
        uint32_t sr[32];
        tmem_ld32_wait(tmem_s, sr);
        float sv[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) sv[e] = __uint_as_float(sr[e]);
        const int key0 = j * BN + cq * 32;
        if (key0 + 31 > key_last) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (key0 + e > key_last) sv[e] = -INFINITY;
        }
        bool move = false;
        float alpha = 1.0f;
        if (!fixed_max) {
          float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
          for (int e = 4; e < 32; ++e) mx[e & 3] = fmaxf(mx[e & 3], sv[e]);
          float* xm = xchg + (s & 1) * 4 * 128;  // [quarter][128]
          xm[cq * 128 + r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
          mbar_arrive(&bars->xmax_full);
          ok = __all_sync(kFull, mbar_wait(&bars->xmax_full, s & 1, a.err, kDevTimeoutSoftmax,
                                           abort));
          if (!ok) break;
          const float mrow = fmaxf(fmaxf(xm[r], xm[128 + r]), fmaxf(xm[256 + r], xm[384 + r]));
          const float m_tile = mrow * kScaleLog2;
          move = m_tile > m + kRescaleThreshold;
          const float m_new = move ? m_tile : m;
          alpha = move ? ex2(m - m_new) : 1.0f;
          m = m_new;
          l *= alpha;
        }
        // p = 2^(s * scale - m), two at a time on the f32x2 pipes
        const uint64_t scale2 = f2_pack(kScaleLog2, kScaleLog2);
        const uint64_t negm2 = f2_pack(-m, -m);
        uint64_t sum2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint64_t x = f2_fma(f2_pack(sv[2 * e], sv[2 * e + 1]), scale2, negm2);
          float x0, x1;
          f2_unpack(x, x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          sum2[e & 1] = f2_add(sum2[e & 1], f2_pack(p0, p1));
          pw[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16_wait(tmem_s, pw);  // P over the first 16 of this thread's S columns
        if (!fixed_max && j > 0 && __any_sync(kFull, move)) {
          // rescale this thread's O columns once PV_{j-1} has completed,
          // before PV_j adds terms relative to the new max
          ok = __all_sync(kFull, mbar_wait_cluster(&bars->pv_done, (s - 1) & 1, a.err,
                                                   kDevTimeoutSoftmax, abort));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            const uint32_t to = tmem + kTmemO + cq * 64 + cc * 32 + lane_off;
            tmem_ld32_wait(to, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32_wait(to, o);
          }
        }
        float a0, a1, b0, b1;
        f2_unpack(sum2[0], a0, a1);
        f2_unpack(sum2[1], b0, b1);
        l += (a0 + a1) + (b0 + b1);
        // the warp's tcgen05.st has completed (wait::st above, warp-collective):
        // one arrive per warp, on the even CTA's barrier, publishes its 32 rows.
        // P is the signal's only payload, so the arrive releases nothing
        // (relaxed): the odd CTA's warps then pay no cluster-scope fence
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive_relaxed(&bars->p_full[s & 1]);
          else
            mbar_arrive_cluster_relaxed(p_full_even[s & 1]);
        }
      }
      // ---- epilogue: the row's four partial sums, then O / l * sigmoid(gate)
      ok = __all_sync(kFull, ok && !*abort);
      const Item it = item_at(item);
      // rows past the sequence, and the 128 - g * (128 / g) rows after the last
      // whole token when g does not divide 128, are padding
      const bool store = ok && tok < a.T && r < g * tile_tok;
      const long long row = ((long long)it.b * a.T + tok) * a.Hq + (it.kv * g + (r % g));
      // the row's first 32-byte gate piece is requested now, so that its
      // latency runs under the partial-sum barrier and the wait for O (the
      // other three follow inside the epilogue: holding them all across the
      // wait spills at the register cap)
      const bool g_wide =
          ((reinterpret_cast<uintptr_t>(a.out) | reinterpret_cast<uintptr_t>(a.qg)) & 31u) == 0;
      uint32_t g_first[8];
      if (store && g_wide)
        asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=r"(g_first[0]), "=r"(g_first[1]), "=r"(g_first[2]), "=r"(g_first[3]),
              "=r"(g_first[4]), "=r"(g_first[5]), "=r"(g_first[6]), "=r"(g_first[7])
            : "l"(a.qg + row * (2 * D) + D + cq * 64));
      // the partial sums go to a slot double-buffered by item; every thread of
      // the four warpgroups reaches this barrier once per item
      float* lsum = xchg + 2 * 4 * 128 + (k & 1) * 4 * 128;  // [quarter][128]
      lsum[cq * 128 + r] = l;
      named_barrier_sync(1, kSoftmaxWGs * 128);
      if (ok) {
        l = (lsum[r] + lsum[128 + r]) + (lsum[256 + r] + lsum[384 + r]);
        // with the fixed shift only a key far outside the norm bound (a cache
        // breaking its precondition) can overflow the sum: report it
        if (store && fixed_max && !(l <= 3.0e38f)) record_error(a.err, kErrWordBound);
        ok = __all_sync(kFull, mbar_wait_cluster(&bars->o_final, k & 1, a.err,
                                                 kDevTimeoutEpilogue, abort));
      }
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.0f / l;
        uint16_t* orow = a.out + row * D + cq * 64;
        const uint4* grow = reinterpret_cast<const uint4*>(a.qg + row * (2 * D) + D + cq * 64);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t o[32];
          tmem_ld32_wait(tmem + kTmemO + cq * 64 + cc * 32 + lane_off, o);
          if (store) {
            // 32-byte stores fill whole sectors of the row (out is 16-byte
            // aligned by contract; 16-byte stores serve the other case)
            const bool wide = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0;
#pragma unroll
            for (int q8 = 0; q8 < 2; ++q8) {
              uint32_t zw[8];
              // the gate's 16 values of this piece: one 32-byte load when aligned
              uint32_t g8[8];
              if (cc == 0 && q8 == 0 && g_wide) {
#pragma unroll
                for (int e = 0; e < 8; ++e) g8[e] = g_first[e];
              } else if (wide && (reinterpret_cast<uintptr_t>(a.qg) & 31u) == 0) {
                asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                             : "=r"(g8[0]), "=r"(g8[1]), "=r"(g8[2]), "=r"(g8[3]), "=r"(g8[4]),
                               "=r"(g8[5]), "=r"(g8[6]), "=r"(g8[7])
                             : "l"(grow + cc * 4 + 2 * q8));
              } else {
                const uint4 ga = grow[cc * 4 + 2 * q8], gb = grow[cc * 4 + 2 * q8 + 1];
                g8[0] = ga.x; g8[1] = ga.y; g8[2] = ga.z; g8[3] = ga.w;
                g8[4] = gb.x; g8[5] = gb.y; g8[6] = gb.z; g8[7] = gb.w;
              }
#pragma unroll
              for (int h4 = 0; h4 < 2; ++h4) {
                const int q4 = 2 * q8 + h4;
                const uint32_t gw[4] = {g8[h4 * 4], g8[h4 * 4 + 1], g8[h4 * 4 + 2], g8[h4 * 4 + 3]};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  // sigmoid(x) = 1 / (1 + 2^(-x log2 e)), the quotient by the
                  // reciprocal-based fast division (a few fp32 ulps, far
                  // below the bf16 rounding of z; 1 + 2^y past 2^126 gives 0,
                  // the limit): an IEEE division per element cost the
                  // epilogue, which sits on the item boundary, ~3 % of K6
                  const float g0 = bf16_lo(gw[e]), g1 = bf16_hi(gw[e]);
                  const float sg0 = __fdividef(1.0f, 1.0f + ex2(-1.4426950408889634f * g0));
                  const float sg1 = __fdividef(1.0f, 1.0f + ex2(-1.4426950408889634f * g1));
                  zw[h4 * 4 + e] = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2 * e]) * inv_l * sg0,
                                               __uint_as_float(o[q4 * 8 + 2 * e + 1]) * inv_l * sg1);
                }
              }
              uint16_t* dst = orow + cc * 32 + q8 * 16;
              if (wide) {
                asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst),
                             "r"(zw[0]), "r"(zw[1]), "r"(zw[2]), "r"(zw[3]), "r"(zw[4]), "r"(zw[5]),
                             "r"(zw[6]), "r"(zw[7]) : "memory");
              } else {
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(zw[0], zw[1], zw[2], zw[3]);
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(zw[4], zw[5], zw[6], zw[7]);
              }
            }
          }
        }
      }
      // O has been read: the next item's first PV may overwrite it (one
      // arrive per warp of both CTAs, on the even CTA's barrier). Relaxed: the
      // epilogue's output stores need not drain before the signal (with a
      // release the arrive waited for them, on the item boundary)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive_relaxed(&bars->o_free);
        else
          mbar_arrive_cluster_relaxed(o_free_even);
      }
      S += (uint32_t)n_tiles;
    }
  }

  // both CTAs meet here once the pair's MMAs have drained and every TMEM
  // access of either CTA is done; then each frees its tensor memory
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair<kTmemCols>(tmem);
  }
}

template <class Args>
cudaError_t launch(const Args& args_in, cudaStream_t stream) {
  Args args = args_in;
  GatedAttnArgs& a = base_args_mut(args);
  static unsigned long long done_mask = 0;  // per-device dynamic smem opt-in, per instantiation
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(done_mask & (1ull << dev))) {
    e = cudaFuncSetAttribute(gated_attention_pair_kernel<Args>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) done_mask |= 1ull << dev;
  }
  // one persistent pair per two SMs over all items
  const long long items = (long long)a.n_mtiles * a.B * a.Hkv;
  if (items == 0) return cudaSuccess;
  if (items > 0x3fffffffLL) return cudaErrorInvalidConfiguration;
  static int sm_count[64];
  int n_sm = dev < 64 ? sm_count[dev] : 0;
  if (n_sm == 0) {
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) sm_count[dev] = n_sm;
  }
  const long long pairs = items < n_sm / 2 ? items : (long long)(n_sm / 2);
  const long long grid = 2 * pairs;
  // a plain prefill keeps one set (its items of one group run from 1 to n
  // KV tiles; longest first over all groups balances them best)
  if constexpr (std::is_same<Args, GatedAttnChunkArgs>::value)
    a.group_sets = choose_group_sets(a.n_mtiles, a.B, a.Hkv, 2 * (BM / a.g), a.T, args.pos_b, BN,
                                     (int)pairs);
  else
    a.group_sets = 1;
  gated_attention_pair_kernel<Args><<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace

int gated_tokens_per_cta(int g) { return 2 * (BM / g); }  // per pair of CTAs

cudaError_t launch_gated_attention(const GatedAttnArgs& a, cudaStream_t stream) {
  return launch(a, stream);
}

cudaError_t launch_gated_attention(const GatedAttnChunkArgs& a, cudaStream_t stream) {
  if (a.base.B > kMaxBatch || !a.base.v_head_major) return cudaErrorInvalidValue;
  return launch(a, stream);
}

}  // namespace q3a
