// prefill_attention.cu — K2, causal grouped-query attention on tcgen05.
//
// Computes, for every query row (b, i, h) with normalised+rotated qhat and the
// normalised+rotated keys khat_j of group h / g:
//   out = sum_{j <= i} softmax_j(qhat . khat_j / sqrt(128)) v_j
// ("7.2 Qwen3 full-scale implementation", §7.2.1 GroupedQueryAttention.forward:
// repeat_interleave of the KV heads, triu causal mask, softmax of the scores
// over head_dim ** 0.5, product with the values).
//
// Tiling. A CTA owns two M tiles of 128 query rows each. A tile holds the g
// query heads of one KV group for 128/g consecutive tokens, packed row
// r = (token, head kv*g + r%g); the two tiles are consecutive token ranges.
// Every 128-key K/V tile the CTA loads is used by all g heads of both tiles,
// so each K/V byte is read once per 256/g tokens. KV tiles above the causal
// diagonal are never loaded; diagonal tiles are masked per element.
//
// Query tiles. A chunk's Q tiles arrive normalised and rotated (Qhat from the
// prologue); the plain prefill loads the raw q rows and the tile's two softmax
// warpgroups apply Q-Norm + RoPE to them in shared memory at the start of each
// item (qnorm_rope_half_row), releasing the tile to the MMA thread on its
// "Q ready" barrier, so Qhat never makes a round trip through HBM.
//
// Work items and persistence. An item is one pair of Q tiles of one KV group
// (longest items first; a chunk's longest first within sets of KV groups, as
// item_index orders them). The plain prefill runs one CTA per SM, each walking
// its items in rounds of gridDim.x in snake order (forward in even rounds,
// backward in odd ones, so long and short items pair up across CTAs); the
// tensor pipe does not drain between items: the next item's Q pair is loaded
// as soon as the current item's last QK^T has completed ("Q free"), the K/V
// ring and every barrier phase run on across items, and the next item's
// first PV of a tile waits only for that tile's epilogue to have read O
// ("O free"). The chunk against the caches runs the same way.
//
// Roles (576 threads):
//   WG 0..3   softmax + epilogue. WG w serves Q tile t = w/2 and the column
//             half c = w%2 of its rows: thread r of the warpgroup owns TMEM
//             lane r (row r) and columns 64c..64c+63 of S_t and O_t;
//   warp 16   TMA producer (per item: Q0, Q1, then K_j, V_j through a ring
//             of four 32 KB slots); warp 17: MMA issuer (one thread).
// TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each. A softmax
// thread writes its 64 probabilities as bf16 pairs (32 columns) over the first
// half of its own S columns, and O_t += P_t V_j reads them from there
// (tcgen05.mma with A in tensor memory), so P never touches shared memory.
// MMA stream: S0_0, S1_0, then per KV tile j: PV0_j, S0_{j+1}, PV1_j,
// S1_{j+1}. tcgen05.mma ops of one thread execute in issue order, so S_t,j+1
// overwrites S_t/P_t only after PV_t,j has read P_t. While the tensor core
// runs one tile's PV and next QK^T, the other tile's softmax computes.
// The commit that signals "S_t,j ready" also covers every earlier MMA of the
// thread, so when a softmax warpgroup sees S_t,j, O_t already holds every
// PV up to j-1 and can be rescaled in place, and K_j and V_{j-1} are no longer
// read by tile t: the softmax warpgroups, not the MMA thread, hand the ring
// slots back to the producer, which keeps commits off the MMA issue path.
//
// Softmax in the exp2 domain. QK-Norm bounds every logit: |qhat| <=
// sqrt(128) max|gamma_q| and |khat| <= sqrt(128) max|gamma_k|, so
// |qhat . khat| / sqrt(128) <= sqrt(128) max|gamma_q| max|gamma_k| (the
// prologue writes this bound to the workspace). While the bound is moderate,
// p = 2^(s - bound) never underflows for the terms that matter, and the
// softmax needs neither a row max nor any rescaling of O: it is then a pure
// elementwise map plus a running sum, and the two threads of a row never talk
// until the epilogue adds their partial sums. For large gammas the kernel
// falls back to an online max with a lazy rescale (the two halves of a row
// exchange their tile maxima through shared memory and an mbarrier; the max only moves, and
// O_t, l are rescaled by 2^(m_old - m_new), when a tile's max exceeds it by
// more than 8).
//
// Chunk against a KV cache ("Chapter 20, Qwen3 and Qwen3.5", §20.3: a
// position counter, new keys rotated at their positions and appended to the
// cached ones, a causal mask that starts at the chunk's first position). The
// second instantiation reads K and V from the head-major caches, into which
// the prologue has already written the chunk's rows; token t of sequence b
// sits at position pos_b[b] + t and sees keys 0..pos_b[b] + t. Rows of the
// last V tile past the valid keys hold whatever the cache holds there (a
// probability of 0 times a NaN is NaN), so the producer warp clears them in
// shared memory before the MMA issuer is allowed to read that tile. Cached
// keys were normalised by earlier calls with the same gamma (the cache's
// precondition), so the fixed shift holds for them too; the shift cancels in
// the normalisation, and only a cache breaking the bound so far that a row
// sum overflows changes the result, which the epilogue reports.
//
// Every mbarrier wait is bounded (q3a_device.cuh); a timeout sets the error
// word, all roles unwind, in-flight copies and MMAs are drained and TMEM is
// freed before the CTA exits.
#include <type_traits>

#include "q3a_device.cuh"
#include "q3a_internal.h"

namespace q3a {

namespace {

constexpr int BM = 128;  // query rows per Q tile
constexpr int BN = 128;  // keys per KV tile
constexpr int kQTiles = 2;
constexpr int kSoftmaxWGs = 4;  // two column halves per Q tile
constexpr int kSlots = 4;       // K/V ring slots
// four softmax warpgroups, then the producer warp and the MMA warp (576
// threads, 18 warps: a scheduler holding five of them caps a thread at 96
// registers)
constexpr int kThreads = kSoftmaxWGs * 128 + 64;
constexpr uint32_t kHalf = 16384;      // 128 rows x 128 bytes
constexpr uint32_t kTile = 2 * kHalf;  // 128 rows x 128 bf16
constexpr uint32_t OFF_Q = 0;          // two Q tiles
constexpr uint32_t OFF_RING = OFF_Q + kQTiles * kTile;
constexpr uint32_t OFF_BAR = OFF_RING + kSlots * kTile;
// row-half exchange: tile maxima [2 tiles][2 halves][2 parities][128] fp32,
// then partial sums [2 item parities][2 tiles][2 halves][128] fp32
constexpr uint32_t OFF_XCHG = OFF_BAR + 256;
// plain prefill's query norm: gamma_q as fp32 [128], then the row sums of
// squares [2 tiles][2 halves][128]
constexpr uint32_t OFF_QNORM = OFF_XCHG + (kQTiles * 2 * 2 * 128 + 2 * kQTiles * 2 * 128) * 4;
constexpr uint32_t kSmemBytes = OFF_QNORM + 128 * 4 + kQTiles * 2 * 128 * 4 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr float kScaleLog2 = 0.12751743074380046f;  // log2(e) / sqrt(128)
constexpr float kRescaleThreshold = 8.0f;
// largest logit bound (log2 units) for which 2^(-2 bound), the smallest
// possible term after the fixed shift, is still a normal float
constexpr float kFixedMaxLimit = 60.0f;
constexpr unsigned kFull = 0xffffffffu;

struct Bars {
  uint64_t q_full, q_empty;  // Q pair landed / free again (the item's last QK^T completed)
  uint64_t q_ready[kQTiles];  // plain prefill: tile t normalised and rotated in place
  uint64_t slot_full[kSlots], slot_empty[kSlots];
  uint64_t s_full[kQTiles], p_full[kQTiles], o_final[kQTiles];
  uint64_t o_free[kQTiles];  // the item's epilogue has read O_t
  uint64_t xmax_full[kQTiles];  // fallback path: both row halves posted their tile max
  uint64_t vtail;               // cache V: rows past the valid keys cleared in the last tile
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// Descriptors of 128-byte-swizzled tiles whose bases are 1024-byte aligned:
// moving the start address by `off` bytes adds off >> 4 to the low field, so
// each MMA step costs one 64-bit add.
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
  mma_ss<0>(tmem_s, q_desc, k_desc, idesc);
#pragma unroll
  for (int kk = 1; kk < 8; ++kk) {
    const uint64_t off = (uint64_t)(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4);
    mma_ss<1>(tmem_s, q_desc + off, k_desc + off, idesc);
  }
}

__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_s, uint64_t v_desc,
                                         uint32_t accumulate) {
  // A = P in TMEM: keys 0..63 as bf16 pairs in S columns 0..31, keys 64..127
  // in S columns 64..95 (16 keys = 8 columns per step). B = V, MN-major: 64-wide
  // d blocks 16 KB apart, 8-key groups 1 KB apart; 16 keys = 2 KB per step.
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
  mma_bf16_ts(tmem_o, tmem_s, v_desc, idesc, accumulate);
#pragma unroll
  for (int kk = 1; kk < 8; ++kk)
    mma_bf16_ts(tmem_o, tmem_s + (kk >> 2) * 64 + (kk & 3) * 8, v_desc + (uint64_t)(kk * 2048 >> 4),
                idesc, 1u);
}

// Q-Norm + RoPE of the query tiles of the plain prefill, in shared memory.
// Thread (r, hc) of a tile's two softmax warpgroups owns row r and the rotate-
// half pairs i = 32hc .. 32hc+31: elements i (chunks 4hc.. of the first 64-
// column half, 128-byte swizzle: chunk c of row r sits at c ^ (r & 7)) and
// i + 64 (the same chunks of the second half). The row's sum of squares meets
// its partner's through `xss` and the tile's named barrier; then
//   y = x / sqrt(mean(x^2) + eps) * gamma,  y'_i = y_i c - y_{i+64} s,
//   y'_{i+64} = y_{i+64} c + y_i s,  a_i = pos * theta^(-2i/128),
// one bf16 rounding, written back in place ("7.2 Qwen3 full-scale
// implementation", §7.2.1 RMSNorm then apply_rope; norm before RoPE). cs points
// at (cos a_i, sin a_i, cos a_{i+1}, sin a_{i+1}) for i = 32hc + 2m, m = 0..15,
// in the prologue's table row of the row's position.
__device__ __forceinline__ void qnorm_rope_half_row(uint8_t* tile, int r, int hc,
                                                    const float4* cs, const float* gam,
                                                    float eps, float* xss, uint32_t bar_id) {
  const uint32_t sw = (uint32_t)(r & 7);
  uint64_t ss2 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t off = (uint32_t)r * 128u + ((((uint32_t)(4 * hc + (j & 3))) ^ sw) << 4);
    const uint4 w = *reinterpret_cast<const uint4*>(tile + (j >> 2) * kHalf + off);
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint64_t x2 = f2_pack(bf16_lo(v[m]), bf16_hi(v[m]));
      ss2 = f2_fma(x2, x2, ss2);
    }
  }
  float s_lo, s_hi;
  f2_unpack(ss2, s_lo, s_hi);
  float ss = s_lo + s_hi;
  xss[hc * 128 + r] = ss;
  named_barrier_sync(bar_id, 256);
  ss += xss[(hc ^ 1) * 128 + r];
  const float inv_rms = rsqrtf(ss * (1.0f / 128.0f) + eps);
  const uint64_t inv2 = f2_pack(inv_rms, inv_rms);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // the chunk is read again after the barrier rather than kept in registers
    const uint32_t off = (uint32_t)r * 128u + ((((uint32_t)(4 * hc + j)) ^ sw) << 4);
    const uint4 wl = *reinterpret_cast<const uint4*>(tile + off);
    const uint4 wh = *reinterpret_cast<const uint4*>(tile + kHalf + off);
    const uint32_t lo[4] = {wl.x, wl.y, wl.z, wl.w};
    const uint32_t hi[4] = {wh.x, wh.y, wh.z, wh.w};
    uint32_t ol[4], oh[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int i0 = 8 * (4 * hc + j) + 2 * m;  // pairs i0, i0 + 1
      const float2 gl = *reinterpret_cast<const float2*>(gam + i0);
      const float2 gh = *reinterpret_cast<const float2*>(gam + 64 + i0);
      const float4 t4 = __ldg(cs + 4 * j + m);
      const uint64_t C2 = f2_pack(t4.x, t4.z), S2 = f2_pack(t4.y, t4.w);
      const uint64_t A = f2_mul(f2_mul(f2_pack(bf16_lo(lo[m]), bf16_hi(lo[m])), f2_pack(gl.x, gl.y)),
                                inv2);  // y_i
      const uint64_t Bv = f2_mul(
          f2_mul(f2_pack(bf16_lo(hi[m]), bf16_hi(hi[m])), f2_pack(gh.x, gh.y)), inv2);  // y_{i+64}
      const uint64_t OL = f2_sub(f2_mul(A, C2), f2_mul(Bv, S2));
      const uint64_t OH = f2_fma(A, S2, f2_mul(Bv, C2));
      float o0, o1;
      f2_unpack(OL, o0, o1);
      ol[m] = pack_bf16x2(o0, o1);
      f2_unpack(OH, o0, o1);
      oh[m] = pack_bf16x2(o0, o1);
    }
    *reinterpret_cast<uint4*>(tile + off) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
    *reinterpret_cast<uint4*>(tile + kHalf + off) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
  }
}

// The plain prefill and the chunk against the caches are two instantiations,
// so the plain one carries none of the chunk's bookkeeping.
__device__ __forceinline__ const PrefillArgs& base_args(const PrefillArgs& a) { return a; }
__device__ __forceinline__ const PrefillArgs& base_args(const PrefillChunkArgs& a) {
  return a.base;
}
__device__ __forceinline__ int chunk_start(const PrefillArgs&, int) { return 0; }
__device__ __forceinline__ int chunk_start(const PrefillChunkArgs& a, int b) { return a.pos_b[b]; }
__device__ __forceinline__ bool fixed_shift_allowed(const PrefillArgs&) { return true; }
__device__ __forceinline__ bool fixed_shift_allowed(const PrefillChunkArgs& a) {
  return a.fixed_shift_ok != 0;
}

template <class Args>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_attention_kernel(const __grid_constant__ Args args) {
  constexpr bool kChunk = sizeof(Args) != sizeof(PrefillArgs);
  const PrefillArgs& a = base_args(args);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  float* xchg = reinterpret_cast<float*>(smem + OFF_XCHG);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work items ------------------------------------------------------------
  // Item i as item_index orders them (longest first within each set of
  // groups). A CTA takes items in rounds of gridDim.x, in snake order (forward
  // in even rounds, backward in odd ones), so the long and short items of
  // consecutive rounds pair up across CTAs.
  const int bk_count = a.B * a.Hkv;
  const int n_items = a.n_mtiles * bk_count;
  const int g = a.g;
  const int tile_tok = BM / g;  // tokens per Q tile
  const int G = (int)gridDim.x, c = (int)blockIdx.x;
  auto item_of_round = [&](int r) { return r * G + ((r & 1) ? G - 1 - c : c); };
  struct Item {
    int b, kv, t0, p0, n_tiles, n_keys;
  };
  auto item_at = [&](int i) {
    Item it;
    ItemIndex ix;
    if (kChunk) {
      // group_sets: a power of two dividing the group count
      ix = item_index(i, a.n_mtiles, bk_count >> (31 - __clz(a.group_sets)));
    } else {
      ix = ItemIndex{i % bk_count, a.n_mtiles - 1 - i / bk_count};  // one set
    }
    it.b = ix.bk / a.Hkv;
    it.kv = ix.bk % a.Hkv;
    it.t0 = ix.mt * kQTiles * tile_tok;
    // token t of the sequence sits at position p0 + t (p0 = 0 for a plain
    // prefill) and sees keys 0..p0+t; keys p0+T.. are not valid
    it.p0 = chunk_start(args, it.b);
    it.n_tiles = item_kv_tiles(it.t0, kQTiles * tile_tok, a.T, it.p0, BN);
    it.n_keys = it.p0 + a.T;
    return it;
  };

  constexpr bool kFuseQ = !kChunk;  // the plain prefill normalises its query tiles itself
  float* qn_gamma = reinterpret_cast<float*>(smem + OFF_QNORM);
  float* qn_ss = reinterpret_cast<float*>(smem + OFF_QNORM + 512);
  if (kFuseQ && threadIdx.x < 128)
    qn_gamma[threadIdx.x] = __uint_as_float((uint32_t)a.q_gamma[threadIdx.x] << 16);
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int t = 0; t < kQTiles; ++t) mbar_init(&bars->q_ready[t], 256);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars->slot_full[s], 1);
      mbar_init(&bars->slot_empty[s], kQTiles);  // one arrive per Q tile's softmax
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 256);
      mbar_init(&bars->o_final[t], 1);
      mbar_init(&bars->o_free[t], 256);
      mbar_init(&bars->xmax_full[t], 256);
    }
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->vtail, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc<kTmemCols>(&bars->tmem_base);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort_flag;

  if (warp >= kSoftmaxWGs * 4) {
    if (warp == kSoftmaxWGs * 4) {
      // ---------------------------------------------------------- producer
      // Lane 0 issues the loads. Cache V (chunked prefill): an item's last V
      // tile may hold rows past the valid keys (whatever the cache holds
      // there). Their weights are 0, but 0 x NaN is NaN in the PV product, so
      // the whole warp clears them once that tile has landed and publishes it
      // on "V tail" (one phase per item that has such a tail).
      if (lane == 0) {
        tma_prefetch_desc(&a.tm_q);
        tma_prefetch_desc(&a.tm_k);
        tma_prefetch_desc(&a.tm_v);
      }
      // K/V tiles are read again by the group's other items (kept in L2
      // ahead of the query tiles, which are read once)
      const uint64_t pol_last = l2_evict_last_policy(), pol_first = l2_evict_first_policy();
      uint32_t L = 0;       // first load index of the current item
      uint32_t issued = 0;  // loads issued (lane 0)
      uint32_t n_q = 0;     // Q pairs issued (lane 0)
      bool ok = kChunk || lane == 0;  // the plain prefill's loop runs on lane 0 only
      for (int r = 0; ok && item_of_round(r) < n_items; ++r) {
        const Item it = item_at(item_of_round(r));
        if (lane == 0) {
          // the Q tiles are free once the previous item's last QK^T completed
          ok = n_q == 0 || mbar_wait(&bars->q_empty, (n_q - 1) & 1, a.err, kDevTimeoutTma, abort);
          if (ok) {
            mbar_arrive_expect_tx(&bars->q_full, kQTiles * kTile);
            for (int t = 0; t < kQTiles; ++t) {
              uint8_t* qd = smem + OFF_Q + t * kTile;
              const int tq = it.t0 + t * tile_tok;
              tma_load_4d_hint(qd, &a.tm_q, &bars->q_full, 0, it.kv * g, tq, it.b, pol_first);
              tma_load_4d_hint(qd + kHalf, &a.tm_q, &bars->q_full, 64, it.kv * g, tq, it.b,
                               pol_first);
            }
            ++n_q;
          }
          const int row3 = it.b * a.Hkv + it.kv;
          for (int i = 0; ok && i < 2 * it.n_tiles; ++i) {  // K_0, V_0, K_1, V_1, ...
            const uint32_t li = L + (uint32_t)i;
            const int s = (int)(li % kSlots);
            if (!mbar_wait(&bars->slot_empty[s], ((li / kSlots) & 1) ^ 1, a.err, kDevTimeoutTma,
                           abort)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->slot_full[s], kTile);
            uint8_t* dst = smem + OFF_RING + s * kTile;
            const int j = i >> 1;
            if ((i & 1) == 0) {
              tma_load_3d_hint(dst, &a.tm_k, &bars->slot_full[s], 0, j * BN, row3, pol_last);
              tma_load_3d_hint(dst + kHalf, &a.tm_k, &bars->slot_full[s], 64, j * BN, row3,
                               pol_last);
            } else if (kChunk) {
              tma_load_3d_hint(dst, &a.tm_v, &bars->slot_full[s], 0, j * BN, row3, pol_last);
              tma_load_3d_hint(dst + kHalf, &a.tm_v, &bars->slot_full[s], 64, j * BN, row3,
                               pol_last);
            } else {
              tma_load_4d_hint(dst, &a.tm_v, &bars->slot_full[s], 0, it.kv, j * BN, it.b,
                               pol_last);
              tma_load_4d_hint(dst + kHalf, &a.tm_v, &bars->slot_full[s], 64, it.kv, j * BN, it.b,
                               pol_last);
            }
            issued = li + 1;
          }
        }
        if (kChunk) ok = __shfl_sync(kFull, ok, 0);  // the whole warp runs the loop
        if (!ok) break;
        if (kChunk && it.n_tiles * BN > it.n_keys) {
          // every load of the item has been issued and none after it, so the
          // slot's barrier is in the phase of the item's last load
          const uint32_t tail_load = L + 2u * (uint32_t)it.n_tiles - 1u;
          const int tail_first = it.n_keys - (it.n_tiles - 1) * BN;  // first row to clear
          ok = __all_sync(kFull, mbar_wait(&bars->slot_full[tail_load % kSlots],
                                           (tail_load / kSlots) & 1, a.err, kDevTimeoutTma,
                                           abort));
          if (!ok) break;
          uint8_t* vt = smem + OFF_RING + (tail_load % kSlots) * kTile;
          const int chunks = (BN - tail_first) * 16;  // 16-byte chunks, both halves
          for (int ch = lane; ch < chunks; ch += 32) {
            const int row = tail_first + (ch >> 4), half = (ch >> 3) & 1, q16 = ch & 7;
            *reinterpret_cast<uint4*>(vt + half * kHalf + row * 128 + q16 * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->vtail);
        }
        L += 2u * (uint32_t)it.n_tiles;
      }
      if (lane == 0 && *abort) {
        // let every copy that was issued land before the CTA goes away
        if (n_q > 0) mbar_wait(&bars->q_full, (n_q - 1) & 1, nullptr, 0, nullptr);
        for (uint32_t i = issued > (uint32_t)kSlots ? issued - kSlots : 0u; i < issued; ++i)
          mbar_wait(&bars->slot_full[i % kSlots], (i / kSlots) & 1, nullptr, 0, nullptr);
      }
    } else if (warp == kSoftmaxWGs * 4 + 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t q_addr = smem_u32(smem + OFF_Q);
      const uint32_t ring = smem_u32(smem + OFF_RING);
      // base descriptors, built once: Q tiles (K-major), ring slots as K
      // (K-major) and as V (MN-major)
      const uint64_t q_desc0 = smem_desc_sw128(q_addr, 16, 1024);
      const uint64_t q_desc1 = smem_desc_sw128(q_addr + kTile, 16, 1024);
      const uint64_t slot_k0 = smem_desc_sw128(ring, 16, 1024);
      const uint64_t slot_v0 = smem_desc_sw128(ring, kHalf, 1024);
      constexpr uint64_t kSlotStep = kTile >> 4;  // descriptor units per slot
      uint32_t L = 0;       // loads consumed before the current item
      uint32_t S = 0;       // S steps (per Q tile) before the current item
      uint32_t n_tail = 0;  // earlier items whose last V tile had a cleared tail
      int k = 0;            // items done
      bool ok = true;
      for (int r = 0; ok && item_of_round(r) < n_items; ++r, ++k) {
        const Item it = item_at(item_of_round(r));
        const int n_tiles = it.n_tiles;
        const bool v_tail = kChunk && n_tiles * BN > it.n_keys;
        // An mbarrier wait issued by this thread after a tcgen05.commit stalls
        // until that commit resolves, i.e. until every earlier MMA has
        // finished. So each commit below is followed by a full MMA group
        // before the next wait, by which time it has resolved: the waits for
        // a group's inputs are placed before the commit of the previous group.
        auto wait_inputs = [&](int j) {  // V_j, K_{j+1} (or the cleared V tail) and P0_j
          const uint32_t iv = L + 2u * j + 1u, ik = L + 2u * j + 2u;
          const bool last = j + 1 == n_tiles;
          uint64_t* second = last ? (v_tail ? &bars->vtail : &bars->slot_full[iv % kSlots])
                                  : &bars->slot_full[ik % kSlots];
          const uint32_t second_par = last ? (v_tail ? n_tail & 1 : (iv / kSlots) & 1)
                                           : (ik / kSlots) & 1;
          return mbar_wait3(&bars->slot_full[iv % kSlots], (iv / kSlots) & 1, second, second_par,
                            &bars->p_full[0], (S + j) & 1, a.err, kDevTimeoutMma, abort);
        };
        // the Q pair has landed (chunk: Qhat) or each tile has been normalised
        // and rotated in place by its softmax warpgroups (plain prefill);
        // polled, as the tensor pipe is idle until this wait returns
        ok = mbar_poll(kFuseQ ? &bars->q_ready[0] : &bars->q_full, k & 1, a.err, kDevTimeoutMma,
                       abort) &&
             mbar_poll(&bars->slot_full[L % kSlots], (L / kSlots) & 1, a.err, kDevTimeoutMma,
                       abort);
        if (!ok) break;
        const uint64_t k_desc0 = slot_k0 + (uint64_t)(L % kSlots) * kSlotStep;
        tc_fence_after();
        issue_qk(tmem, q_desc0, k_desc0);
        mma_commit(&bars->s_full[0]);
        if (kFuseQ) {
          // tile 1's warpgroups finish their previous epilogue later than
          // tile 0's: this wait is longer than the commit above takes to resolve
          ok = mbar_poll(&bars->q_ready[1], k & 1, a.err, kDevTimeoutMma, abort);
          if (!ok) break;
          tc_fence_after();
        }
        issue_qk(tmem + 128, q_desc1, k_desc0);
        // PV0_0 overwrites O0: the previous item's tile-0 epilogue must have
        // read it
        ok = wait_inputs(0) &&
             (k == 0 || mbar_poll(&bars->o_free[0], (k - 1) & 1, a.err, kDevTimeoutMma, abort));
        mma_commit(&bars->s_full[1]);
        if (n_tiles == 1) mma_commit(&bars->q_empty);  // the item's last QK^T is issued
        for (int j = 0; ok && j < n_tiles; ++j) {
          const uint32_t iv = L + 2u * j + 1u, ik = L + 2u * j + 2u;  // V_j and K_{j+1}
          const bool more = j + 1 < n_tiles;
          const uint64_t v_desc = slot_v0 + (uint64_t)(iv % kSlots) * kSlotStep;
          const uint64_t k_desc = slot_k0 + (uint64_t)(ik % kSlots) * kSlotStep;
          // tile 0: PV0_j, S0_{j+1} (inputs waited for above)
          tc_fence_after();
          issue_pv(tmem + 256, tmem, v_desc, j > 0 ? 1u : 0u);
          if (more) issue_qk(tmem, q_desc0, k_desc);
          ok = mbar_poll(&bars->p_full[1], (S + j) & 1, a.err, kDevTimeoutMma, abort) &&
               (j > 0 || k == 0 ||
                mbar_poll(&bars->o_free[1], (k - 1) & 1, a.err, kDevTimeoutMma, abort));
          mma_commit(more ? &bars->s_full[0] : &bars->o_final[0]);
          if (!ok) break;
          // tile 1: PV1_j, S1_{j+1}
          tc_fence_after();
          issue_pv(tmem + 256 + 128, tmem + 128, v_desc, j > 0 ? 1u : 0u);
          if (more) {
            issue_qk(tmem + 128, q_desc1, k_desc);
            ok = wait_inputs(j + 1);
            mma_commit(&bars->s_full[1]);
            if (j + 2 == n_tiles) mma_commit(&bars->q_empty);  // the item's last QK^T
          } else {
            mma_commit(&bars->o_final[1]);
          }
        }
        L += 2u * (uint32_t)n_tiles;
        S += (uint32_t)n_tiles;
        if (v_tail) ++n_tail;
      }
      // drain: every MMA issued above has completed once this phase completes
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, nullptr, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int wg = warp >> 2;
    const int t = wg >> 1;              // Q tile
    const int hc = wg & 1;              // column half: keys / O columns 64hc..64hc+63
    const int r = threadIdx.x & 127;    // row of S_t / O_t, TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tmem_s = tmem + t * 128 + hc * 64 + lane_off;
    const uint32_t tmem_o = tmem + 256 + t * 128 + hc * 64 + lane_off;
    const uint32_t bar_id = 1 + t;      // named barrier of the two halves of tile t (epilogue)
    float* xmax = xchg + (t * 2) * 2 * 128;  // [half][parity][128]
    const float bound = *a.logit_bound;
    const bool fixed_max = fixed_shift_allowed(args) && bound >= 0.f && bound <= kFixedMaxLimit;
    uint32_t L = 0;  // loads of the CTA's earlier items
    uint32_t S = 0;  // S steps of the CTA's earlier items
    // Every thread runs every item of the CTA (even after an abort, when each
    // wait returns at once), so the named barrier of the epilogue is reached
    // the same number of times by both halves of a tile.
    for (int rr = 0, k = 0; item_of_round(rr) < n_items; ++rr, ++k) {
      const int item = item_of_round(rr);
      int n_tiles, tok_pos;  // only these live through the loop
      {
        const Item it = item_at(item);
        n_tiles = it.n_tiles;
        // position of this row's token; padding rows of a chunk (tokens past
        // its end) stop at the last valid key, so they never read cache rows
        // past the valid keys
        const int tok = it.t0 + t * tile_tok + r / g;
        tok_pos = it.p0 + (kChunk ? min(tok, a.T - 1) : tok);
      }
      bool ok = true;
      if (kFuseQ) {
        // Q-Norm + RoPE of this tile's rows once the raw Q pair has landed.
        // The row's cos/sin come from the prologue's table (L2), loaded before
        // the wait. After an abort every wait returns at once and only the
        // named barrier inside is kept, so both halves meet it once per item.
        const float4* trow =
            reinterpret_cast<const float4*>(a.rope_table + (size_t)min(tok_pos, a.T - 1) * 128) +
            16 * hc;
        // the row's 256 table bytes (two cache lines) into L1 while Q lands
        asm volatile("prefetch.global.L1 [%0];" ::"l"(trow));
        asm volatile("prefetch.global.L1 [%0];" ::"l"(trow + 8));
        ok = __all_sync(kFull, mbar_wait(&bars->q_full, k & 1, a.err, kDevTimeoutSoftmax, abort));
        if (ok) {
          qnorm_rope_half_row(smem + OFF_Q + t * kTile, r, hc, trow, qn_gamma, a.eps,
                              qn_ss + t * 256, bar_id);
          fence_proxy_async_smem();  // the tensor core reads the rows next
        } else {
          named_barrier_sync(bar_id, 256);
        }
        mbar_arrive(&bars->q_ready[t]);
      }
      float m = fixed_max ? bound * 1.01f + 0.5f : -INFINITY;
      float l = 0.f;
      for (int j = 0; ok && j < n_tiles; ++j) {
        const uint32_t step = S + (uint32_t)j;
        ok = __all_sync(kFull,
                        mbar_wait(&bars->s_full[t], step & 1, a.err, kDevTimeoutSoftmax, abort));
        if (!ok) break;
        // S_t,j is complete, and so is every earlier MMA of the issuing
        // thread: K_j is no longer read by tile t, nor the V before it (read
        // by the previous PV_t, possibly of the previous item)
        if (hc == 0 && r == 0) {
          const uint32_t lk = L + 2u * (uint32_t)j;
          mbar_arrive(&bars->slot_empty[lk % kSlots]);
          if (lk > 0) mbar_arrive(&bars->slot_empty[(lk - 1) % kSlots]);
        }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64_wait(tmem_s, sr);

        float s[64];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int e = 0; e < 32; ++e) s[cc * 32 + e] = __uint_as_float(sr[cc * 32 + e]);
        const int key0 = j * BN + hc * 64;
        if (key0 + 63 > tok_pos) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (key0 + e > tok_pos) s[e] = -INFINITY;
        }
        bool move = false;
        float alpha = 1.0f;
        if (!fixed_max) {
          float mx[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = s[e];
#pragma unroll
          for (int e = 8; e < 64; ++e) mx[e & 7] = fmaxf(mx[e & 7], s[e]);
#pragma unroll
          for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
            for (int e = 0; e < w; ++e) mx[e] = fmaxf(mx[e], mx[e + w]);
          // the other half of the row: exchange tile maxima (two parity slots)
          xmax[(hc * 2 + (step & 1)) * 128 + r] = mx[0];
          mbar_arrive(&bars->xmax_full[t]);
          ok = __all_sync(kFull, mbar_wait(&bars->xmax_full[t], step & 1, a.err,
                                           kDevTimeoutSoftmax, abort));
          if (!ok) break;
          const float mrow = fmaxf(mx[0], xmax[((hc ^ 1) * 2 + (step & 1)) * 128 + r]);
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
        uint32_t pw[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const uint64_t x = f2_fma(f2_pack(s[2 * e], s[2 * e + 1]), scale2, negm2);
          float x0, x1;
          f2_unpack(x, x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          sum2[e & 1] = f2_add(sum2[e & 1], f2_pack(p0, p1));
          pw[e] = pack_bf16x2(p0, p1);
        }
        tmem_st32_wait(tmem_s, pw);  // P over the first 32 of this thread's S columns
        // O_t holds every PV of this item up to j-1 here (the S_t,j commit
        // covers them); rescale this thread's O columns before PV_t,j adds
        // terms relative to the new max
        if (!fixed_max && j > 0 && __any_sync(kFull, move)) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            tmem_ld32_wait(tmem_o + cc * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32_wait(tmem_o + cc * 32, o);
          }
        }
        float a0, a1, b0, b1;
        f2_unpack(sum2[0], a0, a1);
        f2_unpack(sum2[1], b0, b1);
        l += (a0 + a1) + (b0 + b1);
        tc_fence_before();
        mbar_arrive(&bars->p_full[t]);
      }
      // ---- epilogue: the row's two partial sums, then O / l -> bf16 -> out
      ok = __all_sync(kFull, ok && !*abort);
      // the partial sums go to a slot the loop never uses, double-buffered by
      // item; every thread of both halves reaches this barrier once per item
      float* lsum = xchg + kQTiles * 2 * 2 * 128 + ((k & 1) * kQTiles + t) * 2 * 128;
      lsum[hc * 128 + r] = l;
      named_barrier_sync(bar_id, 256);
      if (ok) {
        l += lsum[(hc ^ 1) * 128 + r];
        ok = __all_sync(kFull, mbar_wait(&bars->o_final[t], k & 1, a.err, kDevTimeoutEpilogue,
                                         abort));
      }
      if (ok) {
        tc_fence_after();
        const Item it = item_at(item);
        const int tok = it.t0 + t * tile_tok + r / g;
        const float inv_l = 1.0f / l;
        const bool store = tok < a.T;  // rows of tokens past the chunk are padding
        // with the fixed shift only a key far outside the norm bound (a cache
        // breaking its precondition) can overflow the sum: report it
        if (fixed_max && store && !(l <= 3.0e38f)) record_error(a.err, kErrWordBound);
        uint16_t* orow = a.out +
                         (((long long)it.b * a.T + tok) * a.Hq + (long long)it.kv * g + (r % g)) *
                             128 +
                         hc * 64;
        uint32_t o[64];
        tmem_ld64_wait(tmem_o, o);  // all 64 columns, one wait
        const uint64_t opol = l2_evict_first_policy();  // outputs are not read again here
        if (store && (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0) {
          // a thread owns 64 columns (128 bytes) of its row: 32-byte stores
          // fill whole sectors, which the memory system takes far faster
          // than 16-byte halves of them (out is 16-byte aligned by contract;
          // the 16-byte path below serves the other case)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t wv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              wv[e] = pack_bf16x2(__uint_as_float(o[q4 * 16 + 2 * e]) * inv_l,
                                  __uint_as_float(o[q4 * 16 + 2 * e + 1]) * inv_l);
            asm volatile(
                "st.global.L2::cache_hint.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;" ::"l"(
                    orow + q4 * 16),
                "r"(wv[0]), "r"(wv[1]), "r"(wv[2]), "r"(wv[3]), "r"(wv[4]), "r"(wv[5]), "r"(wv[6]),
                "r"(wv[7]), "l"(opol)
                : "memory");
          }
        } else if (store) {
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[q8 * 8 + 0]) * inv_l,
                              __uint_as_float(o[q8 * 8 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[q8 * 8 + 2]) * inv_l,
                              __uint_as_float(o[q8 * 8 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[q8 * 8 + 4]) * inv_l,
                              __uint_as_float(o[q8 * 8 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[q8 * 8 + 6]) * inv_l,
                              __uint_as_float(o[q8 * 8 + 7]) * inv_l);
            reinterpret_cast<uint4*>(orow)[q8] = w;
          }
        }
      }
      // O_t has been read: the next item's first PV of this tile may
      // overwrite it
      tc_fence_before();
      mbar_arrive(&bars->o_free[t]);
      L += 2u * (uint32_t)n_tiles;
      S += (uint32_t)n_tiles;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem);
  }
}

}  // namespace

int prefill_tokens_per_cta(int g) { return kQTiles * (BM / g); }

static PrefillArgs& base_args_host(PrefillArgs& a) { return a; }
static PrefillArgs& base_args_host(PrefillChunkArgs& a) { return a.base; }

template <class Args>
static cudaError_t launch(const Args& args_in, cudaStream_t stream) {
  // per-device set-up: the dynamic shared memory limit is a per-device
  // attribute of each instantiation
  static unsigned long long done_mask = 0;
  Args args = args_in;
  PrefillArgs& a = base_args_host(args);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(done_mask & (1ull << dev))) {
    e = cudaFuncSetAttribute(prefill_attention_kernel<Args>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) done_mask |= 1ull << dev;
  }
  // one persistent CTA per SM over all items
  const long long items = (long long)a.n_mtiles * a.B * a.Hkv;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  static int sm_count[64];
  int n_sm = dev < 64 ? sm_count[dev] : 0;
  if (n_sm == 0) {
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) sm_count[dev] = n_sm;
  }
  const long long grid = items < n_sm ? items : (long long)n_sm;
  // a plain prefill's items of one group run from 1 to n_mtiles KV tiles,
  // and longest first over all groups balances them best: one set (the
  // kernel's plain instantiation does not read the field)
  if constexpr (std::is_same<Args, PrefillChunkArgs>::value)
    a.group_sets = choose_group_sets(a.n_mtiles, a.B, a.Hkv, kQTiles * (BM / a.g), a.T,
                                     args.pos_b, BN, (int)grid);
  else
    a.group_sets = 1;
  prefill_attention_kernel<Args><<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(args);
  return cudaGetLastError();
}

cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t stream) {
  return launch(a, stream);
}

cudaError_t launch_prefill_attention(const PrefillChunkArgs& a, cudaStream_t stream) {
  if (a.base.B > kMaxBatch) return cudaErrorInvalidValue;
  return launch(a, stream);
}

}  // namespace q3a
