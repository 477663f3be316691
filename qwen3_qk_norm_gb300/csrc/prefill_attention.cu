// prefill_attention.cu — K2, causal grouped-query attention on tcgen05.
//
// Computes, for every query row (b, i, h) with normalised+rotated qhat and the
// normalised+rotated keys khat_j of group h / g:
//   out = sum_{j <= i} softmax_j(qhat . khat_j / sqrt(128)) v_j
// ("7.2 Qwen3 full-scale implementation", §7.2.1 GroupedQueryAttention.forward:
// repeat_interleave of the KV heads, triu causal mask, softmax of the scores
// over head_dim ** 0.5, product with the values).
//
// Tiling. One CTA owns one M tile of 128 query rows: the g query heads of one
// KV group for 128/g consecutive tokens, packed row r = (token t0 + r/g,
// head kv*g + r%g). Every K/V tile it loads is therefore used by all g heads
// of the group, so each K/V byte is read once per M tile rather than g times.
// KV tiles are 128 keys. Tiles entirely above the causal diagonal are never
// loaded; the diagonal tiles are masked per element.
//
// Roles (192 threads):
//   warps 0-3  softmax + epilogue: thread r owns row r of S and O in tensor
//              memory (TMEM lane r);
//   warp 4     TMA producer: Q once, then K_j and V_j into a 2-stage ring;
//   warp 5     MMA issuer (one thread): S = Q K^T into TMEM, O += P V into TMEM.
// Order of the MMA stream: S_0, then for each j: S_{j+1} (as soon as the
// softmax warps have pulled S_j into registers), PV_j (once P_j is in shared
// memory). So the QK^T of the next tile runs while the softmax of this tile
// computes its exponentials.
//
// Online softmax in the exp2 domain with a lazy rescale: the running row max m
// is only moved (and O, l rescaled by 2^(m_old - m_new)) when the tile max
// exceeds it by more than 8, so P stays below 2^8 and most tiles skip the
// TMEM read-modify-write of O.
//
// Every mbarrier wait is bounded (q3a_device.cuh); a timeout sets the error
// word, all roles unwind, in-flight copies and MMAs are drained and TMEM is
// freed before the CTA exits.
#include "q3a_device.cuh"
#include "q3a_internal.h"

namespace q3a {

namespace {

constexpr int BM = 128;  // query rows per CTA
constexpr int BN = 128;  // keys per KV tile
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr uint32_t kHalf = 16384;      // 128 rows x 128 bytes
constexpr uint32_t kTile = 2 * kHalf;  // 128 rows x 128 bf16
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + kTile;
constexpr uint32_t OFF_V = OFF_K + kStages * kTile;
constexpr uint32_t OFF_P = OFF_V + kStages * kTile;
constexpr uint32_t OFF_BAR = OFF_P + kTile;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 256;                    // S: 0..127, O: 128..255
constexpr float kScaleLog2 = 0.12751743074380046f;     // log2(e) / sqrt(128)
constexpr float kRescaleThreshold = 8.0f;
constexpr unsigned kFull = 0xffffffffu;

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full, s_free, p_full, o_done, drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

__device__ __forceinline__ uint32_t p_chunk_offset(int row, int chunk16) {
  // byte offset of 16-byte chunk `chunk16` (0..15, 8 keys each) of row `row`
  // in a K-major, 128-byte-swizzled 128 x 128 bf16 tile made of two halves
  const int half = chunk16 >> 3, c = chunk16 & 7;
  return half * kHalf + (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_attention_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: longest M tiles first ------------------------------------
  const int bk_count = a.B * a.Hkv;
  const int mt = a.n_mtiles - 1 - (int)(blockIdx.x / bk_count);
  const int bk = (int)(blockIdx.x % bk_count);
  const int b = bk / a.Hkv, kv = bk % a.Hkv;
  const int g = a.g;
  const int rows_tok = BM / g;
  const int t0 = mt * rows_tok;
  const int t_last = min(t0 + rows_tok, a.T) - 1;
  const int n_tiles = t_last / BN + 1;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 128);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc<kTmemCols>(&bars->tmem_base);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tmem_s = tmem;
  const uint32_t tmem_o = tmem + 128;
  volatile int* abort = &bars->abort_flag;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&a.tm_q);
      tma_prefetch_desc(&a.tm_k);
      tma_prefetch_desc(&a.tm_v);
      mbar_arrive_expect_tx(&bars->q_full, kTile);
      tma_load_4d(smem + OFF_Q, &a.tm_q, &bars->q_full, 0, kv * g, t0, b);
      tma_load_4d(smem + OFF_Q + kHalf, &a.tm_q, &bars->q_full, 64, kv * g, t0, b);
      int nk = 0, nv = 0;  // K and V tiles issued
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % kStages;
        const uint32_t par = ((j / kStages) & 1) ^ 1;
        if (!mbar_wait(&bars->k_empty[s], par, a.err, kDevTimeoutTma, abort)) break;
        mbar_arrive_expect_tx(&bars->k_full[s], kTile);
        uint8_t* kd = smem + OFF_K + s * kTile;
        tma_load_3d(kd, &a.tm_k, &bars->k_full[s], 0, j * BN, b * a.Hkv + kv);
        tma_load_3d(kd + kHalf, &a.tm_k, &bars->k_full[s], 64, j * BN, b * a.Hkv + kv);
        nk = j + 1;
        if (!mbar_wait(&bars->v_empty[s], par, a.err, kDevTimeoutTma, abort)) break;
        mbar_arrive_expect_tx(&bars->v_full[s], kTile);
        uint8_t* vd = smem + OFF_V + s * kTile;
        tma_load_4d(vd, &a.tm_v, &bars->v_full[s], 0, kv, j * BN, b);
        tma_load_4d(vd + kHalf, &a.tm_v, &bars->v_full[s], 64, kv, j * BN, b);
        nv = j + 1;
      }
      if (*abort) {
        // let every copy that was issued land before the CTA goes away
        mbar_wait(&bars->q_full, 0, nullptr, 0, nullptr);
        for (int j = max(0, nk - kStages); j < nk; ++j)
          mbar_wait(&bars->k_full[j % kStages], (j / kStages) & 1, nullptr, 0, nullptr);
        for (int j = max(0, nv - kStages); j < nv; ++j)
          mbar_wait(&bars->v_full[j % kStages], (j / kStages) & 1, nullptr, 0, nullptr);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, 128, 0, 1);
      const uint32_t q_addr = smem_u32(smem + OFF_Q);
      const uint32_t p_addr = smem_u32(smem + OFF_P);
      bool ok = mbar_wait(&bars->q_full, 0, a.err, kDevTimeoutMma, abort);
      // S_0
      ok = ok && mbar_wait(&bars->k_full[0], 0, a.err, kDevTimeoutMma, abort);
      if (ok) {
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + OFF_K);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma_bf16_ss(tmem_s, smem_desc_sw128(q_addr + off, 16, 1024),
                      smem_desc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&bars->s_full);
        mma_commit(&bars->k_empty[0]);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int s = j % kStages;
        if (j + 1 < n_tiles) {
          const int s1 = (j + 1) % kStages;
          ok = mbar_wait(&bars->k_full[s1], ((j + 1) / kStages) & 1, a.err, kDevTimeoutMma,
                         abort) &&
               mbar_wait(&bars->s_free, j & 1, a.err, kDevTimeoutMma, abort);
          if (!ok) break;
          tc_fence_after();
          const uint32_t k_addr = smem_u32(smem + OFF_K + s1 * kTile);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            mma_bf16_ss(tmem_s, smem_desc_sw128(q_addr + off, 16, 1024),
                        smem_desc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0);
          }
          mma_commit(&bars->s_full);
          mma_commit(&bars->k_empty[s1]);
        }
        ok = mbar_wait(&bars->p_full, j & 1, a.err, kDevTimeoutMma, abort) &&
             mbar_wait(&bars->v_full[s], (j / kStages) & 1, a.err, kDevTimeoutMma, abort);
        if (!ok) break;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(smem + OFF_V + s * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // A = P (K-major over keys), B = V (MN-major: 64-wide d blocks
          // 16 KB apart, 8-key groups 1 KB apart; 16 keys = 2 KB per step)
          const uint32_t a_off = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma_bf16_ss(tmem_o, smem_desc_sw128(p_addr + a_off, 16, 1024),
                      smem_desc_sw128(v_addr + kk * 2048, kHalf, 1024), idesc_o,
                      (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->o_done);
        mma_commit(&bars->v_empty[s]);
      }
      // drain: every MMA issued above has completed once this phase completes
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, nullptr, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // row of S / O, TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int tok = t0 + r / g;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      ok = __all_sync(kFull, mbar_wait(&bars->s_full, j & 1, a.err, kDevTimeoutSoftmax, abort));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem_s + lane_off + c * 32, sr[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->s_free);

      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(sr[c][e]);
      const int key0 = j * BN;
      if (key0 + BN - 1 > tok) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (key0 + e > tok) s[e] = -INFINITY;
      }
      float mt = s[0];
#pragma unroll
      for (int e = 1; e < 128; ++e) mt = fmaxf(mt, s[e]);
      const float m_tile = mt * kScaleLog2;
      const bool move = m_tile > m + kRescaleThreshold;
      const float m_new = move ? m_tile : m;
      const float alpha = move ? ex2(m - m_new) : 1.0f;

      // PV_{j-1} must be complete before O is rescaled and P is overwritten
      if (j > 0) {
        ok = __all_sync(kFull,
                        mbar_wait(&bars->o_done, (j - 1) & 1, a.err, kDevTimeoutSoftmax, abort));
        if (!ok) break;
      }
      tc_fence_after();
      if (j > 0 && __any_sync(kFull, move)) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem_o + lane_off + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tmem_o + lane_off + c * 32, o);
        }
        tmem_wait_st();
      }
      m = m_new;
      l *= alpha;

      float sum = 0.f;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        uint32_t w[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const float p0 = ex2(fmaf(s[ch * 8 + 2 * e2], kScaleLog2, -m));
          const float p1 = ex2(fmaf(s[ch * 8 + 2 * e2 + 1], kScaleLog2, -m));
          sum += p0 + p1;
          w[e2] = pack_bf16x2(p0, p1);
        }
        *reinterpret_cast<uint4*>(smem + OFF_P + p_chunk_offset(r, ch)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      l += sum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }
    // ---- epilogue: O / l -> bf16 -> out
    if (ok) {
      ok = __all_sync(kFull, mbar_wait(&bars->o_done, (n_tiles - 1) & 1, a.err,
                                       kDevTimeoutEpilogue, abort));
    }
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const bool store = tok < a.T;
      uint16_t* orow =
          a.out + (((long long)b * a.T + tok) * a.Hq + (long long)kv * g + (r % g)) * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem_o + lane_off + c * 32, o);
        tmem_wait_ld();
        if (store) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv_l,
                              __uint_as_float(o[q4 * 8 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv_l,
                              __uint_as_float(o[q4 * 8 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv_l,
                              __uint_as_float(o[q4 * 8 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv_l,
                              __uint_as_float(o[q4 * 8 + 7]) * inv_l);
            reinterpret_cast<uint4*>(orow + c * 32)[q4] = w;
          }
        }
      }
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

cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t stream) {
  // the dynamic shared memory limit is a per-device attribute of the function
  static unsigned long long attr_done_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !(attr_done_mask & (1ull << dev))) {
    e = cudaFuncSetAttribute(prefill_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done_mask |= 1ull << dev;
  }
  const long long grid = (long long)a.n_mtiles * a.B * a.Hkv;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prefill_attention_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace q3a
