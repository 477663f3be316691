// decode_attention.cu — K3 (split-KV decode) and K4 (log-sum-exp combine).
//
// One new token per sequence b at position p = start_pos[b]:
//   qhat_h   = RoPE_p(RMSNorm(q_h) * gamma_q)        for the g heads of group kv
//   khat_new = RoPE_p(RMSNorm(k_new) * gamma_k)      appended at cache row p
//   out_h    = sum_{j <= p} softmax_j(qhat_h . k_j / sqrt(128)) v_j
// where k_j, v_j for j < p are the cache rows as stored (already normalised
// and rotated, never rotated again) and k_p = khat_new, v_p = v_new
// ("Chapter 20, Qwen3 and Qwen3.5", book.ozine.me, §20.3: the new K is
// rotated at start_pos and concatenated; old K already carries its position).
//
// K3: grid (split, kv, b). A split is 1024 consecutive keys of one (b, kv)
// (2048 at head_dim 256). Warp 4 streams the split's K and V in 64-key tiles
// with TMA (128-byte swizzle, 3-stage ring, 32 KB per stage at d = 128). Warps 0-3 each take 16 keys of a
// tile: S = Qhat K^T and O += P V run on the tensor cores as m16n8k16 bf16
// MMAs with the g query heads of the group as the M rows (padded to 16), so
// one pass over the keys serves all g heads. Each warp keeps its own online
// softmax (exp2 domain, lazy rescale); the four warps are merged at the end
// and the split writes (m, l, acc[d]) per head to the workspace.
// The split that holds position p also normalises and rotates k_new, appends
// it and v_new to the caches, and patches them into its shared-memory tile in
// place of the cache row it read (which the caller may not have written yet).
// Cache rows past p are never used: their scores are masked and their values
// zeroed in shared memory before the PV product.
//
// K4: grid (head, b), one thread per output column: merges the splits of a
// head with their log-sum-exp weights and writes bf16.
//
// Gated decode (the global layer of Qwen3-Next / Qwen3.5, "Chapter 20, Qwen3
// and Qwen3.5" §20.4): the same kernels at head_dim 256, with the query taken
// from the first half of each head's 512-element query/gate block, the
// zero-centred norm (scale 1 + w), RoPE on the first d_rot coordinates only
// (frequencies theta^(-2i/d_rot)), and K4 multiplying each output column by
// sigmoid of the gate half. A warp normalises one row there (lane L holds
// elements 8L..8L+7; rotated pairs sit in lanes L and L + d_rot/16), and a
// 64-key stage is 64 KB, so one CTA runs per SM with three stages in flight
// and splits are twice as long, to spread each split's fixed start and merge.
//
// The attention arithmetic is HBM-bound (about 4 flops per cache byte), so the
// design goal is the copy engine never idling: 64 KB+ of loads in flight per
// SM, no per-key shuffles, and the tensor cores doing the dot products.
#include "q3a_internal.h"
#include "q3a_rope.cuh"

namespace q3a {

namespace {

constexpr int kKeysPerTile = 64;
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr uint32_t kBox = 8192;  // 64 keys x 64 d x bf16
constexpr float kRescaleThreshold = 8.0f;
constexpr unsigned kFull = 0xffffffffu;

// Shared-memory layout for head_dim D (128 or 256).
template <int D>
struct DecLayout {
  static constexpr uint32_t kKTile = (D / 64) * kBox;       // 64 keys x D
  static constexpr uint32_t kStageBytes = 2 * kKTile;       // K + V
  static constexpr uint32_t OFF_STAGES = 0;
  static constexpr uint32_t OFF_Q = OFF_STAGES + kStages * kStageBytes;  // bf16 [16][D]
  static constexpr uint32_t OFF_KNEW = OFF_Q + 16 * D * 2;              // bf16 [D]
  static constexpr uint32_t OFF_VNEW = OFF_KNEW + D * 2;                // bf16 [D]
  static constexpr uint32_t OFF_CS = OFF_VNEW + D * 2;                  // float2 [D / 2]
  static constexpr uint32_t OFF_BAR = OFF_CS + D * 4;
  static constexpr uint32_t kSmemBytes = OFF_BAR + 128 + 1024;  // + alignment slack
  // merge area (reuses the stage ring once every tile has been consumed)
  static constexpr uint32_t kMergeAcc = kConsumerWarps * 16 * D * 4;
  static_assert(kMergeAcc + kConsumerWarps * 16 * 8 <= kStages * kStageBytes, "merge area");
  static constexpr int kMinBlocks = D == 128 ? 2 : 1;  // CTAs per SM the registers allow for
  static constexpr float kScaleLog2 = D == 128 ? 0.12751743074380046f   // log2(e) / sqrt(128)
                                               : 0.09016844005556021f;  // log2(e) / sqrt(256)
};

struct DecBars {
  uint64_t full[kStages], empty[kStages];
  int abort_flag;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte offset of 16-byte chunk gc (0..D/8-1 over d) of tile row kt (0..63) in a
// [64 keys][D] tile stored as D/64 128-byte-swizzled [64][64] boxes
__device__ __forceinline__ uint32_t tile_chunk(int kt, int gc) {
  return (gc >> 3) * kBox + kt * 128 + ((((gc & 7) ^ (kt & 7))) << 4);
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Position of sequence b: from the parameters, or from device memory after
// the device-side check (kDevPos).
template <bool kDevPos>
__device__ __forceinline__ int decode_pos(const DecodeArgs& a, int b) {
  return kDevPos ? a.pos_dev[b] : a.start_pos[b];
}

template <int D, bool kGated, bool kDevPos>
__global__ void __launch_bounds__(kThreads, DecLayout<D>::kMinBlocks)
    decode_split_kernel(const __grid_constant__ DecodeArgs a) {
  using L_ = DecLayout<D>;
  constexpr uint32_t kKTile = L_::kKTile, kStageBytes = L_::kStageBytes;
  constexpr uint32_t OFF_STAGES = L_::OFF_STAGES, OFF_Q = L_::OFF_Q, OFF_KNEW = L_::OFF_KNEW;
  constexpr uint32_t OFF_VNEW = L_::OFF_VNEW, OFF_CS = L_::OFF_CS, OFF_BAR = L_::OFF_BAR;
  constexpr float kScaleLog2 = L_::kScaleLog2;
  const int c = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;
  if (kDevPos && *a.pos_valid == 0) return;  // some position out of range: write nothing
  const int p = decode_pos<kDevPos>(a, b);
  const int L = p + 1;  // keys of this sequence, the new one included
  constexpr int kChunk = decode_chunk_keys(D);
  const int n_splits = (L + kChunk - 1) / kChunk;
  if (c >= n_splits) return;
  const int key_begin = c * kChunk;
  const int key_end = min(key_begin + kChunk, L);
  const int n_tiles = (key_end - key_begin + kKeysPerTile - 1) / kKeysPerTile;
  const bool holds_new = (c == n_splits - 1);
  const int g = a.g;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DecBars* bars = reinterpret_cast<DecBars*>(smem + OFF_BAR);
  uint16_t* qs = reinterpret_cast<uint16_t*>(smem + OFF_Q);
  uint16_t* knew_s = reinterpret_cast<uint16_t*>(smem + OFF_KNEW);
  uint16_t* vnew_s = reinterpret_cast<uint16_t*>(smem + OFF_VNEW);
  float2* cs = reinterpret_cast<float2*>(smem + OFF_CS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long bkv = (long long)b * a.Hkv + kv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], kConsumerWarps);
    }
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (kGated) {
    for (int i = threadIdx.x; i < (a.d_rot >> 1); i += kThreads)
      cs[i] = rope_cos_sin(p, a.turn_freq[i]);
  } else if (threadIdx.x < 64) {
    cs[threadIdx.x] = rope_cos_sin(p, a.turn_freq[threadIdx.x]);
  }
  __syncthreads();
  volatile int* abort = &bars->abort_flag;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&a.tm_kc);
      tma_prefetch_desc(&a.tm_vc);
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&bars->empty[s], ((i / kStages) & 1) ^ 1, a.err, kDevTimeoutTma, abort))
          break;
        const int key0 = key_begin + i * kKeysPerTile;
        uint8_t* st = smem + OFF_STAGES + s * kStageBytes;
        mbar_arrive_expect_tx(&bars->full[s], kStageBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(st + c * kBox, &a.tm_kc, &bars->full[s], 64 * c, key0, (int)bkv);
          tma_load_3d(st + kKTile + c * kBox, &a.tm_vc, &bars->full[s], 64 * c, key0, (int)bkv);
        }
        issued = i + 1;
      }
      if (*abort) {
        for (int i = max(0, issued - kStages); i < issued; ++i)
          mbar_wait(&bars->full[i % kStages], (i / kStages) & 1, nullptr, 0, nullptr);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  // 1. qhat for the g heads (rows g..15 zero), and khat_new / v_new if this
  //    split holds position p.
  if constexpr (!kGated) {
    // Qwen3, d = 128: two rows per warp (half-warps), QK-Norm with gamma,
    // rotate-half RoPE over all 128 coordinates
    const int lane16 = lane & 15;
    float glq[4], ghq[4], glk[4], ghk[4];
    unpack4(reinterpret_cast<const uint2*>(a.q_gamma)[lane16], glq);
    unpack4(reinterpret_cast<const uint2*>(a.q_gamma + 64)[lane16], ghq);
    unpack4(reinterpret_cast<const uint2*>(a.k_gamma)[lane16], glk);
    unpack4(reinterpret_cast<const uint2*>(a.k_gamma + 64)[lane16], ghk);
    float2 c_s[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) c_s[j] = cs[4 * lane16 + j];
    const int n_rows = g + (holds_new ? 1 : 0);
    const int n_rows_even = (n_rows + 1) & ~1;
    for (int r = (threadIdx.x >> 4); r < n_rows_even; r += 2 * kConsumerWarps) {
      const bool live = r < n_rows;
      const bool is_k = live && r == g;
      const int rr = live ? r : 0;
      const uint16_t* src = is_k ? a.k_new + bkv * 128
                                 : a.q + ((long long)b * a.Hq + (long long)kv * g + rr) * 128;
      float xl[4], xh[4], ol[4], oh[4];
      unpack4(reinterpret_cast<const uint2*>(src)[lane16], xl);
      unpack4(reinterpret_cast<const uint2*>(src + 64)[lane16], xh);
      float gl[4], gh[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        gl[j] = is_k ? glk[j] : glq[j];
        gh[j] = is_k ? ghk[j] : ghq[j];
      }
      qknorm_rope_halfwarp(xl, xh, gl, gh, c_s, a.eps, ol, oh);
      if (live) {
        uint16_t* dst = is_k ? knew_s : qs + rr * 128;
        reinterpret_cast<uint2*>(dst)[lane16] = pack4(ol);
        reinterpret_cast<uint2*>(dst + 64)[lane16] = pack4(oh);
        if (is_k) {
          // append: k_cache[b, kv, p] = bf16(khat_new), v_cache[b, kv, p] = v_new
          uint16_t* kc = a.k_cache + (bkv * a.S_max + p) * 128;
          uint16_t* vc = a.v_cache + (bkv * a.S_max + p) * 128;
          const uint2* vn = reinterpret_cast<const uint2*>(a.v_new + bkv * 128);
          const uint2 v_lo = vn[lane16], v_hi = vn[16 + lane16];
          reinterpret_cast<uint2*>(kc)[lane16] = pack4(ol);
          reinterpret_cast<uint2*>(kc + 64)[lane16] = pack4(oh);
          reinterpret_cast<uint2*>(vc)[lane16] = v_lo;
          reinterpret_cast<uint2*>(vc)[16 + lane16] = v_hi;
          reinterpret_cast<uint2*>(vnew_s)[lane16] = v_lo;
          reinterpret_cast<uint2*>(vnew_s)[16 + lane16] = v_hi;
        }
      }
    }
    // zero the padding rows g..15 of qhat
    for (int idx = threadIdx.x; idx < (16 - g) * 64; idx += 128)
      reinterpret_cast<uint32_t*>(qs + g * 128)[idx] = 0u;
  }
  if constexpr (kGated) {
    // gated layer, d = 256: one row per warp, zero-centred norm (scale 1 + w),
    // RoPE of the first d_rot coordinates; the query is the first half of the
    // head's 512-element query/gate block
    float sq[8], sk[8];
    unpack8(reinterpret_cast<const uint4*>(a.q_gamma)[lane], sq);
    unpack8(reinterpret_cast<const uint4*>(a.k_gamma)[lane], sk);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sq[e] += 1.0f;
      sk[e] += 1.0f;
    }
    const int hl = a.d_rot >> 4;  // rotated pairs sit in lanes L and L + hl
    const bool rotated = lane < 2 * hl;
    const bool lower = lane < hl;
    const int partner = rotated ? (lower ? lane + hl : lane - hl) : lane;
    const int ang0 = rotated ? 8 * (lower ? lane : lane - hl) : 0;
    const int n_rows = g + (holds_new ? 1 : 0);
    for (int r = warp; r < n_rows; r += kConsumerWarps) {
      const bool is_k = r == g;
      const uint16_t* src =
          is_k ? a.k_new + bkv * D : a.q + ((long long)b * a.Hq + (long long)kv * g + r) * (2 * D);
      float x[8], y[8], o8[8];
      unpack8(reinterpret_cast<const uint4*>(src)[lane], x);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(kFull, ss, off);
      const float inv_rms = rsqrtf(ss * (1.0f / D) + a.eps);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = x[e] * inv_rms * (is_k ? sk[e] : sq[e]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float yp = __shfl_sync(kFull, y[e], partner);
        if (rotated) {
          const float2 c_s = cs[ang0 + e];
          o8[e] = lower ? y[e] * c_s.x - yp * c_s.y : y[e] * c_s.x + yp * c_s.y;
        } else {
          o8[e] = y[e];
        }
      }
      const uint4 packed = pack8(o8);
      if (is_k) {
        // append: k_cache[b, kv, p] = bf16(khat_new), v_cache[b, kv, p] = v_new
        const uint4 vn = reinterpret_cast<const uint4*>(a.v_new + bkv * D)[lane];
        reinterpret_cast<uint4*>(a.k_cache + (bkv * a.S_max + p) * D)[lane] = packed;
        reinterpret_cast<uint4*>(a.v_cache + (bkv * a.S_max + p) * D)[lane] = vn;
        reinterpret_cast<uint4*>(knew_s)[lane] = packed;
        reinterpret_cast<uint4*>(vnew_s)[lane] = vn;
      } else {
        reinterpret_cast<uint4*>(qs + r * D)[lane] = packed;
      }
    }
    // zero the padding rows g..15 of qhat
    for (int idx = threadIdx.x; idx < (16 - g) * (D / 2); idx += 128)
      reinterpret_cast<uint32_t*>(qs + g * D)[idx] = 0u;
  }
  consumer_sync();

  // 2. A fragments of qhat (16 x D): rows lane/4 and lane/4 + 8
  const int r0 = lane >> 2, cq = lane & 3;
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int col = ks * 16 + 2 * cq;
    qa[ks][0] = *reinterpret_cast<const uint32_t*>(qs + r0 * D + col);
    qa[ks][1] = *reinterpret_cast<const uint32_t*>(qs + (r0 + 8) * D + col);
    qa[ks][2] = *reinterpret_cast<const uint32_t*>(qs + r0 * D + col + 8);
    qa[ks][3] = *reinterpret_cast<const uint32_t*>(qs + (r0 + 8) * D + col + 8);
  }

  float o[D / 8][4];
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

  bool ok = true;
  for (int i = 0; i < n_tiles; ++i) {
    const int s = i % kStages;
    ok = __all_sync(kFull,
                    mbar_wait(&bars->full[s], (i / kStages) & 1, a.err, kDevTimeoutDecode, abort));
    if (!ok) break;
    uint8_t* st = smem + OFF_STAGES + s * kStageBytes;
    const int kt0 = warp * 16;                         // first tile row of this warp
    const int kw0 = key_begin + i * kKeysPerTile + kt0;  // its first key
    if (kw0 < L) {
      if (kw0 + 15 >= L - 1) {
        // patch the new key / value in, zero values past the end
        for (int rr = 0; rr < 16; ++rr) {
          const int key = kw0 + rr;
          if (key < L - 1) continue;
          const bool is_v = lane >= 16;
          // keys past the end are masked; only their values are zeroed
          if (key != L - 1 && !is_v) continue;
#pragma unroll
          for (int gc = lane & 15; gc < D / 8; gc += 16) {
            uint8_t* dst = st + (is_v ? kKTile : 0) + tile_chunk(kt0 + rr, gc);
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (key == L - 1) val = reinterpret_cast<const uint4*>(is_v ? vnew_s : knew_s)[gc];
            *reinterpret_cast<uint4*>(dst) = val;
          }
        }
        __syncwarp();
      }
      const uint32_t kbase = smem_u32(st);
      const uint32_t vbase = kbase + kKTile;
      // S = Qhat K^T for 16 keys: two n8 tiles
      float sc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        const int kt = kt0 + nt * 8 + (lane & 7);
#pragma unroll
        for (int kp = 0; kp < D / 32; ++kp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + tile_chunk(kt, 4 * kp + (lane >> 3)), b0, b1, b2, b3);
          mma16816(sc[nt], qa[2 * kp], b0, b1);
          mma16816(sc[nt], qa[2 * kp + 1], b2, b3);
        }
      }
      // mask keys past the end, scale into the exp2 domain
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kw0 + nt * 8 + 2 * cq + (e & 1);
          sc[nt][e] = key < L ? sc[nt][e] * kScaleLog2 : -INFINITY;
        }
      float tA = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float tB = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      tA = fmaxf(tA, __shfl_xor_sync(kFull, tA, 1));
      tA = fmaxf(tA, __shfl_xor_sync(kFull, tA, 2));
      tB = fmaxf(tB, __shfl_xor_sync(kFull, tB, 1));
      tB = fmaxf(tB, __shfl_xor_sync(kFull, tB, 2));
      const bool moveA = tA > mA + kRescaleThreshold;
      const bool moveB = tB > mB + kRescaleThreshold;
      if (moveA || moveB) {
        const float alA = moveA ? ex2(mA - tA) : 1.f;
        const float alB = moveB ? ex2(mB - tB) : 1.f;
        mA = moveA ? tA : mA;
        mB = moveB ? tB : mB;
        lA *= alA;
        lB *= alB;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          o[dn][0] *= alA;
          o[dn][1] *= alA;
          o[dn][2] *= alB;
          o[dn][3] *= alB;
        }
      }
      float pr[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        pr[nt][0] = ex2(sc[nt][0] - mA);
        pr[nt][1] = ex2(sc[nt][1] - mA);
        pr[nt][2] = ex2(sc[nt][2] - mB);
        pr[nt][3] = ex2(sc[nt][3] - mB);
        lA += pr[nt][0] + pr[nt][1];
        lB += pr[nt][2] + pr[nt][3];
      }
      const uint32_t pa[4] = {pack_bf16x2(pr[0][0], pr[0][1]), pack_bf16x2(pr[0][2], pr[0][3]),
                              pack_bf16x2(pr[1][0], pr[1][1]), pack_bf16x2(pr[1][2], pr[1][3])};
      // O += P V over the 16 keys: D/8 n8 tiles of d
      const int vkt = kt0 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + tile_chunk(vkt, 2 * dp + (lane >> 4)), b0, b1, b2, b3);
        mma16816(o[2 * dp], pa, b0, b1);
        mma16816(o[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->empty[s]);
  }

  // 3. merge the four warps; write this split's (m, l, acc) per head
  lA += __shfl_xor_sync(kFull, lA, 1);
  lA += __shfl_xor_sync(kFull, lA, 2);
  lB += __shfl_xor_sync(kFull, lB, 1);
  lB += __shfl_xor_sync(kFull, lB, 2);
  consumer_sync();  // every consumer is past its last tile read
  ok = ok && !*abort;
  float* acc_s = reinterpret_cast<float*>(smem + OFF_STAGES);  // [4][16][D]
  float* ml_s = acc_s + kConsumerWarps * 16 * D;               // [4][16][2]
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) {
    const int col = dn * 8 + 2 * cq;
    acc_s[(warp * 16 + r0) * D + col] = o[dn][0];
    acc_s[(warp * 16 + r0) * D + col + 1] = o[dn][1];
    acc_s[(warp * 16 + r0 + 8) * D + col] = o[dn][2];
    acc_s[(warp * 16 + r0 + 8) * D + col + 1] = o[dn][3];
  }
  if (cq == 0) {
    ml_s[(warp * 16 + r0) * 2] = mA;
    ml_s[(warp * 16 + r0) * 2 + 1] = lA;
    ml_s[(warp * 16 + r0 + 8) * 2] = mB;
    ml_s[(warp * 16 + r0 + 8) * 2 + 1] = lB;
  }
  consumer_sync();
  if (!ok) return;
  constexpr int kPartial = decode_partial_floats(D);
  float* part = a.partial + ((bkv * a.split_stride + c) * g) * kPartial;
  for (int idx = threadIdx.x; idx < g * D; idx += 128) {
    const int h = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, ml_s[(w * 16 + h) * 2]);
    float lsum = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = ml_s[(w * 16 + h) * 2];
      const float wt = mw == -INFINITY ? 0.f : ex2(mw - M);
      lsum += wt * ml_s[(w * 16 + h) * 2 + 1];
      acc += wt * acc_s[(w * 16 + h) * D + d];
    }
    float* ph = part + h * kPartial;
    if (d == 0) {
      ph[0] = M;
      ph[1] = lsum;
    }
    ph[2 + d] = acc;
  }
}

template <int D, bool kGated, bool kDevPos>
__global__ void __launch_bounds__(D) decode_combine_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int kPartial = decode_partial_floats(D);
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  if (kDevPos && *a.pos_valid == 0) return;
  const int g = a.g, kv = h / g, j = h % g;
  const int L = decode_pos<kDevPos>(a, b) + 1;
  const int n_splits = (L + decode_chunk_keys(D) - 1) / decode_chunk_keys(D);
  const float* base =
      a.partial + ((((long long)b * a.Hkv + kv) * a.split_stride) * g + j) * kPartial;
  const long long split_step = (long long)g * kPartial;
  float M = -INFINITY;
  for (int c = 0; c < n_splits; ++c) M = fmaxf(M, base[c * split_step]);
  float lsum = 0.f, acc = 0.f;
  for (int c = 0; c < n_splits; ++c) {
    const float* pc = base + c * split_step;
    const float wt = ex2(pc[0] - M);
    lsum += wt * pc[1];
    acc += wt * pc[2 + d];
  }
  float v = acc / lsum;
  if constexpr (kGated) {
    // z = o * sigmoid(gate), the gate being the second half of the head's
    // query/gate block: sigmoid(x) = 1 / (1 + 2^(-x log2 e))
    const float gt = __uint_as_float((uint32_t)a.q[((long long)b * a.Hq + h) * (2 * D) + D + d]
                                     << 16);
    v *= 1.0f / (1.0f + ex2(-1.4426950408889634f * gt));
  }
  a.out[((long long)b * a.Hq + h) * D + d] = (uint16_t)(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

// Device-side validation of positions that live in device memory: every
// start_pos[b] must satisfy 0 <= p < S_max. One block; writes the verdict and
// the error word (0, or kErrWordRange) before any decode kernel runs.
__global__ void __launch_bounds__(256) decode_pos_check_kernel(const int32_t* pos, int B, int S_max,
                                                               uint32_t* err, uint32_t* valid) {
  int bad = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int p = pos[b];
    bad |= (p < 0 || p >= S_max) ? 1 : 0;
  }
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    *valid = bad ? 0u : 1u;
    *err = bad ? kErrWordRange : 0u;
  }
}

}  // namespace

template <int D, bool kGated>
static cudaError_t launch(const DecodeArgs& a, cudaStream_t stream) {
  constexpr uint32_t kSmemBytes = DecLayout<D>::kSmemBytes;
  static unsigned long long attr_done_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(attr_done_mask & (1ull << dev))) {
    e = cudaFuncSetAttribute(decode_split_kernel<D, kGated, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_split_kernel<D, kGated, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_done_mask |= 1ull << dev;
  }
  if (a.B == 0) return cudaSuccess;
  dim3 grid1(a.max_splits, a.Hkv, a.B);
  dim3 grid2(a.Hq, a.B);
  if (a.pos_dev) {
    // positions unknown on the host: the check decides, and every split a
    // sequence may need is launched (the ones past its length exit at once)
    decode_pos_check_kernel<<<1, 256, 0, stream>>>(a.pos_dev, a.B, a.S_max, a.err, a.pos_valid);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_split_kernel<D, kGated, true><<<grid1, kThreads, kSmemBytes, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_combine_kernel<D, kGated, true><<<grid2, D, 0, stream>>>(a);
    return cudaGetLastError();
  }
  decode_split_kernel<D, kGated, false><<<grid1, kThreads, kSmemBytes, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<D, kGated, false><<<grid2, D, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  return launch<128, false>(a, stream);
}

cudaError_t launch_gated_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.d_rot < 0 || a.d_rot > 256 || (a.d_rot & 15)) return cudaErrorInvalidValue;
  return launch<kGatedD, true>(a, stream);
}

}  // namespace q3a
