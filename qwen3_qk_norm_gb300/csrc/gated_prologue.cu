// gated_prologue.cu — K5, the prologue of the gated global-attention layer of
// Qwen3-Next / Qwen3.5 (head_dim 256).
//
// Per head row x (d = 256 bf16):
//   y_i = x_i * rsqrt(mean(x^2) + eps) * (1 + w_i)              (fp32)
//   for i < d_r/2, with a_i = p * theta^(-2i/d_r):
//     y'_i         = y_i cos a_i - y_{i+d_r/2} sin a_i
//     y'_{i+d_r/2} = y_{i+d_r/2} cos a_i + y_i sin a_i
//   coordinates d_r .. 255 pass through; one rounding to bf16 at the end.
// Sources: "Chapter 20, Qwen3 and Qwen3.5" §20.4 (norm weight initialised to
// 0 and applied as 1 + w; per-head norm of Q and K, then RoPE; partial rotary
// over the first d_r coordinates with d_r as the frequency denominator) and
// "14. The Qwen family", Qwen3-Next section (head_dim 256, RoPE on 64 dims).
// The query of head h is the first half of the 512-element block that the
// query projection emits for that head; the second half (the gate) is left for
// the attention kernel's epilogue and never read here.
//
// Layout of the work (HBM-bound stream, as in the Qwen3 prologue): a CTA owns
// a few consecutive tokens. Their key rows are contiguous and come in with one
// bulk copy; each query row is a 512-byte bulk copy out of the interleaved
// query/gate projection. A warp owns a row. Lanes L < d_r/8 hold rotated
// pairs: elements 4L..4L+3 and their partners d_r/2 + 4L..d_r/2 + 4L+3, so
// each pair (i, i + d_r/2) sits in one lane and the rotation needs no
// exchange; the other lanes hold eight consecutive pass-through elements from
// d_r on, and rotate by the angle 0 (cos 1, sin 0) with the same
// instructions, so no lane branches. Q rows go back out as one
// block per CTA ([B, T, Hq, 256] keeps the token order), K rows one 512-byte
// store each into the head-major [B, Hkv, T, 256] layout.
//
// A chunk against the caches ("Chapter 20, Qwen3 and Qwen3.5" §20.3: the
// position counter starts at the number of cached tokens) is the same kernel
// with a per-sequence start position: token t of sequence b is rotated at
// pos_b[b] + t and its key and value land in cache row pos_b[b] + t.
#include "q3a_internal.h"
#include "q3a_rope.cuh"

namespace q3a {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxTok = 8;
constexpr int kRowBytes = kGatedD * 2;
constexpr int kMaxRows = 192;  // (Hq + Hkv) rows of one token must fit the staging buffer

__host__ __device__ __forceinline__ const GatedPrologueArgs& base_args(const GatedPrologueArgs& a) {
  return a;
}
__host__ __device__ __forceinline__ const GatedPrologueArgs& base_args(
    const GatedPrologueChunkArgs& a) {
  return a.base;
}
GatedPrologueArgs& base_args(GatedPrologueArgs& a) { return a; }
GatedPrologueArgs& base_args(GatedPrologueChunkArgs& a) { return a.base; }
__device__ __forceinline__ int chunk_start(const GatedPrologueArgs&, long long) { return 0; }
__device__ __forceinline__ int chunk_start(const GatedPrologueChunkArgs& a, long long b) {
  return a.pos_b[b];
}

template <class Args>
__global__ void __launch_bounds__(kThreads)
    gated_prologue_kernel(const __grid_constant__ Args args) {
  const GatedPrologueArgs& a = base_args(args);
  extern __shared__ __align__(128) uint8_t smem[];
  // per (token, lane): the cos / sin of the lane's four pair angles
  // (1 and 0 for lanes without rotated pairs)
  __shared__ __align__(16) float4 cos_s[kMaxTok][32];
  __shared__ __align__(16) float4 sin_s[kMaxTok][32];
  __shared__ uint64_t bar[2];  // one per half of the CTA's tokens
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hq = a.Hq, Hkv = a.Hkv;
  const long long n_tok = (long long)a.B * a.T;
  const long long tok0 = (long long)blockIdx.x * a.tok_per_cta;
  const int tok_here = (int)min((long long)a.tok_per_cta, n_tok - tok0);
  uint16_t* rows_q = reinterpret_cast<uint16_t*>(smem);  // [tok][Hq][256]
  uint16_t* rows_k = rows_q + (size_t)a.tok_per_cta * Hq * kGatedD;  // [tok][Hkv][256]
  uint16_t* rows_v = rows_k + (size_t)a.tok_per_cta * Hkv * kGatedD;  // [tok][Hkv][256]
  // The tokens are taken in two halves, each with its own barrier: the first
  // half is normalised and its stores are issued while the second is still
  // arriving. Half h covers tokens [h ? tok_a : 0, h ? tok_here : tok_a).
  const int tok_a = (tok_here + 1) >> 1;
  const int vrows = a.v ? Hkv : 0;

  if (warp == 0) {
    if (lane == 0) {
      mbar_init(&bar[0], 1);
      mbar_init(&bar[1], 1);
      fence_mbar_init();
      for (int h = 0; h < 2; ++h) {
        const int t_lo = h ? tok_a : 0, n = (h ? tok_here : tok_a) - t_lo;
        if (n == 0) continue;
        const uint32_t kv_bytes = (uint32_t)n * Hkv * kRowBytes;
        mbar_arrive_expect_tx(&bar[h], (uint32_t)n * (Hq + Hkv + vrows) * kRowBytes);
        bulk_load(rows_k + (size_t)t_lo * Hkv * kGatedD, a.k + (tok0 + t_lo) * Hkv * kGatedD,
                  kv_bytes, &bar[h]);
        if (vrows)
          bulk_load(rows_v + (size_t)t_lo * Hkv * kGatedD, a.v + (tok0 + t_lo) * Hkv * kGatedD,
                    kv_bytes, &bar[h]);
      }
    }
    __syncwarp();
    for (int r = lane; r < tok_here * Hq; r += 32)  // query halves of the q|gate blocks
      bulk_load(rows_q + (size_t)r * kGatedD, a.qg + (tok0 * Hq + r) * (2 * kGatedD), kRowBytes,
                &bar[r >= tok_a * Hq ? 1 : 0]);
  }
  if (blockIdx.x == 0 && warp == 1) {
    if (a.err_clear && lane == 0) *a.err_clear = 0u;
    if (a.logit_bound) {
      float gq = 0.f, gk = 0.f;
      for (int i = lane; i < kGatedD; i += 32) {
        gq = fmaxf(gq, fabsf(1.0f + __uint_as_float((uint32_t)a.q_w[i] << 16)));
        gk = fmaxf(gk, fabsf(1.0f + __uint_as_float((uint32_t)a.k_w[i] << 16)));
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        gq = fmaxf(gq, __shfl_xor_sync(0xffffffffu, gq, o));
        gk = fmaxf(gk, __shfl_xor_sync(0xffffffffu, gk, o));
      }
      if (lane == 0) *a.logit_bound = 16.0f * gq * gk * 1.4426950408889634f;
    }
  }
  // (b, t) of the CTA's first token; the others by counting
  const long long b_first = tok0 / a.T;
  const int t_first = (int)(tok0 - b_first * a.T);
  // lane layout (see the top of the file)
  const int nrot = a.d_r >> 3;  // lanes holding rotated pairs
  const bool rotated = lane < nrot;
  const int off_a = rotated ? 4 * lane : a.d_r + 8 * (lane - nrot);
  const int off_b = rotated ? (a.d_r >> 1) + 4 * lane : off_a + 4;
  // rotation table of this CTA's tokens while the rows are in flight
  float* cos_f = reinterpret_cast<float*>(cos_s);
  float* sin_f = reinterpret_cast<float*>(sin_s);
  for (int e = tid; e < tok_here * 128; e += kThreads) {
    const int tt = e >> 7, i = e & 127;  // i = 4 * lane + j
    float c = 1.0f, sn = 0.0f;
    if (i < (a.d_r >> 1)) {
      long long b;
      int t;
      token_bt(b_first, t_first, tt, a.T, b, t);
      const float2 c_s = rope_cos_sin((long long)chunk_start(args, b) + t, a.turn_freq[i]);
      c = c_s.x;
      sn = c_s.y;
    }
    cos_f[e] = c;
    sin_f[e] = sn;
  }
  __syncthreads();  // barriers initialised, table written

  // token of a row: (rr + 0.5) / H is below kMaxTok and at least 0.5 / H >=
  // 2^-9 away from an integer, far more than its fp32 error, so truncation
  // gives rr / H exactly
  const float inv_hq = 1.0f / (float)Hq, inv_hkv = 1.0f / (float)Hkv;
  bool issued = false;
  for (int h = 0; h < 2; ++h) {
    const int t_lo = h ? tok_a : 0, t_hi = h ? tok_here : tok_a;
    if (t_hi == t_lo) break;  // one token: no second half (uniform over the CTA)
    mbar_wait(&bar[h], 0, nullptr, 0, nullptr);
    const int nq = (t_hi - t_lo) * Hq;
    const int rows = nq + (t_hi - t_lo) * Hkv;
    // scales 1 + w of the lane's elements for the current tensor (a warp's
    // rows run through Q first, then K: one reload at the switch)
    float sa[4], sb[4];
    int scale_of = -1;
    for (int q = warp; q < rows; q += kWarps) {
      const int is_q = q < nq ? 1 : 0;
      if (is_q != scale_of) {
        const uint16_t* w = is_q ? a.q_w : a.k_w;
        unpack4(*reinterpret_cast<const uint2*>(w + off_a), sa);
        unpack4(*reinterpret_cast<const uint2*>(w + off_b), sb);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          sa[j] += 1.0f;
          sb[j] += 1.0f;
        }
        scale_of = is_q;
      }
      const int rr = is_q ? t_lo * Hq + q : t_lo * Hkv + (q - nq);  // row within the CTA
      const int tt = (int)(((float)rr + 0.5f) * (is_q ? inv_hq : inv_hkv));
      uint16_t* row = (is_q ? rows_q : rows_k) + (size_t)rr * kGatedD;
      float xa[4], xb[4], oa[4], ob[4];
      unpack4(*reinterpret_cast<const uint2*>(row + off_a), xa);
      unpack4(*reinterpret_cast<const uint2*>(row + off_b), xb);
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) ss = fmaf(xa[j], xa[j], fmaf(xb[j], xb[j], ss));
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float inv_rms = rsqrtf(ss * (1.0f / kGatedD) + a.eps);
      const float4 c4 = cos_s[tt][lane], s4 = sin_s[tt][lane];
      const float c[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float ya = xa[j] * inv_rms * sa[j];
        const float yb = xb[j] * inv_rms * sb[j];
        oa[j] = fmaf(yb, -sn[j], ya * c[j]);  // y_i c - y_{i+d_r/2} s
        ob[j] = fmaf(ya, sn[j], yb * c[j]);   // y_{i+d_r/2} c + y_i s
      }
      *reinterpret_cast<uint2*>(row + off_a) = pack4(oa);
      *reinterpret_cast<uint2*>(row + off_b) = pack4(ob);
    }
    fence_proxy_async_smem();  // the bulk stores below read what was just written
    __syncthreads();

    if (tid == 0) {
      bulk_store(a.qhat + (tok0 + t_lo) * Hq * kGatedD, rows_q + (size_t)t_lo * Hq * kGatedD,
                 (uint32_t)nq * kRowBytes);
      issued = true;
    }
    for (int rr = t_lo * Hkv + tid; rr < t_hi * Hkv; rr += kThreads) {
      const int tt = rr / Hkv, kv = rr - tt * Hkv;
      long long b;
      int t;
      token_bt(b_first, t_first, tt, a.T, b, t);
      const long long dst_row = (b * Hkv + kv) * a.khat_rows + chunk_start(args, b) + t;
      bulk_store(a.khat + dst_row * kGatedD, rows_k + (size_t)rr * kGatedD, kRowBytes);
      if (vrows)
        bulk_store(a.v_cache + dst_row * kGatedD, rows_v + (size_t)rr * kGatedD, kRowBytes);
      issued = true;
    }
  }
  if (issued) bulk_commit_and_wait_read();  // shared memory stays valid until read
}

template <class Args>
cudaError_t launch(const Args& args_in, cudaStream_t stream) {
  Args args = args_in;
  GatedPrologueArgs& a = base_args(args);
  const long long n_tok = (long long)a.B * a.T;
  if (n_tok == 0) return cudaSuccess;
  const int rows_per_tok = a.Hq + (a.v ? 2 : 1) * a.Hkv;  // staged rows per token
  if (a.Hq <= 0 || a.Hkv <= 0 || rows_per_tok > kMaxRows) return cudaErrorInvalidValue;
  if (a.d_r < 0 || a.d_r > kGatedD || (a.d_r & 15)) return cudaErrorInvalidValue;
  int tok = (40 * 1024) / (rows_per_tok * kRowBytes);
  tok = tok < 1 ? 1 : (tok > kMaxTok ? kMaxTok : tok);
  a.tok_per_cta = tok;
  const size_t smem = (size_t)tok * rows_per_tok * kRowBytes;
  static unsigned long long attr_mask = 0;  // per-device dynamic smem opt-in, per instantiation
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(attr_mask & (1ull << dev))) {
    e = cudaFuncSetAttribute(gated_prologue_kernel<Args>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxRows * kRowBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_mask |= 1ull << dev;
  }
  const long long grid = (n_tok + tok - 1) / tok;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  gated_prologue_kernel<Args><<<(unsigned)grid, kThreads, smem, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace

int gated_prologue_max_heads() { return kMaxRows; }

cudaError_t launch_gated_prologue(const GatedPrologueArgs& a, cudaStream_t stream) {
  return launch(a, stream);
}

cudaError_t launch_gated_prologue(const GatedPrologueChunkArgs& a, cudaStream_t stream) {
  if (a.base.B > kMaxBatch) return cudaErrorInvalidValue;
  return launch(a, stream);
}

}  // namespace q3a
