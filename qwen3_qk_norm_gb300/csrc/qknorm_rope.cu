// qknorm_rope.cu — K1, the fused QK-Norm + RoPE prologue.
//
// Per head row x (d = 128 bf16):
//   y = x * rsqrt(mean(x^2) + eps) * gamma          (fp32 accumulation)
//   y'_i      = y_i cos(p w_i) - y_{i+64} sin(p w_i)   i < 64
//   y'_{i+64} = y_{i+64} cos(p w_i) + y_i sin(p w_i),  w_i = theta^(-2i/128)
// rounded once to bf16. Norm before RoPE, as in "7.2 Qwen3 full-scale
// implementation" (§7.2.1 GroupedQueryAttention.forward: q_norm/k_norm, then
// apply_rope) and the transformers Qwen3Attention quoted on the "Qwen3" note.
//
// Layout of the work: one CTA per 8 tokens. The 8 x 64 rotation angles of its
// tokens are formed once per CTA in fp64 (p * w_i, reduced modulo 2 pi) and
// turned into fp32 (cos, sin) pairs in shared memory; every head row of those
// tokens (Q and K rows in the same launch) reuses them. A half-warp owns one
// row: lane L holds elements 4L..4L+3 and their rotate-half partners
// 64+4L..64+4L+3, so the rotation needs no data exchange and the RMS needs a
// 4-step shuffle reduction inside the half-warp. Loads and stores are 8-byte
// vectors, 128 contiguous bytes per half-warp per instruction. Row addresses
// come from per-token offsets computed once per CTA, so the row loop has no
// integer division.
#include "q3a_internal.h"
#include "q3a_rope.cuh"

namespace q3a {

namespace {

constexpr int kTokPerCta = 8;
constexpr int kThreads = 256;
constexpr int kHalfWarps = kThreads / 16;
constexpr int kUnroll = 2;  // rows in flight per half-warp

__global__ void __launch_bounds__(kThreads) qknorm_rope_kernel(RopeArgs a) {
  __shared__ __align__(16) float cos_s[kTokPerCta][64];
  __shared__ __align__(16) float sin_s[kTokPerCta][64];
  __shared__ long long xbase[kTokPerCta][2], ybase[kTokPerCta][2];  // in rows of 128
  const int tid = threadIdx.x;
  const long long n_tok = (long long)a.B * a.T;
  const long long tok0 = (long long)blockIdx.x * kTokPerCta;
  const int tok_here = (int)min((long long)kTokPerCta, n_tok - tok0);

  if (blockIdx.x == 0 && tid < 32) {
    if (a.err_clear && tid == 0) *a.err_clear = 0u;
    if (a.logit_bound && a.ntensors == 2) {
      // QK-Norm bounds every logit: |qhat| <= sqrt(128) max|gamma_q| and the
      // same for khat, so |qhat . khat| / sqrt(128) <= sqrt(128) gq gk
      float gq = 0.f, gk = 0.f;
      for (int i = tid; i < 128; i += 32) {
        gq = fmaxf(gq, fabsf(__uint_as_float((uint32_t)a.t[0].gamma[i] << 16)));
        gk = fmaxf(gk, fabsf(__uint_as_float((uint32_t)a.t[1].gamma[i] << 16)));
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        gq = fmaxf(gq, __shfl_xor_sync(0xffffffffu, gq, o));
        gk = fmaxf(gk, __shfl_xor_sync(0xffffffffu, gk, o));
      }
      if (tid == 0) *a.logit_bound = 11.313708498984761f * gq * gk * 1.4426950408889634f;
    }
  }

  // rotation table of this CTA's tokens (two entries per thread)
  for (int e = tid; e < kTokPerCta * 64; e += kThreads) {
    const int tt = e >> 6, i = e & 63;
    if (tt < tok_here) {
      const float2 c_s = rope_cos_sin(a.pos0 + (tok0 + tt) % a.T, a.inv_freq[i]);
      cos_s[tt][i] = c_s.x;
      sin_s[tt][i] = c_s.y;
    }
  }
  // per-token row offsets of both tensors: the only divisions of the kernel
  if (tid < kTokPerCta * 2) {
    const int tt = tid >> 1, s = tid & 1;
    if (tt < tok_here && s < a.ntensors) {
      const long long tok = tok0 + tt;
      const long long b = tok / a.T, t = tok - b * a.T;
      xbase[tt][s] = b * (s ? a.t[1].xsb : a.t[0].xsb) + t * (s ? a.t[1].xst : a.t[0].xst);
      ybase[tt][s] = b * (s ? a.t[1].ysb : a.t[0].ysb) + t * (s ? a.t[1].yst : a.t[0].yst);
    }
  }

  const int lane16 = tid & 15;
  const int hw = tid >> 4;
  // gamma slices of both tensors, reused for every row
  float gl[2][4], gh[2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const uint16_t* gp = s ? a.t[1].gamma : a.t[0].gamma;
    if (s < a.ntensors) {
      unpack4(reinterpret_cast<const uint2*>(gp)[lane16], gl[s]);
      unpack4(reinterpret_cast<const uint2*>(gp + 64)[lane16], gh[s]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) gl[s][j] = gh[s][j] = 0.f;
    }
  }
  __syncthreads();

  const int H0 = a.t[0].H;
  const int rows_per_tok = H0 + (a.ntensors > 1 ? a.t[1].H : 0);
  const int rows = tok_here * rows_per_tok;
  const int rows_even = (rows + 1) & ~1;  // whole warps, so the shuffles stay converged
  const uint16_t* x0 = a.t[0].x;
  const uint16_t* x1 = a.t[1].x;
  uint16_t* y0 = a.t[0].y;
  uint16_t* y1 = a.t[1].y;
  const long long xsh0 = a.t[0].xsh, xsh1 = a.t[1].xsh, ysh0 = a.t[0].ysh, ysh1 = a.t[1].ysh;

  // (tt, h) of row r = hw, advanced by kHalfWarps rows at a time without
  // division; kUnroll rows per half-warp are loaded before any is used
  int tt = 0, h = hw;
  while (h >= rows_per_tok) {
    h -= rows_per_tok;
    ++tt;
  }
  for (int r = hw; r < rows_even; r += kHalfWarps * kUnroll) {
    float xl[kUnroll][4], xh[kUnroll][4];
    uint16_t* yr[kUnroll];
    int tsel[kUnroll], ssel[kUnroll];
    bool live[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      live[u] = r + u * kHalfWarps < rows;
      const int ttl = live[u] ? tt : tok_here - 1;
      const int hl = live[u] ? h : rows_per_tok - 1;
      const int sl = hl < H0 ? 0 : 1;
      const int hs = sl ? hl - H0 : hl;
      const uint16_t* xr =
          (sl ? x1 : x0) + (xbase[ttl][sl] + (long long)hs * (sl ? xsh1 : xsh0)) * 128;
      yr[u] = (sl ? y1 : y0) + (ybase[ttl][sl] + (long long)hs * (sl ? ysh1 : ysh0)) * 128;
      tsel[u] = ttl;
      ssel[u] = sl;
      unpack4(reinterpret_cast<const uint2*>(xr)[lane16], xl[u]);
      unpack4(reinterpret_cast<const uint2*>(xr + 64)[lane16], xh[u]);
      h += kHalfWarps;
      while (h >= rows_per_tok) {
        h -= rows_per_tok;
        ++tt;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (r + u * kHalfWarps >= rows_even) break;  // same for both halves of a warp
      const float4 c4 = reinterpret_cast<const float4*>(cos_s[tsel[u]])[lane16];
      const float4 s4 = reinterpret_cast<const float4*>(sin_s[tsel[u]])[lane16];
      const float2 c_s[4] = {make_float2(c4.x, s4.x), make_float2(c4.y, s4.y),
                             make_float2(c4.z, s4.z), make_float2(c4.w, s4.w)};
      float gls[4], ghs[4], ol[4], oh[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        gls[j] = ssel[u] ? gl[1][j] : gl[0][j];
        ghs[j] = ssel[u] ? gh[1][j] : gh[0][j];
      }
      qknorm_rope_halfwarp(xl[u], xh[u], gls, ghs, c_s, a.eps, ol, oh);
      if (live[u]) {
        reinterpret_cast<uint2*>(yr[u])[lane16] = pack4(ol);
        reinterpret_cast<uint2*>(yr[u] + 64)[lane16] = pack4(oh);
      }
    }
  }
}

}  // namespace

void fill_inv_freq(double theta, double* inv_freq) {
  for (int i = 0; i < 64; ++i) inv_freq[i] = pow(theta, -(2.0 * i) / 128.0);
}

cudaError_t launch_qknorm_rope(const RopeArgs& a, cudaStream_t stream) {
  const long long n_tok = (long long)a.B * a.T;
  if (n_tok == 0) return cudaSuccess;
  const long long grid = (n_tok + kTokPerCta - 1) / kTokPerCta;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  qknorm_rope_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace q3a
