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
// Layout of the work: one CTA per 4 tokens. The 4 x 64 rotation angles of its
// tokens are formed once per CTA in fp64 (p * w_i, reduced modulo 2 pi) and
// turned into fp32 (cos, sin) pairs in shared memory; every head row of those
// tokens (Q and K rows in the same launch) reuses them. A half-warp owns one
// row: lane L holds elements 4L..4L+3 and their rotate-half partners
// 64+4L..64+4L+3, so the rotation needs no data exchange and the RMS needs a
// 4-step shuffle reduction inside the half-warp. Loads and stores are 8-byte
// vectors, 128 contiguous bytes per half-warp per instruction.
#include "q3a_internal.h"
#include "q3a_rope.cuh"

namespace q3a {

namespace {

constexpr int kTokPerCta = 4;  // 64 angle-table entries per token
constexpr int kThreads = 256;
constexpr int kHalfWarps = kThreads / 16;
constexpr int kUnroll = 4;  // rows per half-warp per pass

__global__ void __launch_bounds__(kThreads) qknorm_rope_kernel(RopeArgs a) {
  __shared__ float2 cs[kTokPerCta][64];
  const int tid = threadIdx.x;
  const long long n_tok = (long long)a.B * a.T;
  const long long tok0 = (long long)blockIdx.x * kTokPerCta;

  if (a.err_clear && blockIdx.x == 0 && tid == 0) *a.err_clear = 0u;

  {  // rotation table of this CTA's tokens
    const int tt = tid >> 6, i = tid & 63;
    const long long tok = tok0 + tt;
    if (tok < n_tok) cs[tt][i] = rope_cos_sin(a.pos0 + tok % a.T, a.inv_freq[i]);
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
  const long long tok_here = min((long long)kTokPerCta, n_tok - tok0);
  const int rows = (int)tok_here * rows_per_tok;
  // rows are taken by whole warps (two per warp) so the shuffles stay converged
  const int rows_even = (rows + 1) & ~1;

  // Each half-warp handles kUnroll rows per pass, all loads first, so that
  // kUnroll x 256 bytes per half-warp are in flight at once.
  for (int r0 = hw; r0 < rows_even; r0 += kHalfWarps * kUnroll) {
    float xl[kUnroll][4], xh[kUnroll][4];
    uint16_t* yr[kUnroll];
    int sel[kUnroll], tts[kUnroll];
    bool live[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int r = r0 + u * kHalfWarps;
      live[u] = r < rows;
      const int rr = live[u] ? r : rows - 1;
      const int tt = rr / rows_per_tok;
      int h = rr - tt * rows_per_tok;
      const int s = (h < H0) ? 0 : 1;
      if (s) h -= H0;
      const long long tok = tok0 + tt;
      const long long b = tok / a.T, t = tok - b * a.T;
      // field-wise selects keep the parameter struct out of local memory
      const uint16_t* xr =
          (s ? a.t[1].x : a.t[0].x) +
          (b * (s ? a.t[1].xsb : a.t[0].xsb) + t * (s ? a.t[1].xst : a.t[0].xst) +
           (long long)h * (s ? a.t[1].xsh : a.t[0].xsh)) * 128;
      yr[u] = (s ? a.t[1].y : a.t[0].y) +
              (b * (s ? a.t[1].ysb : a.t[0].ysb) + t * (s ? a.t[1].yst : a.t[0].yst) +
               (long long)h * (s ? a.t[1].ysh : a.t[0].ysh)) * 128;
      sel[u] = s;
      tts[u] = tt;
      unpack4(reinterpret_cast<const uint2*>(xr)[lane16], xl[u]);
      unpack4(reinterpret_cast<const uint2*>(xr + 64)[lane16], xh[u]);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (r0 + u * kHalfWarps >= rows_even) break;  // uniform across the warp
      float2 c_s[4];
      float gls[4], ghs[4], ol[4], oh[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        c_s[j] = cs[tts[u]][4 * lane16 + j];
        gls[j] = sel[u] ? gl[1][j] : gl[0][j];
        ghs[j] = sel[u] ? gh[1][j] : gh[0][j];
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
