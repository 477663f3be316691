// q3a_rope.cuh — device pieces of QK-Norm + rotate-half RoPE shared by the
// prologue kernels (K1, K5) and the decode kernel (K3).
//
//   y = x * rsqrt(mean(x^2) + eps) * gamma                       (fp32)
//   y'_i = y_i cos a_i - y_{i+64} sin a_i ; y'_{i+64} = y_{i+64} cos a_i + y_i sin a_i
//   a_i = p * theta^(-2i/128)
// ("7.2 Qwen3 full-scale implementation", §7.2.1 RMSNorm, compute_rope_params,
// apply_rope; norm first, then RoPE.)
#pragma once

#include "q3a_device.cuh"

namespace q3a {

// (cos a, sin a) for a = p * w with w = 2 pi * turn / 2^64. p * turn modulo
// 2^64 is the angle in turns, exactly (integer wrap-around); its top 32 bits,
// as a signed fraction x of half a turn, give a = pi * x with |x| < 1, and
// sincospif evaluates it without a range reduction. The error of the 64-bit
// frequency (below 2^-64 turn) times p stays under 2^-34 turn for p < 2^30.
__device__ __forceinline__ float2 rope_cos_sin(long long p, unsigned long long turn) {
  const unsigned long long f = (unsigned long long)p * turn;
  const float x = (float)(int)(f >> 32) * 4.656612873077393e-10f;  // 2^-31
  float s, c;
  sincospif(x, &s, &c);
  return make_float2(c, s);
}

// One head row held by a half-warp: lane L (0..15) holds x[4L..4L+3] in xl and
// their rotate-half partners x[64+4L..64+4L+3] in xh, with the matching gamma
// slices gl/gh and the (cos, sin) of angles 4L..4L+3 in cs[0..3]. All 32 lanes
// of the warp must call this together (two rows per warp).
__device__ __forceinline__ void qknorm_rope_halfwarp(const float (&xl)[4], const float (&xh)[4],
                                                     const float (&gl)[4], const float (&gh)[4],
                                                     const float2 (&cs)[4], float eps,
                                                     float (&ol)[4], float (&oh)[4]) {
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) ss = fmaf(xl[j], xl[j], fmaf(xh[j], xh[j], ss));
  ss += __shfl_xor_sync(0xffffffffu, ss, 8);
  ss += __shfl_xor_sync(0xffffffffu, ss, 4);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  const float inv_rms = rsqrtf(ss * (1.0f / 128.0f) + eps);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float yl = xl[j] * inv_rms * gl[j];
    const float yh = xh[j] * inv_rms * gh[j];
    ol[j] = yl * cs[j].x - yh * cs[j].y;
    oh[j] = yh * cs[j].x + yl * cs[j].y;
  }
}

// Sequence b and in-sequence index t of token first + tt of a [B, T] token
// range, given those of `first` (computed once per CTA): a CTA owns a few
// consecutive tokens, so counting forward replaces a 64-bit division per use.
__device__ __forceinline__ void token_bt(long long b_first, int t_first, int tt, int T,
                                         long long& b, int& t) {
  b = b_first;
  t = t_first + tt;
  while (t >= T) {
    t -= T;
    ++b;
  }
}

__device__ __forceinline__ void unpack4(uint2 v, float (&f)[4]) {
  f[0] = bf16_lo(v.x);
  f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y);
  f[3] = bf16_hi(v.y);
}

__device__ __forceinline__ uint2 pack4(const float (&f)[4]) {
  return make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
}

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
  f[0] = bf16_lo(v.x);
  f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y);
  f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z);
  f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w);
  f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

}  // namespace q3a
