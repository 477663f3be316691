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
// Layout of the work. The kernel is a pure stream (HBM-bound), so it is built
// around keeping many bytes in flight: a CTA owns a few consecutive tokens,
// and the head rows of those tokens are contiguous in the [tokens, H, 128]
// inputs, so one bulk copy per tensor (cp.async.bulk, completion on an
// mbarrier) brings them all into shared memory. While that copy is in flight
// the CTA forms the rotation angles of its tokens (p * w_i as an exact 64-bit
// fixed-point count of turns, then sincospif: rope_cos_sin in q3a_rope.cuh)
// and their fp32 cos/sin. A half-warp then owns one row:
// lane L holds elements 4L..4L+3 and their rotate-half partners 64+4L..,
// so the rotation needs no data exchange and the RMS needs a 4-step shuffle
// reduction. Results overwrite the staged rows, and bulk stores write them
// out: one store per tensor when the output has the input's layout, one per
// row otherwise (the head-major K layout of the prefill workspace).
#include <math.h>
#include <string.h>

#include <mutex>

#include "q3a_internal.h"
#include "q3a_rope.cuh"

namespace q3a {

namespace {

constexpr int kThreads = 256;
constexpr int kHalfWarps = kThreads / 16;
constexpr int kMaxTok = 32;

__global__ void __launch_bounds__(kThreads) qknorm_rope_kernel(const __grid_constant__ RopeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bar;
  const int tid = threadIdx.x;
  const int tok_per_cta = a.tok_per_cta;
  const long long n_tok = (long long)a.B * a.T;
  const long long tok0 = (long long)blockIdx.x * tok_per_cta;
  const int tok_here = (int)min((long long)tok_per_cta, n_tok - tok0);
  const int H0 = a.t[0].H, H1 = a.ntensors > 1 ? a.t[1].H : 0;
  const int H2 = a.ntensors > 2 ? a.t[2].H : 0;
  const uint32_t bytes0 = (uint32_t)tok_here * H0 * 256, bytes1 = (uint32_t)tok_here * H1 * 256;
  const uint32_t bytes2 = (uint32_t)tok_here * H2 * 256;
  uint16_t* rows0 = reinterpret_cast<uint16_t*>(smem);
  uint16_t* rows1 = reinterpret_cast<uint16_t*>(smem + (size_t)tok_per_cta * H0 * 256);
  uint16_t* rows2 = reinterpret_cast<uint16_t*>(smem + (size_t)tok_per_cta * (H0 + H1) * 256);
  // the CTA's tokens' cos and sin [tok][64] each, after the staged rows
  float* cos_s = reinterpret_cast<float*>(smem + (size_t)tok_per_cta * (H0 + H1 + H2) * 256);
  float* sin_s = cos_s + tok_per_cta * 64;
  // per normalised tensor and token: the output row (in rows of 128) of head 0
  long long* obase_s = reinterpret_cast<long long*>(sin_s + tok_per_cta * 64);

  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, bytes0 + bytes1 + bytes2);
    if (bytes0) bulk_load(rows0, a.t[0].x + tok0 * H0 * 128, bytes0, &bar);
    if (bytes1) bulk_load(rows1, a.t[1].x + tok0 * H1 * 128, bytes1, &bar);
    if (bytes2) bulk_load(rows2, a.t[2].x + tok0 * H2 * 128, bytes2, &bar);
  }
  if (blockIdx.x == 0 && tid >= 32 && tid < 64) {
    const int l = tid - 32;
    if (a.err_clear && l == 0) *a.err_clear = 0u;
    if (a.logit_bound) {
      // QK-Norm bounds every logit: |qhat| <= sqrt(128) max|gamma_q| and the
      // same for khat, so |qhat . khat| / sqrt(128) <= sqrt(128) gq gk
      float gq = 0.f, gk = 0.f;
      for (int i = l; i < 128; i += 32) {
        gq = fmaxf(gq, fabsf(__uint_as_float((uint32_t)a.bound_gamma[0][i] << 16)));
        gk = fmaxf(gk, fabsf(__uint_as_float((uint32_t)a.bound_gamma[1][i] << 16)));
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        gq = fmaxf(gq, __shfl_xor_sync(0xffffffffu, gq, o));
        gk = fmaxf(gk, __shfl_xor_sync(0xffffffffu, gk, o));
      }
      if (l == 0) *a.logit_bound = 11.313708498984761f * gq * gk * 1.4426950408889634f;
    }
  }
  // (b, t) of the CTA's first token; the others by counting
  const long long b_first = tok0 / a.T;
  const int t_first = (int)(tok0 - b_first * a.T);
  // rotation table of this CTA's tokens while the rows are in flight
  for (int e = tid; e < tok_here * 64; e += kThreads) {
    const int tt = e >> 6, i = e & 63;
    long long b;
    int t;
    token_bt(b_first, t_first, tt, a.T, b, t);
    const long long pos = (a.per_b_pos ? (long long)a.pos_b[b] : a.pos0) + t;
    const float2 c_s = rope_cos_sin(pos, a.turn_freq[i]);
    cos_s[tt * 64 + i] = c_s.x;
    sin_s[tt * 64 + i] = c_s.y;
    // the prefill's table of (cos, sin) per position, for the query tiles that
    // the attention kernel normalises itself: written by sequence 0's tokens
    if (a.rope_table && b == 0) reinterpret_cast<float2*>(a.rope_table)[t * 64 + i] = c_s;
  }
  for (int e = tid; e < 2 * tok_here; e += kThreads) {
    const int s = e >= tok_here ? 1 : 0, tt = e - s * tok_here;
    if (s >= a.ntensors) continue;
    const RopeTensor& ts = a.t[s];
    long long b;
    int t;
    token_bt(b_first, t_first, tt, a.T, b, t);
    obase_s[s * tok_per_cta + tt] =
        b * ts.ysb + (t + (ts.y_at_position ? (long long)a.pos_b[b] : 0)) * ts.yst;
  }
  const int lane16 = tid & 15;
  const int hw = tid >> 4;
  __syncthreads();  // barrier initialised, tables written
  mbar_wait(&bar, 0, nullptr, 0, nullptr);

  // Normalised rows whose output is not in the input's layout (head-major
  // Khat, cache rows) go straight from registers to global memory: a half-warp
  // writes one 256-byte row, instead of a bulk store per row afterwards.
  auto contiguous_out = [&](int s, int H) {
    const RopeTensor& ts = a.t[s];
    return !ts.y_at_position && ts.ysh == 1 && ts.yst == H && ts.ysb == (long long)a.T * H;
  };
#pragma unroll 1
  for (int s = 0; s < 2; ++s) {
    if (s >= a.ntensors || a.t[s].copy_only) break;  // tensors that normalise come first
    const RopeTensor& ts = a.t[s];
    const int H = s ? H1 : H0;
    const int R = tok_here * H;
    uint16_t* base = s ? rows1 : rows0;
    const bool direct = !contiguous_out(s, H);
    // this lane's gamma (elements 4L..4L+3 and 64+4L..) as packed fp32 pairs
    uint64_t GL[2], GH[2];
    {
      const uint2 gl = reinterpret_cast<const uint2*>(ts.gamma)[lane16];
      const uint2 gh = reinterpret_cast<const uint2*>(ts.gamma + 64)[lane16];
      GL[0] = f2_pack(bf16_lo(gl.x), bf16_hi(gl.x));
      GL[1] = f2_pack(bf16_lo(gl.y), bf16_hi(gl.y));
      GH[0] = f2_pack(bf16_lo(gh.x), bf16_hi(gh.x));
      GH[1] = f2_pack(bf16_lo(gh.y), bf16_hi(gh.y));
    }
    // token of row r: floor(r / H) = umulhi(r, ceil(2^32 / H)), exact for r * H < 2^32
    // (H = 1, whose multiplier does not fit 32 bits, is r itself)
    const uint32_t magic = H > 1 ? 0xFFFFFFFFu / (uint32_t)H + 1u : 0u;
    const int R_even = (R + 1) & ~1;  // whole warps, so the shuffles stay converged
#pragma unroll 1
    for (int q = hw; q < R_even; q += kHalfWarps) {
      const bool live = q < R;
      const int rr = live ? q : R - 1;
      const int tt = H > 1 ? (int)__umulhi((uint32_t)rr, magic) : rr;
      uint16_t* row = base + (size_t)rr * 128;
      const uint2 wl = reinterpret_cast<const uint2*>(row)[lane16];
      const uint2 wh = reinterpret_cast<const uint2*>(row + 64)[lane16];
      const uint64_t XL0 = f2_pack(bf16_lo(wl.x), bf16_hi(wl.x));
      const uint64_t XL1 = f2_pack(bf16_lo(wl.y), bf16_hi(wl.y));
      const uint64_t XH0 = f2_pack(bf16_lo(wh.x), bf16_hi(wh.x));
      const uint64_t XH1 = f2_pack(bf16_lo(wh.y), bf16_hi(wh.y));
      uint64_t ss2 = f2_mul(XL0, XL0);
      ss2 = f2_fma(XL1, XL1, ss2);
      ss2 = f2_fma(XH0, XH0, ss2);
      ss2 = f2_fma(XH1, XH1, ss2);
      float s0, s1;
      f2_unpack(ss2, s0, s1);
      float ss = s0 + s1;
      ss += __shfl_xor_sync(0xffffffffu, ss, 8);
      ss += __shfl_xor_sync(0xffffffffu, ss, 4);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      const float inv_rms = rsqrtf(ss * (1.0f / 128.0f) + a.eps);
      const uint64_t INV2 = f2_pack(inv_rms, inv_rms);
      const float4 c4 = reinterpret_cast<const float4*>(cos_s + tt * 64)[lane16];
      const float4 s4 = reinterpret_cast<const float4*>(sin_s + tt * 64)[lane16];
      const uint64_t C2[2] = {f2_pack(c4.x, c4.y), f2_pack(c4.z, c4.w)};
      const uint64_t S2[2] = {f2_pack(s4.x, s4.y), f2_pack(s4.z, s4.w)};
      const uint64_t XL[2] = {XL0, XL1}, XH[2] = {XH0, XH1};
      uint32_t ol[2], oh[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        // y = x * gamma / rms; y'_i = y_i c - y_{i+64} s; y'_{i+64} = y_{i+64} c + y_i s
        const uint64_t A = f2_mul(f2_mul(XL[j], GL[j]), INV2);
        const uint64_t Bv = f2_mul(f2_mul(XH[j], GH[j]), INV2);
        const uint64_t OL = f2_sub(f2_mul(A, C2[j]), f2_mul(Bv, S2[j]));
        const uint64_t OH = f2_fma(A, S2[j], f2_mul(Bv, C2[j]));
        float o0, o1;
        f2_unpack(OL, o0, o1);
        ol[j] = pack_bf16x2(o0, o1);
        f2_unpack(OH, o0, o1);
        oh[j] = pack_bf16x2(o0, o1);
      }
      if (live) {
        uint16_t* dst = row;
        if (direct) {
          const int h = rr - tt * H;
          dst = ts.y + (obase_s[s * tok_per_cta + tt] + (long long)h * ts.ysh) * 128;
        }
        reinterpret_cast<uint2*>(dst)[lane16] = make_uint2(ol[0], ol[1]);
        reinterpret_cast<uint2*>(dst + 64)[lane16] = make_uint2(oh[0], oh[1]);
      }
    }
  }
  fence_proxy_async_smem();  // the bulk stores below read what was just written
  __syncthreads();

  // bulk stores: a tensor whose output has the input's layout goes out as one
  // block; otherwise one 256-byte row per store, spread over the threads
  bool issued = false;
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    if (s >= a.ntensors) break;
    const int H = s == 2 ? H2 : (s ? H1 : H0);
    const uint16_t* src = s == 2 ? rows2 : (s ? rows1 : rows0);
    const RopeTensor& ts = a.t[s];  // s is a compile-time index after unrolling
    uint16_t* y = ts.y;
    const long long ysb = ts.ysb, yst = ts.yst, ysh = ts.ysh;
    const int at_pos = ts.y_at_position;
    const bool contiguous = !at_pos && ysh == 1 && yst == H && ysb == (long long)a.T * H;
    if (!ts.copy_only && !contiguous) continue;  // written from registers above
    if (contiguous) {
      const uint32_t bytes = s == 2 ? bytes2 : (s ? bytes1 : bytes0);
      if (tid == 0 && bytes) {
        bulk_store(y + tok0 * H * 128, src, bytes);
        issued = true;
      }
    } else {
      for (int rr = tid; rr < tok_here * H; rr += kThreads) {
        const int tt = rr / H, h = rr - tt * H;
        long long b;
        int t_in;
        token_bt(b_first, t_first, tt, a.T, b, t_in);
        const long long t = t_in + (at_pos ? (long long)a.pos_b[b] : 0);
        bulk_store(y + (b * ysb + t * yst + (long long)h * ysh) * 128, src + (size_t)rr * 128, 256);
        issued = true;
      }
    }
  }
  if (issued) bulk_commit_and_wait_read();  // shared memory stays valid until read
}

}  // namespace

void fill_turn_freq(double theta, int d_rot, unsigned long long* turn_freq) {
  // w_i / (2 pi) in long double (64 or more mantissa bits), scaled to 2^64.
  // long double arithmetic can be slow (software quad precision on some
  // hosts), so the last few (theta, d_rot) pairs are remembered.
  struct Entry {
    double theta;
    int d_rot;
    unsigned long long f[128];
  };
  static Entry cache[4];
  static int n_cached = 0, next = 0;
  static std::mutex mu;
  const int n = d_rot / 2;
  std::lock_guard<std::mutex> lock(mu);
  for (int c = 0; c < n_cached; ++c)
    if (cache[c].theta == theta && cache[c].d_rot == d_rot) {
      memcpy(turn_freq, cache[c].f, sizeof(unsigned long long) * n);
      return;
    }
  const long double two_pi = 6.283185307179586476925286766559L;
  Entry& e = cache[next];
  e.theta = theta;
  e.d_rot = d_rot;
  for (int i = 0; i < n; ++i) {
    const long double w = powl((long double)theta, -(long double)(2 * i) / (long double)d_rot);
    e.f[i] = (unsigned long long)llroundl(w / two_pi * 18446744073709551616.0L);
  }
  memcpy(turn_freq, e.f, sizeof(unsigned long long) * n);
  next = (next + 1) % 4;
  if (n_cached < 4) ++n_cached;
}

int qknorm_rope_max_heads() { return 512; }

cudaError_t launch_qknorm_rope(const RopeArgs& a_in, cudaStream_t stream) {
  const long long n_tok = (long long)a_in.B * a_in.T;
  if (n_tok == 0) return cudaSuccess;
  RopeArgs a = a_in;
  const int rows_per_tok =
      a.t[0].H + (a.ntensors > 1 ? a.t[1].H : 0) + (a.ntensors > 2 ? a.t[2].H : 0);
  if (rows_per_tok <= 0 || rows_per_tok > qknorm_rope_max_heads()) return cudaErrorInvalidValue;
  if (a.ntensors < 1 || a.ntensors > 3 || (a.ntensors == 3 && !a.t[2].copy_only))
    return cudaErrorInvalidValue;  // only the first two tensors normalise
  if (a.per_b_pos && a.B > kMaxBatch) return cudaErrorInvalidValue;
  // 32-40 KB of staged rows per CTA: several CTAs per SM keep ~150+ KB of
  // loads in flight
  int tok = (40 * 1024) / (rows_per_tok * 256);
  tok = tok < 1 ? 1 : (tok > kMaxTok ? kMaxTok : tok);
  a.tok_per_cta = tok;
  const size_t smem = (size_t)tok * rows_per_tok * 256 + (size_t)tok * 64 * 2 * 4 + (size_t)tok * 2 * 8;
  static unsigned long long attr_mask = 0;  // per-device dynamic smem opt-in
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(attr_mask & (1ull << dev))) {
    e = cudaFuncSetAttribute(qknorm_rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             512 * 256 + kMaxTok * (64 * 2 * 4 + 2 * 8));
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_mask |= 1ull << dev;
  }
  const long long grid = (n_tok + tok - 1) / tok;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  qknorm_rope_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace q3a
