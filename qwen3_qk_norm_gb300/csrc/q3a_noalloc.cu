// q3a_noalloc.cu — q3a_decode_noalloc: the decode step for callers that have
// no way to hand the library a device workspace.
//
// Some callers cannot allocate device memory at the point where they need a
// decode step: a host framework that owns every device allocation and gives
// plugins none, code that must not call cudaMalloc because it synchronises
// the device (a latency-critical serving loop), or code running where the
// allocator is unavailable. For them, the split partials and the error word
// that q3a_decode keeps in the caller's workspace live here instead, in one
// file-scope device array of fixed size that every GPU loading this library
// holds until the process exits.
//
// The kernels are the same as q3a_decode's (decode_attention.cu); only where
// their scratch lives differs.
#include <math.h>
#include <string.h>

#include <mutex>

#include "q3a.h"
#include "q3a_internal.h"

namespace q3a {
namespace {

constexpr size_t kScratchBytes = Q3A_DECODE_NOALLOC_SCRATCH_BYTES;
constexpr size_t kScratchHeader = 256;  // error word, then padding

// The scratch array. In host code this name is only a stand-in for the
// device symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, looked up once
// per device (with that device current).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// The error word of q3a_decode_noalloc on the current device (offset 0 of the
// scratch array), for q3a_last_device_error(NULL, stream).
cudaError_t noalloc_error_word(void** out) { return scratch_address(out); }

}  // namespace q3a

using namespace q3a;

extern "C" q3a_status q3a_decode_noalloc(const q3a_bf16* q, const q3a_bf16* k_new,
                                         const q3a_bf16* v_new, q3a_bf16* k_cache,
                                         q3a_bf16* v_cache, const int32_t* start_pos,
                                         const q3a_bf16* q_gamma, const q3a_bf16* k_gamma,
                                         q3a_bf16* out, int B, int Hq, int Hkv, int d, int S_max,
                                         double theta, float eps, void* stream) {
  // the argument rules of q3a_decode
  if (d != 128 || B < 0 || B > kDecodeMaxB || S_max <= 0 || S_max > (1 << 30)) return Q3A_EINVAL;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return Q3A_EINVAL;
  const int g = Hq / Hkv;
  if (!(g == 1 || g == 2 || g == 4 || g == 8 || g == 16)) return Q3A_EINVAL;
  if (!(isfinite(theta) && theta > 1.0 && isfinite(eps) && eps > 0.0f)) return Q3A_EINVAL;
  if (B == 0) return Q3A_OK;
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, q_gamma, k_gamma, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return Q3A_EINVAL;
  if (!start_pos) return Q3A_EINVAL;
  int max_splits = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t p = start_pos[b];
    if (p < 0 || (long long)p + 1 > S_max) return Q3A_ERANGE;  // nothing written yet
    const int n = (p + 1 + kDecodeChunk - 1) / kDecodeChunk;
    if (n > max_splits) max_splits = n;
  }
  // partials are laid out with the splits this call uses, not S_max's
  const size_t need = kScratchHeader + (size_t)B * Hkv * max_splits * g * kDecodePartialFloats *
                                           sizeof(float);
  if (need > kScratchBytes) return Q3A_EINVAL;

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return Q3A_ECUDA;

  DecodeArgs da;
  memset(&da, 0, sizeof da);
  const uint64_t dc[3] = {128, (uint64_t)S_max, (uint64_t)B * Hkv};
  const uint64_t sc[2] = {256, (uint64_t)S_max * 256};
  const uint32_t bc[3] = {64, 64, 1};
  if (encode_tensor_map(&da.tm_kc, k_cache, 3, dc, sc, bc) != CUDA_SUCCESS ||
      encode_tensor_map(&da.tm_vc, v_cache, 3, dc, sc, bc) != CUDA_SUCCESS)
    return Q3A_ECUDA;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  da.q = q;
  da.k_new = k_new;
  da.v_new = v_new;
  da.q_gamma = q_gamma;
  da.k_gamma = k_gamma;
  da.k_cache = k_cache;
  da.v_cache = v_cache;
  da.partial = reinterpret_cast<float*>(base + kScratchHeader);
  da.out = out;
  da.err = reinterpret_cast<uint32_t*>(base);
  da.B = B;
  da.Hq = Hq;
  da.Hkv = Hkv;
  da.g = g;
  da.S_max = S_max;
  da.split_stride = max_splits;
  da.max_splits = max_splits;
  da.eps = eps;
  fill_turn_freq(theta, 128, da.turn_freq);
  for (int b = 0; b < B; ++b) da.start_pos[b] = start_pos[b];

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the error word must start at zero; the partials are written before read
  cudaError_t e = cudaMemsetAsync(da.err, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = launch_decode(da, st);
  return e == cudaSuccess ? Q3A_OK : Q3A_ECUDA;
}
