// q3a_api.cu — the C ABI of include/q3a.h: argument validation (always before
// anything is launched or written), workspace layout, TMA tensor maps, and the
// kernel launches. The library allocates nothing and keeps no per-call state.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "q3a.h"
#include "q3a_internal.h"

namespace q3a {
namespace {

constexpr size_t kHeader = 256;  // error word and padding at the start of a workspace

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Gated layer: any whole ratio up to 16 (the decode kernel's MMA rows hold 16
// heads; the attention tile holds g heads for floor(128/g) tokens)
bool gated_group_ok(int Hq, int Hkv) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return false;
  return Hq / Hkv <= 16;
}

bool group_ok(int Hq, int Hkv) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return false;
  const int g = Hq / Hkv;
  return g == 1 || g == 2 || g == 4 || g == 8 || g == 16;
}

bool scalars_ok(double theta, float eps) {
  return isfinite(theta) && theta > 1.0 && isfinite(eps) && eps > 0.0f;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

q3a_status from_cuda(cudaError_t e) { return e == cudaSuccess ? Q3A_OK : Q3A_ECUDA; }

size_t prefill_q_bytes(int B, int T, int Hq) { return (size_t)B * T * Hq * 128 * 2; }
size_t prefill_k_bytes(int B, int T, int Hkv) { return (size_t)B * T * Hkv * 128 * 2; }

int decode_split_stride(int S_max, int d = 128) {
  return (S_max + decode_chunk_keys(d) - 1) / decode_chunk_keys(d);
}

}  // namespace

CUresult encode_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t d[5], s[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d,
            s, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace q3a

using namespace q3a;

extern "C" {

const char* q3a_status_string(q3a_status s) {
  switch (s) {
    case Q3A_OK: return "ok";
    case Q3A_EINVAL: return "invalid argument";
    case Q3A_ERANGE: return "start_pos out of range (context overflow)";
    case Q3A_ECUDA: return "CUDA error";
    case Q3A_ETIMEOUT: return "device-side wait timed out";
    case Q3A_ENOTIMPL: return "not implemented";
  }
  return "unknown status";
}

q3a_status q3a_qknorm_rope(const q3a_bf16* x, const q3a_bf16* gamma, q3a_bf16* y, int B, int T,
                           int H, int d, int pos0, double theta, float eps, void* stream) {
  if (d != 128 || B < 0 || T < 0 || H < 0 || pos0 < 0) return Q3A_EINVAL;
  if (H > qknorm_rope_max_heads()) return Q3A_EINVAL;
  if ((long long)pos0 + (long long)T - 1 > (1LL << 30)) return Q3A_EINVAL;
  if (!scalars_ok(theta, eps)) return Q3A_EINVAL;
  if (B == 0 || T == 0 || H == 0) return Q3A_OK;
  if (!x || !gamma || !y || !aligned16(x) || !aligned16(gamma) || !aligned16(y))
    return Q3A_EINVAL;
  RopeArgs a;
  memset(&a, 0, sizeof a);
  a.t[0] = RopeTensor{x, gamma, y, H, (long long)T * H, H, 1, (long long)T * H, H, 1};
  a.ntensors = 1;
  a.B = B;
  a.T = T;
  a.pos0 = pos0;
  a.eps = eps;
  fill_turn_freq(theta, 128, a.turn_freq);
  return from_cuda(launch_qknorm_rope(a, static_cast<cudaStream_t>(stream)));
}

// prefill workspace: header, Khat, then the RoPE table [T][64] (cos, sin)
size_t q3a_prefill_workspace_size(int B, int T, int Hq, int Hkv, int d) {
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || d != 128) return 0;
  return kHeader + align256(prefill_k_bytes(B, T, Hkv)) + align256((size_t)T * 64 * 8);
}

static q3a_status prefill_check(const void* const* ptrs, int nptrs, int B, int T, int Hq,
                                int Hkv, int d, void* workspace, size_t ws_bytes, bool* empty) {
  *empty = false;
  if (d != 128 || B < 0 || T < 0 || !group_ok(Hq, Hkv)) return Q3A_EINVAL;
  if ((long long)B * T * Hq > 0x7fffffffLL || T > (1 << 30)) return Q3A_EINVAL;
  if (Hq + Hkv > qknorm_rope_max_heads()) return Q3A_EINVAL;
  if (B == 0 || T == 0) {
    *empty = true;
    return Q3A_OK;
  }
  for (int i = 0; i < nptrs; ++i)
    if (!ptrs[i] || !aligned16(ptrs[i])) return Q3A_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return Q3A_EINVAL;
  if (ws_bytes < q3a_prefill_workspace_size(B, T, Hq, Hkv, d)) return Q3A_EINVAL;
  return Q3A_OK;
}

// chunk workspace: header, then Qhat; prefill workspace: header, Khat, RoPE table
static uint16_t* ws_qhat(void* ws) { return reinterpret_cast<uint16_t*>((uint8_t*)ws + kHeader); }
static uint16_t* ws_khat(void* ws) { return reinterpret_cast<uint16_t*>((uint8_t*)ws + kHeader); }
static float* ws_rope_table(void* ws, int B, int T, int Hkv) {
  return reinterpret_cast<float*>((uint8_t*)ws + kHeader + align256(prefill_k_bytes(B, T, Hkv)));
}

// Prefill prologue: K -> Khat (QK-Norm + RoPE at positions 0..T-1) in the
// head-major layout [B, Hkv, T] (a 128-key tile of one group is contiguous),
// plus the logit bound and the cleared error word. The query tiles are
// normalised and rotated by the attention kernel itself.
static void prologue_args(RopeArgs& ra, const q3a_bf16* k, const q3a_bf16* q_gamma,
                          const q3a_bf16* k_gamma, int B, int T, int Hkv, double theta, float eps,
                          void* workspace) {
  memset(&ra, 0, sizeof ra);
  ra.t[0] = RopeTensor{k, k_gamma, ws_khat(workspace), Hkv, (long long)T * Hkv, Hkv, 1,
                       (long long)Hkv * T, 1, T};
  ra.ntensors = 1;
  ra.B = B;
  ra.T = T;
  ra.pos0 = 0;
  ra.eps = eps;
  ra.err_clear = reinterpret_cast<uint32_t*>(workspace);
  ra.logit_bound = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 8);
  ra.bound_gamma[0] = q_gamma;
  ra.bound_gamma[1] = k_gamma;
  ra.rope_table = ws_rope_table(workspace, B, T, Hkv);
  fill_turn_freq(theta, 128, ra.turn_freq);
}

static q3a_status attention_args(PrefillArgs& pa, const q3a_bf16* q, const q3a_bf16* v,
                                 const q3a_bf16* q_gamma, q3a_bf16* out, int B, int T, int Hq,
                                 int Hkv, float eps, void* workspace) {
  memset(&pa, 0, sizeof pa);
  const int g = Hq / Hkv;
  const uint64_t dq[4] = {128, (uint64_t)Hq, (uint64_t)T, (uint64_t)B};
  const uint64_t sq[3] = {256, (uint64_t)Hq * 256, (uint64_t)T * Hq * 256};
  const uint32_t bq[4] = {64, (uint32_t)g, (uint32_t)(128 / g), 1};
  const uint64_t dk[3] = {128, (uint64_t)T, (uint64_t)B * Hkv};
  const uint64_t sk[2] = {256, (uint64_t)T * 256};
  const uint32_t bk[3] = {64, 128, 1};
  const uint64_t dv[4] = {128, (uint64_t)Hkv, (uint64_t)T, (uint64_t)B};
  const uint64_t sv[3] = {256, (uint64_t)Hkv * 256, (uint64_t)T * Hkv * 256};
  const uint32_t bv[4] = {64, 1, 128, 1};
  if (encode_tensor_map(&pa.tm_q, q, 4, dq, sq, bq) != CUDA_SUCCESS ||
      encode_tensor_map(&pa.tm_k, ws_khat(workspace), 3, dk, sk, bk) != CUDA_SUCCESS ||
      encode_tensor_map(&pa.tm_v, v, 4, dv, sv, bv) != CUDA_SUCCESS)
    return Q3A_ECUDA;
  pa.q_gamma = q_gamma;
  pa.eps = eps;
  pa.rope_table = ws_rope_table(workspace, B, T, Hkv);
  pa.out = out;
  pa.err = reinterpret_cast<uint32_t*>(workspace);
  pa.logit_bound = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + 8);
  pa.B = B;
  pa.T = T;
  pa.Hq = Hq;
  pa.Hkv = Hkv;
  pa.g = g;
  const int rows_tok = prefill_tokens_per_cta(g);
  pa.n_mtiles = (T + rows_tok - 1) / rows_tok;
  return Q3A_OK;
}

q3a_status q3a_prefill_prologue(const q3a_bf16* k, const q3a_bf16* q_gamma,
                                const q3a_bf16* k_gamma, int B, int T, int Hq, int Hkv, int d,
                                double theta, float eps, void* workspace, size_t ws_bytes,
                                void* stream) {
  if (!scalars_ok(theta, eps)) return Q3A_EINVAL;
  const void* ptrs[] = {k, q_gamma, k_gamma};
  bool empty;
  q3a_status s = prefill_check(ptrs, 3, B, T, Hq, Hkv, d, workspace, ws_bytes, &empty);
  if (s != Q3A_OK || empty) return s;
  RopeArgs ra;
  prologue_args(ra, k, q_gamma, k_gamma, B, T, Hkv, theta, eps, workspace);
  return from_cuda(launch_qknorm_rope(ra, static_cast<cudaStream_t>(stream)));
}

q3a_status q3a_prefill_attention(const q3a_bf16* q, const q3a_bf16* v, const q3a_bf16* q_gamma,
                                 q3a_bf16* out, int B, int T, int Hq, int Hkv, int d, float eps,
                                 void* workspace, size_t ws_bytes, void* stream) {
  if (!scalars_ok(2.0, eps)) return Q3A_EINVAL;
  const void* ptrs[] = {q, v, q_gamma, out};
  bool empty;
  q3a_status s = prefill_check(ptrs, 4, B, T, Hq, Hkv, d, workspace, ws_bytes, &empty);
  if (s != Q3A_OK || empty) return s;
  PrefillArgs pa;
  s = attention_args(pa, q, v, q_gamma, out, B, T, Hq, Hkv, eps, workspace);
  if (s != Q3A_OK) return s;
  return from_cuda(launch_prefill_attention(pa, static_cast<cudaStream_t>(stream)));
}

q3a_status q3a_prefill(const q3a_bf16* q, const q3a_bf16* k, const q3a_bf16* v,
                       const q3a_bf16* q_gamma, const q3a_bf16* k_gamma, q3a_bf16* out, int B,
                       int T, int Hq, int Hkv, int d, double theta, float eps, void* workspace,
                       size_t ws_bytes, void* stream) {
  if (!scalars_ok(theta, eps)) return Q3A_EINVAL;
  const void* ptrs[] = {q, k, v, q_gamma, k_gamma, out};
  bool empty;
  q3a_status s = prefill_check(ptrs, 6, B, T, Hq, Hkv, d, workspace, ws_bytes, &empty);
  if (s != Q3A_OK || empty) return s;
  // tensor maps first: a failure there launches nothing
  PrefillArgs pa;
  s = attention_args(pa, q, v, q_gamma, out, B, T, Hq, Hkv, eps, workspace);
  if (s != Q3A_OK) return s;
  RopeArgs ra;
  prologue_args(ra, k, q_gamma, k_gamma, B, T, Hkv, theta, eps, workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_qknorm_rope(ra, st);
  if (e == cudaSuccess) e = launch_prefill_attention(pa, st);
  return from_cuda(e);
}

size_t q3a_prefill_chunk_workspace_size(int B, int Tq, int Hq, int Hkv, int d) {
  if (B < 0 || Tq < 0 || Hq <= 0 || Hkv <= 0 || d != 128) return 0;
  return kHeader + align256(prefill_q_bytes(B, Tq, Hq));
}

q3a_status q3a_prefill_chunk(const q3a_bf16* q, const q3a_bf16* k, const q3a_bf16* v,
                             q3a_bf16* k_cache, q3a_bf16* v_cache, const int32_t* start_pos,
                             const q3a_bf16* q_gamma, const q3a_bf16* k_gamma, q3a_bf16* out,
                             int B, int Tq, int Hq, int Hkv, int d, int S_max, double theta,
                             float eps, void* workspace, size_t ws_bytes, void* stream) {
  if (d != 128 || B < 0 || Tq < 0 || B > kMaxBatch || !group_ok(Hq, Hkv)) return Q3A_EINVAL;
  if (S_max <= 0 || S_max > (1 << 30)) return Q3A_EINVAL;
  if (!scalars_ok(theta, eps)) return Q3A_EINVAL;
  if ((long long)B * Tq * Hq > 0x7fffffffLL) return Q3A_EINVAL;
  if (Hq + 2 * Hkv > qknorm_rope_max_heads()) return Q3A_EINVAL;
  if (B == 0 || Tq == 0) return Q3A_OK;
  const void* ptrs[] = {q, k, v, k_cache, v_cache, q_gamma, k_gamma, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return Q3A_EINVAL;
  if (!start_pos) return Q3A_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return Q3A_EINVAL;
  if (ws_bytes < q3a_prefill_chunk_workspace_size(B, Tq, Hq, Hkv, d)) return Q3A_EINVAL;
  for (int b = 0; b < B; ++b) {
    const int32_t p = start_pos[b];
    if (p < 0 || (long long)p + Tq > S_max) return Q3A_ERANGE;  // nothing written yet
  }
  const int g = Hq / Hkv;
  uint16_t* qhat = ws_qhat(workspace);

  // tensor maps first: a failure there launches nothing
  PrefillChunkArgs ca;
  memset(&ca, 0, sizeof ca);
  PrefillArgs& pa = ca.base;
  {
    const uint64_t dq[4] = {128, (uint64_t)Hq, (uint64_t)Tq, (uint64_t)B};
    const uint64_t sq[3] = {256, (uint64_t)Hq * 256, (uint64_t)Tq * Hq * 256};
    const uint32_t bq[4] = {64, (uint32_t)g, (uint32_t)(128 / g), 1};
    const uint64_t dc[3] = {128, (uint64_t)S_max, (uint64_t)B * Hkv};
    const uint64_t sc[2] = {256, (uint64_t)S_max * 256};
    const uint32_t bc[3] = {64, 128, 1};
    if (encode_tensor_map(&pa.tm_q, qhat, 4, dq, sq, bq) != CUDA_SUCCESS ||
        encode_tensor_map(&pa.tm_k, k_cache, 3, dc, sc, bc) != CUDA_SUCCESS ||
        encode_tensor_map(&pa.tm_v, v_cache, 3, dc, sc, bc) != CUDA_SUCCESS)
      return Q3A_ECUDA;
  }
  pa.out = out;
  pa.err = reinterpret_cast<uint32_t*>(workspace);
  pa.logit_bound = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + 8);
  pa.B = B;
  pa.T = Tq;
  pa.Hq = Hq;
  pa.Hkv = Hkv;
  pa.g = g;
  const int rows_tok = prefill_tokens_per_cta(g);
  pa.n_mtiles = (Tq + rows_tok - 1) / rows_tok;
  // cached keys were normalised with the same k_gamma by earlier calls (the
  // documented precondition), so the logit bound holds for them too; a cache
  // that breaks it badly enough to overflow a softmax sum is reported
  // (kErrWordBound)
  ca.fixed_shift_ok = 1;
  for (int b = 0; b < B; ++b) ca.pos_b[b] = start_pos[b];

  RopeArgs ra;
  memset(&ra, 0, sizeof ra);
  const long long S = S_max;
  // Q -> Qhat [B, Tq, Hq]; K -> k_cache rows start_pos[b] + t (normalised,
  // rotated); V -> v_cache rows start_pos[b] + t (copied)
  ra.t[0] = RopeTensor{q, q_gamma, qhat, Hq, (long long)Tq * Hq, Hq, 1, (long long)Tq * Hq, Hq, 1,
                       0, 0};
  ra.t[1] = RopeTensor{k, k_gamma, k_cache, Hkv, (long long)Tq * Hkv, Hkv, 1,
                       (long long)Hkv * S, 1, S, 0, 1};
  ra.t[2] = RopeTensor{v, nullptr, v_cache, Hkv, (long long)Tq * Hkv, Hkv, 1,
                       (long long)Hkv * S, 1, S, 1, 1};
  ra.ntensors = 3;
  ra.B = B;
  ra.T = Tq;
  ra.per_b_pos = 1;
  for (int b = 0; b < B; ++b) ra.pos_b[b] = start_pos[b];
  ra.eps = eps;
  ra.err_clear = reinterpret_cast<uint32_t*>(workspace);
  ra.logit_bound = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 8);
  ra.bound_gamma[0] = q_gamma;
  ra.bound_gamma[1] = k_gamma;
  fill_turn_freq(theta, 128, ra.turn_freq);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_qknorm_rope(ra, st);
  if (e == cudaSuccess) e = launch_prefill_attention(ca, st);
  return from_cuda(e);
}

size_t q3a_decode_workspace_size(int B, int Hq, int Hkv, int d, int S_max) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || d != 128 || S_max <= 0 || Hq % Hkv) return 0;
  const size_t parts = (size_t)B * Hkv * decode_split_stride(S_max) * (Hq / Hkv) *
                       kDecodePartialFloats * sizeof(float);
  return kHeader + align256(parts);
}

q3a_status q3a_decode(const q3a_bf16* q, const q3a_bf16* k_new, const q3a_bf16* v_new,
                      q3a_bf16* k_cache, q3a_bf16* v_cache, const int32_t* start_pos,
                      const q3a_bf16* q_gamma, const q3a_bf16* k_gamma, q3a_bf16* out, int B,
                      int Hq, int Hkv, int d, int S_max, double theta, float eps,
                      void* workspace, size_t ws_bytes, void* stream) {
  if (d != 128 || B < 0 || B > kDecodeMaxB || S_max <= 0 || !group_ok(Hq, Hkv))
    return Q3A_EINVAL;
  if (S_max > (1 << 30)) return Q3A_EINVAL;
  if (!scalars_ok(theta, eps)) return Q3A_EINVAL;
  if (B == 0) return Q3A_OK;
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, q_gamma, k_gamma, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return Q3A_EINVAL;
  if (!start_pos) return Q3A_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return Q3A_EINVAL;
  if (ws_bytes < q3a_decode_workspace_size(B, Hq, Hkv, d, S_max)) return Q3A_EINVAL;
  int max_splits = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t p = start_pos[b];
    if (p < 0 || (long long)p + 1 > S_max) return Q3A_ERANGE;  // nothing written yet
    const int n = (p + 1 + kDecodeChunk - 1) / kDecodeChunk;
    if (n > max_splits) max_splits = n;
  }

  static_assert(sizeof(DecodeArgs) < 32000, "kernel parameter limit");
  DecodeArgs dargs;  // kernel parameters, staged on the host stack
  DecodeArgs* da = &dargs;
  memset(da, 0, sizeof *da);
  const uint64_t dc[3] = {128, (uint64_t)S_max, (uint64_t)B * Hkv};
  const uint64_t sc[2] = {256, (uint64_t)S_max * 256};
  const uint32_t bc[3] = {64, 64, 1};
  if (encode_tensor_map(&da->tm_kc, k_cache, 3, dc, sc, bc) != CUDA_SUCCESS ||
      encode_tensor_map(&da->tm_vc, v_cache, 3, dc, sc, bc) != CUDA_SUCCESS)
    return Q3A_ECUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  da->q = q;
  da->k_new = k_new;
  da->v_new = v_new;
  da->q_gamma = q_gamma;
  da->k_gamma = k_gamma;
  da->k_cache = k_cache;
  da->v_cache = v_cache;
  da->partial = reinterpret_cast<float*>(ws + kHeader);
  da->out = out;
  da->err = reinterpret_cast<uint32_t*>(ws);
  da->B = B;
  da->Hq = Hq;
  da->Hkv = Hkv;
  da->g = Hq / Hkv;
  da->S_max = S_max;
  da->split_stride = decode_split_stride(S_max);
  da->max_splits = max_splits;
  da->eps = eps;
  fill_turn_freq(theta, 128, da->turn_freq);
  for (int b = 0; b < B; ++b) da->start_pos[b] = start_pos[b];

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(da->err, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = launch_decode(*da, st);
  return from_cuda(e);
}

q3a_status q3a_decode_device_pos(const q3a_bf16* q, const q3a_bf16* k_new,
                                 const q3a_bf16* v_new, q3a_bf16* k_cache, q3a_bf16* v_cache,
                                 const int32_t* start_pos, const q3a_bf16* q_gamma,
                                 const q3a_bf16* k_gamma, q3a_bf16* out, int B, int Hq, int Hkv,
                                 int d, int S_max, double theta, float eps, void* workspace,
                                 size_t ws_bytes, void* stream) {
  if (d != 128 || B < 0 || B > kDecodeMaxB || S_max <= 0 || !group_ok(Hq, Hkv))
    return Q3A_EINVAL;
  if (S_max > (1 << 30)) return Q3A_EINVAL;
  if (!scalars_ok(theta, eps)) return Q3A_EINVAL;
  if (B == 0) return Q3A_OK;
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, q_gamma, k_gamma, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return Q3A_EINVAL;
  if (!start_pos || (reinterpret_cast<uintptr_t>(start_pos) & 3u)) return Q3A_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return Q3A_EINVAL;
  if (ws_bytes < q3a_decode_workspace_size(B, Hq, Hkv, d, S_max)) return Q3A_EINVAL;

  DecodeArgs dargs;  // kernel parameters, staged on the host stack
  DecodeArgs* da = &dargs;
  memset(da, 0, sizeof *da);
  const uint64_t dc[3] = {128, (uint64_t)S_max, (uint64_t)B * Hkv};
  const uint64_t sc[2] = {256, (uint64_t)S_max * 256};
  const uint32_t bc[3] = {64, 64, 1};
  if (encode_tensor_map(&da->tm_kc, k_cache, 3, dc, sc, bc) != CUDA_SUCCESS ||
      encode_tensor_map(&da->tm_vc, v_cache, 3, dc, sc, bc) != CUDA_SUCCESS)
    return Q3A_ECUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  da->q = q;
  da->k_new = k_new;
  da->v_new = v_new;
  da->q_gamma = q_gamma;
  da->k_gamma = k_gamma;
  da->k_cache = k_cache;
  da->v_cache = v_cache;
  da->partial = reinterpret_cast<float*>(ws + kHeader);
  da->out = out;
  da->err = reinterpret_cast<uint32_t*>(ws);
  da->B = B;
  da->Hq = Hq;
  da->Hkv = Hkv;
  da->g = Hq / Hkv;
  da->S_max = S_max;
  da->split_stride = decode_split_stride(S_max);
  da->max_splits = da->split_stride;  // positions are not known here
  da->eps = eps;
  fill_turn_freq(theta, 128, da->turn_freq);
  da->pos_dev = start_pos;
  da->pos_valid = reinterpret_cast<uint32_t*>(ws + 16);
  // no host synchronisation and no host-side reads of device memory: the
  // call can be captured into a CUDA graph and replayed with new positions
  return from_cuda(launch_decode(*da, static_cast<cudaStream_t>(stream)));
}

// ----- gated global attention (Qwen3-Next / Qwen3.5) -------------------------

static size_t gated_q_bytes(int B, int T, int Hq) { return (size_t)B * T * Hq * kGatedD * 2; }
static size_t gated_k_bytes(int B, int T, int Hkv) { return (size_t)B * T * Hkv * kGatedD * 2; }

size_t q3a_gated_prefill_workspace_size(int B, int T, int Hq, int Hkv, int d) {
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || d != kGatedD) return 0;
  return kHeader + align256(gated_q_bytes(B, T, Hq)) + align256(gated_k_bytes(B, T, Hkv));
}

static q3a_status gated_check(const void* const* ptrs, int nptrs, int B, int T, int Hq, int Hkv,
                              int d, void* workspace, size_t ws_bytes, bool* empty) {
  *empty = false;
  if (d != kGatedD || B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv) return Q3A_EINVAL;
  if ((long long)B * T * Hq > 0x7fffffffLL || T > (1 << 30)) return Q3A_EINVAL;
  if (Hq + Hkv > gated_prologue_max_heads()) return Q3A_EINVAL;
  // a valid grouping that the 128-row GQA packing does not cover (e.g. 24/4)
  if (!gated_group_ok(Hq, Hkv)) return Q3A_ENOTIMPL;
  if (B == 0 || T == 0) {
    *empty = true;
    return Q3A_OK;
  }
  for (int i = 0; i < nptrs; ++i)
    if (!ptrs[i] || !aligned16(ptrs[i])) return Q3A_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return Q3A_EINVAL;
  if (ws_bytes < q3a_gated_prefill_workspace_size(B, T, Hq, Hkv, d)) return Q3A_EINVAL;
  return Q3A_OK;
}

static uint16_t* gated_ws_q(void* ws) { return reinterpret_cast<uint16_t*>((uint8_t*)ws + kHeader); }
static uint16_t* gated_ws_k(void* ws, int B, int T, int Hq) {
  return reinterpret_cast<uint16_t*>((uint8_t*)ws + kHeader + align256(gated_q_bytes(B, T, Hq)));
}

static void gated_prologue_args(GatedPrologueArgs& ga, const q3a_bf16* qg, const q3a_bf16* k,
                                const q3a_bf16* q_w, const q3a_bf16* k_w, int B, int T, int Hq,
                                int Hkv, int d_rot, double theta, float eps, void* workspace) {
  memset(&ga, 0, sizeof ga);
  ga.qg = qg;
  ga.k = k;
  ga.q_w = q_w;
  ga.k_w = k_w;
  ga.qhat = gated_ws_q(workspace);
  ga.khat = gated_ws_k(workspace, B, T, Hq);
  ga.khat_rows = T;
  ga.err_clear = reinterpret_cast<uint32_t*>(workspace);
  ga.logit_bound = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 8);
  ga.B = B;
  ga.T = T;
  ga.Hq = Hq;
  ga.Hkv = Hkv;
  ga.d_r = d_rot;
  ga.eps = eps;
  if (d_rot > 0) fill_turn_freq(theta, d_rot, ga.turn_freq);
}

static q3a_status gated_attention_args(GatedAttnArgs& ga, const q3a_bf16* qg, const q3a_bf16* v,
                                       q3a_bf16* out, int B, int T, int Hq, int Hkv,
                                       void* workspace) {
  memset(&ga, 0, sizeof ga);
  const int g = Hq / Hkv;
  const uint64_t row = kGatedD * 2;  // bytes of one head row
  const uint64_t dq[4] = {kGatedD, (uint64_t)Hq, (uint64_t)T, (uint64_t)B};
  const uint64_t sq[3] = {row, (uint64_t)Hq * row, (uint64_t)T * Hq * row};
  const uint32_t bq[4] = {64, (uint32_t)g, (uint32_t)(128 / g), 1};
  const uint64_t dk[3] = {kGatedD, (uint64_t)T, (uint64_t)B * Hkv};
  const uint64_t sk[2] = {row, (uint64_t)T * row};
  const uint32_t bk[3] = {64, 64, 1};
  const uint64_t dv[4] = {kGatedD, (uint64_t)Hkv, (uint64_t)T, (uint64_t)B};
  const uint64_t sv[3] = {row, (uint64_t)Hkv * row, (uint64_t)T * Hkv * row};
  const uint32_t bv[4] = {64, 1, 128, 1};
  if (encode_tensor_map(&ga.tm_q, gated_ws_q(workspace), 4, dq, sq, bq) != CUDA_SUCCESS ||
      encode_tensor_map(&ga.tm_k, gated_ws_k(workspace, B, T, Hq), 3, dk, sk, bk) !=
          CUDA_SUCCESS ||
      encode_tensor_map(&ga.tm_v, v, 4, dv, sv, bv) != CUDA_SUCCESS)
    return Q3A_ECUDA;
  ga.qg = qg;
  ga.out = out;
  ga.err = reinterpret_cast<uint32_t*>(workspace);
  ga.logit_bound = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + 8);
  ga.B = B;
  ga.T = T;
  ga.Hq = Hq;
  ga.Hkv = Hkv;
  ga.g = g;
  const int tok = gated_tokens_per_cta(g);
  ga.n_mtiles = (T + tok - 1) / tok;
  return Q3A_OK;
}

// K6 reading K and V from head-major caches [B, Hkv, S_max, 256] (rows
// 0..T-1 written by the prologue): the maps stop at row T, so the tensor-memory
// unit returns zeros past the prompt whatever the cache holds there.
static q3a_status gated_attention_cache_args(GatedAttnArgs& ga, const q3a_bf16* qg,
                                             const q3a_bf16* k_cache, const q3a_bf16* v_cache,
                                             q3a_bf16* out, int B, int T, int Hq, int Hkv,
                                             int S_max, void* workspace) {
  memset(&ga, 0, sizeof ga);
  const int g = Hq / Hkv;
  const uint64_t row = kGatedD * 2;
  const uint64_t dq[4] = {kGatedD, (uint64_t)Hq, (uint64_t)T, (uint64_t)B};
  const uint64_t sq[3] = {row, (uint64_t)Hq * row, (uint64_t)T * Hq * row};
  const uint32_t bq[4] = {64, (uint32_t)g, (uint32_t)(128 / g), 1};
  const uint64_t dc[3] = {kGatedD, (uint64_t)T, (uint64_t)B * Hkv};
  const uint64_t sc[2] = {row, (uint64_t)S_max * row};
  const uint32_t bk[3] = {64, 64, 1};
  const uint32_t bv[3] = {64, 128, 1};
  if (encode_tensor_map(&ga.tm_q, gated_ws_q(workspace), 4, dq, sq, bq) != CUDA_SUCCESS ||
      encode_tensor_map(&ga.tm_k, k_cache, 3, dc, sc, bk) != CUDA_SUCCESS ||
      encode_tensor_map(&ga.tm_v, v_cache, 3, dc, sc, bv) != CUDA_SUCCESS)
    return Q3A_ECUDA;
  ga.qg = qg;
  ga.out = out;
  ga.err = reinterpret_cast<uint32_t*>(workspace);
  ga.logit_bound = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + 8);
  ga.B = B;
  ga.T = T;
  ga.Hq = Hq;
  ga.Hkv = Hkv;
  ga.g = g;
  const int tok = gated_tokens_per_cta(g);
  ga.n_mtiles = (T + tok - 1) / tok;
  ga.v_head_major = 1;
  return Q3A_OK;
}

static bool d_rot_ok(int d_rot) { return d_rot >= 0 && d_rot <= kGatedD && (d_rot & 15) == 0; }

q3a_status q3a_gated_prefill(const q3a_bf16* qg, const q3a_bf16* k, const q3a_bf16* v,
                             const q3a_bf16* q_w, const q3a_bf16* k_w, q3a_bf16* out, int B,
                             int T, int Hq, int Hkv, int d, int d_rot, double theta, float eps,
                             void* workspace, size_t ws_bytes, void* stream) {
  if (!scalars_ok(theta, eps) || !d_rot_ok(d_rot)) return Q3A_EINVAL;
  const void* ptrs[] = {qg, k, v, q_w, k_w, out};
  bool empty;
  q3a_status s = gated_check(ptrs, 6, B, T, Hq, Hkv, d, workspace, ws_bytes, &empty);
  if (s != Q3A_OK || empty) return s;
  GatedAttnArgs aa;  // tensor maps first: a failure there launches nothing
  s = gated_attention_args(aa, qg, v, out, B, T, Hq, Hkv, workspace);
  if (s != Q3A_OK) return s;
  GatedPrologueArgs pa;
  gated_prologue_args(pa, qg, k, q_w, k_w, B, T, Hq, Hkv, d_rot, theta, eps, workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_gated_prologue(pa, st);
  if (e == cudaSuccess) e = launch_gated_attention(aa, st);
  return from_cuda(e);
}

q3a_status q3a_gated_prefill_prologue(const q3a_bf16* qg, const q3a_bf16* k,
                                      const q3a_bf16* q_w, const q3a_bf16* k_w, int B, int T,
                                      int Hq, int Hkv, int d, int d_rot, double theta, float eps,
                                      void* workspace, size_t ws_bytes, void* stream) {
  if (!scalars_ok(theta, eps) || !d_rot_ok(d_rot)) return Q3A_EINVAL;
  const void* ptrs[] = {qg, k, q_w, k_w};
  bool empty;
  q3a_status s = gated_check(ptrs, 4, B, T, Hq, Hkv, d, workspace, ws_bytes, &empty);
  if (s != Q3A_OK || empty) return s;
  GatedPrologueArgs pa;
  gated_prologue_args(pa, qg, k, q_w, k_w, B, T, Hq, Hkv, d_rot, theta, eps, workspace);
  return from_cuda(launch_gated_prologue(pa, static_cast<cudaStream_t>(stream)));
}

q3a_status q3a_gated_prefill_attention(const q3a_bf16* qg, const q3a_bf16* v, q3a_bf16* out,
                                       int B, int T, int Hq, int Hkv, int d, void* workspace,
                                       size_t ws_bytes, void* stream) {
  const void* ptrs[] = {qg, v, out};
  bool empty;
  q3a_status s = gated_check(ptrs, 3, B, T, Hq, Hkv, d, workspace, ws_bytes, &empty);
  if (s != Q3A_OK || empty) return s;
  GatedAttnArgs aa;
  s = gated_attention_args(aa, qg, v, out, B, T, Hq, Hkv, workspace);
  if (s != Q3A_OK) return s;
  return from_cuda(launch_gated_attention(aa, static_cast<cudaStream_t>(stream)));
}

size_t q3a_gated_decode_workspace_size(int B, int Hq, int Hkv, int d, int S_max) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || d != kGatedD || S_max <= 0 || Hq % Hkv) return 0;
  const size_t parts = (size_t)B * Hkv * decode_split_stride(S_max, kGatedD) * (Hq / Hkv) *
                       decode_partial_floats(kGatedD) * sizeof(float);
  return kHeader + align256(parts);
}

size_t q3a_gated_prefill_fill_workspace_size(int B, int T, int Hq, int Hkv, int d) {
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || d != kGatedD) return 0;
  return kHeader + align256(gated_q_bytes(B, T, Hq));
}

q3a_status q3a_gated_prefill_fill(const q3a_bf16* qg, const q3a_bf16* k, const q3a_bf16* v,
                                  q3a_bf16* k_cache, q3a_bf16* v_cache, const q3a_bf16* q_w,
                                  const q3a_bf16* k_w, q3a_bf16* out, int B, int T, int Hq,
                                  int Hkv, int d, int d_rot, int S_max, double theta, float eps,
                                  void* workspace, size_t ws_bytes, void* stream) {
  if (!scalars_ok(theta, eps) || !d_rot_ok(d_rot)) return Q3A_EINVAL;
  if (d != kGatedD || B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv) return Q3A_EINVAL;
  if (S_max <= 0 || S_max > (1 << 30)) return Q3A_EINVAL;
  if ((long long)B * T * Hq > 0x7fffffffLL) return Q3A_EINVAL;
  if (Hq + 2 * Hkv > gated_prologue_max_heads()) return Q3A_EINVAL;
  if (!gated_group_ok(Hq, Hkv)) return Q3A_ENOTIMPL;
  if (T > S_max) return Q3A_ERANGE;  // the prompt does not fit the caches; nothing written
  if (B == 0 || T == 0) return Q3A_OK;
  const void* ptrs[] = {qg, k, v, k_cache, v_cache, q_w, k_w, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return Q3A_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return Q3A_EINVAL;
  if (ws_bytes < q3a_gated_prefill_fill_workspace_size(B, T, Hq, Hkv, d)) return Q3A_EINVAL;
  GatedAttnArgs aa;  // tensor maps first: a failure there launches nothing
  q3a_status s = gated_attention_cache_args(aa, qg, k_cache, v_cache, out, B, T, Hq, Hkv, S_max,
                                            workspace);
  if (s != Q3A_OK) return s;
  GatedPrologueArgs pa;
  gated_prologue_args(pa, qg, k, q_w, k_w, B, T, Hq, Hkv, d_rot, theta, eps, workspace);
  pa.khat = k_cache;  // normalised, rotated keys straight into cache rows 0..T-1
  pa.khat_rows = S_max;
  pa.v = v;
  pa.v_cache = v_cache;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_gated_prologue(pa, st);
  if (e == cudaSuccess) e = launch_gated_attention(aa, st);
  return from_cuda(e);
}

size_t q3a_gated_prefill_chunk_workspace_size(int B, int Tq, int Hq, int Hkv, int d) {
  return q3a_gated_prefill_fill_workspace_size(B, Tq, Hq, Hkv, d);
}

q3a_status q3a_gated_prefill_chunk(const q3a_bf16* qg, const q3a_bf16* k, const q3a_bf16* v,
                                   q3a_bf16* k_cache, q3a_bf16* v_cache,
                                   const int32_t* start_pos, const q3a_bf16* q_w,
                                   const q3a_bf16* k_w, q3a_bf16* out, int B, int Tq, int Hq,
                                   int Hkv, int d, int d_rot, int S_max, double theta, float eps,
                                   void* workspace, size_t ws_bytes, void* stream) {
  if (!scalars_ok(theta, eps) || !d_rot_ok(d_rot)) return Q3A_EINVAL;
  if (d != kGatedD || B < 0 || Tq < 0 || B > kMaxBatch || Hq <= 0 || Hkv <= 0 || Hq % Hkv)
    return Q3A_EINVAL;
  if (S_max <= 0 || S_max > (1 << 30)) return Q3A_EINVAL;
  if ((long long)B * Tq * Hq > 0x7fffffffLL) return Q3A_EINVAL;
  if (Hq + 2 * Hkv > gated_prologue_max_heads()) return Q3A_EINVAL;
  if (!gated_group_ok(Hq, Hkv)) return Q3A_ENOTIMPL;
  if (B == 0 || Tq == 0) return Q3A_OK;
  const void* ptrs[] = {qg, k, v, k_cache, v_cache, q_w, k_w, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return Q3A_EINVAL;
  if (!start_pos) return Q3A_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return Q3A_EINVAL;
  if (ws_bytes < q3a_gated_prefill_chunk_workspace_size(B, Tq, Hq, Hkv, d)) return Q3A_EINVAL;
  for (int b = 0; b < B; ++b) {
    const int32_t p = start_pos[b];
    if (p < 0 || (long long)p + Tq > S_max) return Q3A_ERANGE;  // nothing written yet
  }
  const int g = Hq / Hkv;
  uint16_t* qhat = gated_ws_q(workspace);

  // tensor maps first: a failure there launches nothing. K and V maps cover
  // all S_max rows of each (b, kv): the valid rows differ per sequence, so the
  // attention kernel masks the keys and clears the V rows past them itself
  GatedAttnChunkArgs ca;
  memset(&ca, 0, sizeof ca);
  GatedAttnArgs& aa = ca.base;
  {
    const uint64_t row = kGatedD * 2;
    const uint64_t dq[4] = {kGatedD, (uint64_t)Hq, (uint64_t)Tq, (uint64_t)B};
    const uint64_t sq[3] = {row, (uint64_t)Hq * row, (uint64_t)Tq * Hq * row};
    const uint32_t bq[4] = {64, (uint32_t)g, (uint32_t)(128 / g), 1};
    const uint64_t dc[3] = {kGatedD, (uint64_t)S_max, (uint64_t)B * Hkv};
    const uint64_t sc[2] = {row, (uint64_t)S_max * row};
    const uint32_t bk[3] = {64, 64, 1};
    const uint32_t bv[3] = {64, 128, 1};
    if (encode_tensor_map(&aa.tm_q, qhat, 4, dq, sq, bq) != CUDA_SUCCESS ||
        encode_tensor_map(&aa.tm_k, k_cache, 3, dc, sc, bk) != CUDA_SUCCESS ||
        encode_tensor_map(&aa.tm_v, v_cache, 3, dc, sc, bv) != CUDA_SUCCESS)
      return Q3A_ECUDA;
  }
  aa.qg = qg;
  aa.out = out;
  aa.err = reinterpret_cast<uint32_t*>(workspace);
  aa.logit_bound = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + 8);
  aa.B = B;
  aa.T = Tq;
  aa.Hq = Hq;
  aa.Hkv = Hkv;
  aa.g = g;
  const int tok = gated_tokens_per_cta(g);
  aa.n_mtiles = (Tq + tok - 1) / tok;
  aa.v_head_major = 1;
  // cached keys were normalised with the same k_w by earlier calls (the
  // documented precondition), so the logit bound holds for them too; a cache
  // that breaks it badly enough to overflow a softmax sum is reported
  // (kErrWordBound)
  ca.fixed_shift_ok = 1;
  for (int b = 0; b < B; ++b) ca.pos_b[b] = start_pos[b];

  // Q -> Qhat [B, Tq, Hq]; K -> k_cache rows start_pos[b] + t (normalised,
  // rotated at their positions); V -> v_cache rows start_pos[b] + t (copied)
  GatedPrologueChunkArgs pc;
  memset(&pc, 0, sizeof pc);
  gated_prologue_args(pc.base, qg, k, q_w, k_w, B, Tq, Hq, Hkv, d_rot, theta, eps, workspace);
  pc.base.khat = k_cache;
  pc.base.khat_rows = S_max;
  pc.base.v = v;
  pc.base.v_cache = v_cache;
  for (int b = 0; b < B; ++b) pc.pos_b[b] = start_pos[b];

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_gated_prologue(pc, st);
  if (e == cudaSuccess) e = launch_gated_attention(ca, st);
  return from_cuda(e);
}

// Shared by q3a_gated_decode (positions on the host) and
// q3a_gated_decode_device_pos (positions in device memory, checked by a
// device-side pre-pass; no host read or synchronisation).
static q3a_status gated_decode_impl(const q3a_bf16* qg, const q3a_bf16* k_new,
                                    const q3a_bf16* v_new, q3a_bf16* k_cache, q3a_bf16* v_cache,
                                    const int32_t* start_pos, bool pos_on_device,
                                    const q3a_bf16* q_w, const q3a_bf16* k_w, q3a_bf16* out,
                                    int B, int Hq, int Hkv, int d, int d_rot, int S_max,
                                    double theta, float eps, void* workspace, size_t ws_bytes,
                                    void* stream) {
  if (d != kGatedD || B < 0 || B > kDecodeMaxB || S_max <= 0 || Hq <= 0 || Hkv <= 0 ||
      Hq % Hkv)
    return Q3A_EINVAL;
  if (S_max > (1 << 30) || !d_rot_ok(d_rot)) return Q3A_EINVAL;
  if (!scalars_ok(theta, eps)) return Q3A_EINVAL;
  if (!gated_group_ok(Hq, Hkv)) return Q3A_ENOTIMPL;  // the MMA rows hold at most 16 heads
  if (B == 0) return Q3A_OK;
  const void* ptrs[] = {qg, k_new, v_new, k_cache, v_cache, q_w, k_w, out};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return Q3A_EINVAL;
  if (!start_pos || (reinterpret_cast<uintptr_t>(start_pos) & 3u)) return Q3A_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return Q3A_EINVAL;
  if (ws_bytes < q3a_gated_decode_workspace_size(B, Hq, Hkv, d, S_max)) return Q3A_EINVAL;
  // device positions: every split may be needed
  int max_splits = decode_split_stride(S_max, kGatedD);
  if (!pos_on_device) {
    max_splits = 0;
    for (int b = 0; b < B; ++b) {
      const int32_t p = start_pos[b];
      if (p < 0 || (long long)p + 1 > S_max) return Q3A_ERANGE;  // nothing written yet
      const int n = (p + decode_chunk_keys(kGatedD)) / decode_chunk_keys(kGatedD);
      if (n > max_splits) max_splits = n;
    }
  }

  DecodeArgs dargs;  // kernel parameters, staged on the host stack
  DecodeArgs* da = &dargs;
  memset(da, 0, sizeof *da);
  const uint64_t row = kGatedD * 2;
  const uint64_t dc[3] = {kGatedD, (uint64_t)S_max, (uint64_t)B * Hkv};
  const uint64_t sc[2] = {row, (uint64_t)S_max * row};
  const uint32_t bc[3] = {64, 64, 1};
  if (encode_tensor_map(&da->tm_kc, k_cache, 3, dc, sc, bc) != CUDA_SUCCESS ||
      encode_tensor_map(&da->tm_vc, v_cache, 3, dc, sc, bc) != CUDA_SUCCESS)
    return Q3A_ECUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  da->q = qg;
  da->k_new = k_new;
  da->v_new = v_new;
  da->q_gamma = q_w;
  da->k_gamma = k_w;
  da->k_cache = k_cache;
  da->v_cache = v_cache;
  da->partial = reinterpret_cast<float*>(ws + kHeader);
  da->out = out;
  da->err = reinterpret_cast<uint32_t*>(ws);
  da->B = B;
  da->Hq = Hq;
  da->Hkv = Hkv;
  da->g = Hq / Hkv;
  da->S_max = S_max;
  da->split_stride = decode_split_stride(S_max, kGatedD);
  da->max_splits = max_splits;
  da->eps = eps;
  da->d_rot = d_rot;
  if (d_rot > 0) fill_turn_freq(theta, d_rot, da->turn_freq);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (pos_on_device) {
    da->pos_dev = start_pos;
    da->pos_valid = reinterpret_cast<uint32_t*>(ws + 16);
    return from_cuda(launch_gated_decode(*da, st));  // the check kernel writes the error word
  }
  for (int b = 0; b < B; ++b) da->start_pos[b] = start_pos[b];
  cudaError_t e = cudaMemsetAsync(da->err, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = launch_gated_decode(*da, st);
  return from_cuda(e);
}

q3a_status q3a_gated_decode(const q3a_bf16* qg, const q3a_bf16* k_new, const q3a_bf16* v_new,
                            q3a_bf16* k_cache, q3a_bf16* v_cache, const int32_t* start_pos,
                            const q3a_bf16* q_w, const q3a_bf16* k_w, q3a_bf16* out, int B,
                            int Hq, int Hkv, int d, int d_rot, int S_max, double theta, float eps,
                            void* workspace, size_t ws_bytes, void* stream) {
  return gated_decode_impl(qg, k_new, v_new, k_cache, v_cache, start_pos, false, q_w, k_w, out,
                           B, Hq, Hkv, d, d_rot, S_max, theta, eps, workspace, ws_bytes, stream);
}

q3a_status q3a_gated_decode_device_pos(const q3a_bf16* qg, const q3a_bf16* k_new,
                                       const q3a_bf16* v_new, q3a_bf16* k_cache,
                                       q3a_bf16* v_cache, const int32_t* start_pos,
                                       const q3a_bf16* q_w, const q3a_bf16* k_w, q3a_bf16* out,
                                       int B, int Hq, int Hkv, int d, int d_rot, int S_max,
                                       double theta, float eps, void* workspace,
                                       size_t ws_bytes, void* stream) {
  return gated_decode_impl(qg, k_new, v_new, k_cache, v_cache, start_pos, true, q_w, k_w, out,
                           B, Hq, Hkv, d, d_rot, S_max, theta, eps, workspace, ws_bytes, stream);
}

q3a_status q3a_last_device_error(const void* workspace, void* stream) {
  if (!workspace) {  // q3a_decode_noalloc's error word on the current device
    void* p = nullptr;
    if (noalloc_error_word(&p) != cudaSuccess) return Q3A_ECUDA;
    workspace = p;
  }
  uint32_t word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return Q3A_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return Q3A_ECUDA;
  if (word == 0) return Q3A_OK;
  if (word == kErrWordRange) return Q3A_ERANGE;
  if (word == kErrWordBound) return Q3A_EINVAL;
  return Q3A_ETIMEOUT;
}

}  // extern "C"
