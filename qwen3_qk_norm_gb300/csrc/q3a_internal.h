// q3a_internal.h — host-side interfaces between the C ABI (q3a_api.cu) and the
// kernels of libq3a. Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <vector>

namespace q3a {

// ----- K1: QK-Norm + RoPE prologue ------------------------------------------
// One tensor of head rows. The input x is token-contiguous: row (b, t, h) at
// element ((b * T + t) * H + h) * 128, i.e. xsb = T*H, xst = H, xsh = 1 (the
// kernel stages whole token blocks with bulk copies). Output row (b, t, h) of
// y starts at element (b * ysb + t * yst + h * ysh) * 128 (strides counted in
// rows of 128 elements).
struct RopeTensor {
  const uint16_t* x;
  const uint16_t* gamma;  // unused when copy_only
  uint16_t* y;
  int H;
  long long xsb, xst, xsh;
  long long ysb, yst, ysh;
  int copy_only;     // 1: rows are copied unchanged (values into a cache)
  int y_at_position; // 1: output row t of sequence b goes to row pos_b[b] + t
};

constexpr int kMaxBatch = 2048;  // sequences per call of the position-aware paths

struct RopeArgs {
  RopeTensor t[3];
  int ntensors;  // 1..3 (all tensors share B, T and the positions); tensors
                 // that normalise come first
  int B, T;
  long long pos0;  // row (b, t, h) is rotated at pos0 + t ...
  int per_b_pos;   // ... or, if set, at pos_b[b] + t
  int pos_b[kMaxBatch];
  float eps;
  int tok_per_cta;      // set by launch_qknorm_rope
  uint32_t* err_clear;  // if non-null, block 0 zeroes this error word
  // if non-null, block 0 writes here the bound on |q.k| / sqrt(128) * log2(e)
  // that QK-Norm guarantees: sqrt(128) * max|gamma_q| * max|gamma_k| * log2(e),
  // from bound_gamma[0] (gamma_q) and bound_gamma[1] (gamma_k)
  float* logit_bound;
  const uint16_t* bound_gamma[2];
  // if non-null: the (cos, sin) of every angle i < 64 at positions 0..T-1,
  // [T][64] float2, written by the CTAs of sequence 0 (plain prefill only)
  float* rope_table;
  unsigned long long turn_freq[64];  // theta^(-2i/128) / (2 pi), 0.64 fixed point
};

// RoPE frequencies theta^(-2i/d_rot), i < d_rot/2, as fractions of a turn in
// 0.64 fixed point, so that the angle of position p is p * turn_freq[i] modulo
// 2^64 (exact wrap-around). Writes d_rot/2 entries (d_rot even, <= 256).
void fill_turn_freq(double theta, int d_rot, unsigned long long* turn_freq);
int qknorm_rope_max_heads();  // largest H0 + H1 one launch accepts
cudaError_t launch_qknorm_rope(const RopeArgs& a, cudaStream_t stream);

// ----- K2: causal GQA prefill attention (tcgen05) ---------------------------
struct PrefillArgs {
  // plain prefill: raw q [B, T, Hq, 128], normalised and rotated in shared
  // memory by the kernel itself; chunk: Qhat from the prologue. Box {64, g, 128/g, 1}
  CUtensorMap tm_q;
  CUtensorMap tm_k;  // Khat [B*Hkv, rows, 128] bf16, box {64, 128, 1} (workspace or cache)
  CUtensorMap tm_v;  // V [B, T, Hkv, 128], box {64, 1, 128, 1}; or, for a chunk,
                     // [B*Hkv, S_max, 128] (the cache), box {64, 128, 1}
  uint16_t* out;     // [B, T, Hq, 128] bf16
  uint32_t* err;     // device error word
  const float* logit_bound;  // written by the prologue (see RopeArgs)
  int B, T, Hq, Hkv, g;
  int n_mtiles;      // ceil(T / prefill_tokens_per_cta(g))
  int group_sets;    // chunk: the (b, kv) groups' work items in this many
                     // sets, one after another (a power of two dividing
                     // B * Hkv, set by the launcher)
  // the plain prefill's Q-Norm + RoPE of the query tiles (unused by a chunk)
  const uint16_t* q_gamma;   // [128]
  float eps;
  const float* rope_table;   // [T][64] (cos, sin) pairs, written by the prologue
};

// A chunk against the caches: keys and values are read from the head-major
// caches, and token t of sequence b sits at position pos_b[b] + t.
struct PrefillChunkArgs {
  PrefillArgs base;
  int fixed_shift_ok;  // 0: cached keys present, always use the online max
  int pos_b[kMaxBatch];
};

// Work items of the persistent attention kernels (K2, K6). Item i is a pair
// of Q tiles (m-tile mt) of one (b, kv) group. The groups are split into
// equal sets of `per` groups taken one after another; within a set items go
// longest first (mt descending), the set's groups interleaved. With one set
// every group is in flight at once; with more, fewer groups are, so more
// workers read each group's K/V prefix at about the same time and fewer K/V
// bytes have to stay in L2 between their reads.
struct ItemIndex {
  int bk, mt;
};
__host__ __device__ __forceinline__ ItemIndex item_index(int i, int n_mtiles, int per) {
  const int set = i / (per * n_mtiles), j = i - set * per * n_mtiles;
  return ItemIndex{set * per + j % per, n_mtiles - 1 - j / per};
}
// KV tiles of `keys_per_tile` keys that an item of tokens_per_item tokens
// from token t0 reaches: its last token t_last sits at position p0 + t_last
__host__ __device__ __forceinline__ int item_kv_tiles(int t0, int tokens_per_item, int T, int p0,
                                                      int keys_per_tile) {
  const int t_last = (t0 + tokens_per_item < T ? t0 + tokens_per_item : T) - 1;
  return (p0 + t_last) / keys_per_tile + 1;
}
// The number of group sets (1, 2, 4 or 8, a power of two dividing B * Hkv)
// for `workers` persistent workers taking items in snake order over rounds:
// the schedule is replayed on the host for each count, an item costing its KV
// tiles plus a fixed boundary cost of about four tiles (the last PV, the
// epilogue and the next item's first QK^T, measured at an item boundary), and
// the count with the smallest busiest-worker total is kept; on a tie the
// larger count (fewer groups in flight). p0_b: each sequence's first position
// (null: 0).
inline int choose_group_sets(int n_mtiles, int B, int Hkv, int tokens_per_item, int T,
                             const int* p0_b, int keys_per_tile, int workers) {
  constexpr int kItemCost = 4;
  constexpr long long kMaxReplay = 1 << 16;  // beyond this many items: one set
  const int bk_count = B * Hkv;
  const long long n_items = (long long)n_mtiles * bk_count;
  if (n_items <= 0 || n_items > kMaxReplay || workers <= 0) return 1;
  std::vector<long long> load((size_t)workers);
  int best = 1;
  long long best_max = -1;
  for (int sets = 1; sets <= 8; sets *= 2) {
    if (bk_count % sets) break;
    std::fill(load.begin(), load.end(), 0LL);
    for (long long i = 0; i < n_items; ++i) {
      const long long r = i / workers, k = i % workers;
      const int w = (int)((r & 1) ? workers - 1 - k : k);
      const ItemIndex ix = item_index((int)i, n_mtiles, bk_count / sets);
      const int p0 = p0_b ? p0_b[ix.bk / Hkv] : 0;
      load[(size_t)w] +=
          item_kv_tiles(ix.mt * tokens_per_item, tokens_per_item, T, p0, keys_per_tile) + kItemCost;
    }
    const long long mx = *std::max_element(load.begin(), load.end());
    if (best_max < 0 || mx <= best_max) {
      best = sets;
      best_max = mx;
    }
  }
  return best;
}

cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_attention(const PrefillChunkArgs& a, cudaStream_t stream);
// tokens of one KV group that one attention CTA covers (n_mtiles = ceil(T / this))
int prefill_tokens_per_cta(int g);

// ----- K3/K4: split-KV decode ------------------------------------------------
// One kernel pair serves the Qwen3 decode (head_dim 128, QK-Norm with gamma,
// full rotate-half RoPE) and the gated decode of the Qwen3-Next / Qwen3.5
// global layer (head_dim 256, zero-centred norm with scale 1 + w, RoPE of the
// first d_rot coordinates, output multiplied by sigmoid(gate)).
constexpr int kDecodeMaxB = kMaxBatch;
constexpr int kDecodeChunk = 1024;  // keys per split at head_dim 128
// keys per split: at head_dim 256 one CTA runs per SM, so longer splits
// amortise each split's fixed start and merge over more streamed keys
constexpr int decode_chunk_keys(int d) { return d == 128 ? kDecodeChunk : 2 * kDecodeChunk; }
// m, l, acc[d] per (split, head)
constexpr int decode_partial_floats(int d) { return 2 + d; }
constexpr int kDecodePartialFloats = decode_partial_floats(128);

struct DecodeArgs {
  CUtensorMap tm_kc;  // k_cache [B*Hkv, S_max, d] bf16, box {64, 64, 1}
  CUtensorMap tm_vc;  // v_cache, same
  const uint16_t* q;      // [B, Hq, d]; gated: [B, Hq, 2d], query then gate per head
  const uint16_t* k_new;  // [B, Hkv, d]
  const uint16_t* v_new;  // [B, Hkv, d]
  const uint16_t* q_gamma;  // [d]; gated: the zero-centred weights w_q
  const uint16_t* k_gamma;  // [d]; gated: w_k
  uint16_t* k_cache;  // for the append
  uint16_t* v_cache;
  float* partial;     // [B, Hkv, split_stride, g, decode_partial_floats(d)] fp32
  uint16_t* out;      // [B, Hq, d]
  uint32_t* err;
  int B, Hq, Hkv, g, S_max, split_stride, max_splits;
  float eps;
  int d_rot;  // gated: rotated leading coordinates (a multiple of 16)
  unsigned long long turn_freq[128];  // theta^(-2i/d_rot) / (2 pi); d_rot = 128 for Qwen3
  int start_pos[kDecodeMaxB];  // host positions, copied into the parameters ...
  // ... or, when pos_dev is set, positions read on the device: a one-block
  // check writes *pos_valid (1: every position in range) and the error word
  // before the decode kernels run; with *pos_valid == 0 they write nothing
  const int32_t* pos_dev;
  uint32_t* pos_valid;
};

// error word value of a device-side position check that failed
constexpr uint32_t kErrWordRange = 0x201;
// error word value when a chunk's softmax sum overflowed: its cached keys
// exceed the norm bound that this library's keys obey by far
constexpr uint32_t kErrWordBound = 0x301;

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);        // d = 128
// device address of q3a_decode_noalloc's error word on the current device
cudaError_t noalloc_error_word(void** out);
cudaError_t launch_gated_decode(const DecodeArgs& a, cudaStream_t stream);  // d = 256

// ----- K5/K6: gated global attention of Qwen3-Next / Qwen3.5 (d = 256) ------
constexpr int kGatedD = 256;
// K5: zero-centred QK-Norm + partial RoPE. The query rows are the first 256
// elements of each 512-element head block of qg [B, T, Hq, 512] (the last 256
// are the gate, read by K6); k is [B, T, Hkv, 256].
struct GatedPrologueArgs {
  const uint16_t* qg;
  const uint16_t* k;
  const uint16_t* q_w;  // [256] zero-centred weights: the scale is 1 + w
  const uint16_t* k_w;
  uint16_t* qhat;       // [B, T, Hq, 256]
  uint16_t* khat;       // head-major: row (b, kv, t) at ((b * Hkv + kv) * khat_rows + t) * 256
  long long khat_rows;  // T for the workspace, S_max for a K cache
  // if non-null: v [B, T, Hkv, 256] is copied unchanged into v_cache rows
  // (same head-major addressing as khat)
  const uint16_t* v;
  uint16_t* v_cache;
  uint32_t* err_clear;  // block 0 zeroes this error word
  // block 0 writes here sqrt(256) * max|1 + w_q| * max|1 + w_k| * log2(e), the
  // bound on |qhat . khat| / sqrt(256) * log2(e) that the norm guarantees
  float* logit_bound;
  int B, T, Hq, Hkv, d_r;
  float eps;
  int tok_per_cta;  // set by launch_gated_prologue
  unsigned long long turn_freq[128];  // theta^(-2i/d_r) / (2 pi), i < d_r/2
};
// A chunk against the caches: token t of sequence b is rotated at position
// pos_b[b] + t and its key and value go to cache row pos_b[b] + t
// (khat = k_cache, khat_rows = S_max, v and v_cache set).
struct GatedPrologueChunkArgs {
  GatedPrologueArgs base;
  int pos_b[kMaxBatch];
};
int gated_prologue_max_heads();
cudaError_t launch_gated_prologue(const GatedPrologueArgs& a, cudaStream_t stream);
cudaError_t launch_gated_prologue(const GatedPrologueChunkArgs& a, cudaStream_t stream);

// K6: causal GQA attention over Qhat/Khat with the sigmoid output gate, on
// pairs of CTAs (clusters of two).
struct GatedAttnArgs {
  CUtensorMap tm_q;  // Qhat [B, T, Hq, 256], box {64, g, 128/g, 1}
  CUtensorMap tm_k;  // Khat [B*Hkv, T, 256], box {64, 64, 1}
  CUtensorMap tm_v;  // V [B, T, Hkv, 256], box {64, 1, 128, 1}; or, when v_head_major,
                     // a V cache [B*Hkv, T rows, 256] (row stride S_max), box {64, 128, 1}
  const uint16_t* qg;  // gate = qg[b, t, h, 256 .. 511]
  uint16_t* out;       // [B, T, Hq, 256] bf16
  uint32_t* err;
  const float* logit_bound;
  int B, T, Hq, Hkv, g;
  int n_mtiles;  // pair tiles: ceil(T / gated_tokens_per_cta(g))
  int v_head_major;
  int group_sets;  // chunk: the (b, kv) groups' work items in this many sets,
                   // one after another (a power of two dividing B * Hkv,
                   // set by the launcher)
};
// A chunk against the caches: K and V come from the head-major caches (maps
// over all S_max rows, v_head_major set) and token t of sequence b sits at
// position pos_b[b] + t, seeing keys 0..pos_b[b] + t.
struct GatedAttnChunkArgs {
  GatedAttnArgs base;
  int fixed_shift_ok;  // 0: cached keys present, always use the online max
  int pos_b[kMaxBatch];
};
cudaError_t launch_gated_attention(const GatedAttnArgs& a, cudaStream_t stream);
cudaError_t launch_gated_attention(const GatedAttnChunkArgs& a, cudaStream_t stream);
int gated_tokens_per_cta(int g);  // tokens of one KV group that a pair of CTAs covers

// ----- tensor maps -----------------------------------------------------------
// cuTensorMapEncodeTiled (bf16, 128-byte swizzle, zero fill out of bounds),
// obtained through the runtime's driver entry point. dims[0] is innermost;
// strides_bytes has rank-1 entries (dims 1..rank-1).
CUresult encode_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace q3a
