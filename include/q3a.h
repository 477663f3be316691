/*
 * q3a.h — C ABI of the Qwen3 attention core for one NVIDIA GB300 (sm_103a).
 *
 * The library computes, from already-projected Q/K/V, the span of the Qwen3
 * attention sublayer between the projections and o_proj:
 *
 *   1. QK-Norm: per-head RMSNorm over head_dim with fp32 accumulation and a
 *      learned gamma, one gamma[d] shared by all Q heads and one by all K heads
 *      ("Qwen3" note, llm.rainlin.net, QK-Norm section and the quoted
 *      transformers Qwen3Attention; "7.2 Qwen3 full-scale implementation",
 *      paper.xwysyy.cn, §7.2.1 RMSNorm).
 *   2. Rotate-half RoPE with inv_freq_i = theta^(-2i/d), applied AFTER the norm
 *      (§7.2.1 compute_rope_params / apply_rope; the transformers forward
 *      quoted on the llm.rainlin.net page).
 *   3. Causal grouped-query softmax attention, softmax(q.k / sqrt(d)) . V, where
 *      query head h reads KV group floor(h / g), g = Hq / Hkv (§7.2.1
 *      GroupedQueryAttention: repeat_interleave, triu mask, scale head_dim^0.5).
 *   4. Decode: the new K is normalised and rotated at position start_pos and
 *      appended to the cache; cached K is used as stored and never re-rotated
 *      ("Chapter 20, Qwen3 and Qwen3.5", book.ozine.me, §20.3 KV cache).
 *
 * Conventions shared by every entry point
 *   - bf16 means IEEE bfloat16 bit patterns (q3a_bf16), round-to-nearest-even.
 *   - Every tensor pointer is a DEVICE pointer unless the comment says HOST.
 *     All device tensors are dense, row-major in the order given, and 16-byte
 *     aligned.
 *   - The caller owns every buffer, including the workspace. The library never
 *     allocates or frees memory. It launches asynchronously on `stream`
 *     (a cudaStream_t passed as void*; NULL = legacy default stream).
 *   - Arguments are validated on the host BEFORE anything is launched or
 *     written. A rejected call leaves every buffer untouched (the
 *     validate-then-mutate rule of the context-length tests, §20.9 of the
 *     book.ozine.me chapter).
 *   - The library never aborts and never prints.
 *   - head_dim d must be 128 (the fixed Qwen3 head width, §7.2.1).
 *   - Hq % Hkv == 0 and g = Hq/Hkv in {1, 2, 4, 8, 16}.
 *   - eps > 0 and theta > 1.
 */
#ifndef Q3A_H_
#define Q3A_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t q3a_bf16;

typedef enum {
  Q3A_OK = 0,
  Q3A_EINVAL = 1,   /* bad argument: null/misaligned pointer, shape, eps, theta, workspace too small */
  Q3A_ERANGE = 2,   /* decode: start_pos[b] < 0 or start_pos[b] + 1 > S_max (context overflow) */
  Q3A_ECUDA = 3,    /* a CUDA launch or runtime call failed */
  Q3A_ETIMEOUT = 4, /* a device-side bounded wait gave up; see q3a_last_device_error */
  Q3A_ENOTIMPL = 5  /* combination of arguments that this build does not implement */
} q3a_status;

/* Human-readable name of a status code. Static storage; never NULL. */
const char* q3a_status_string(q3a_status s);

/* ---------------------------------------------------------------------------
 * q3a_qknorm_rope — steps 1 and 2 alone (QK-Norm then RoPE) on one tensor.
 *
 *   x     [B, T, H, d] bf16, projected Q or K as viewed per head.
 *   gamma [d] bf16, the norm's learned scale (shared by all H heads).
 *   y     [B, T, H, d] bf16, y = RoPE_pos(RMSNorm(x) * gamma), rounded once.
 *         y may equal x (in place); any other overlap is undefined.
 *   Row (b, t, h) is rotated at position pos0 + t.
 *   pos0 >= 0 and pos0 + T - 1 <= 2^30; H <= 512.
 *   B == 0, T == 0 or H == 0: returns Q3A_OK and launches nothing.
 * Sources: §7.2.1 RMSNorm forward (fp32 variance, rsqrt(var + eps), times
 * scale, cast back) and apply_rope (x*cos + cat(-x2, x1)*sin).
 * ------------------------------------------------------------------------- */
q3a_status q3a_qknorm_rope(const q3a_bf16* x, const q3a_bf16* gamma, q3a_bf16* y,
                           int B, int T, int H, int d, int pos0,
                           double theta, float eps, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_prefill — causal prefill of the whole attention core.
 *
 *   q       [B, T, Hq, d]  bf16 projected queries (token-major, per head).
 *   k, v    [B, T, Hkv, d] bf16 projected keys / values.
 *   q_gamma, k_gamma [d]   bf16 QK-Norm scales.
 *   out     [B, T, Hq, d]  bf16 attention output, i.e. [B, T, Hq*d], the layout
 *           that feeds o_proj (§7.2.1: context.transpose(1,2).reshape(b,T,d_out)).
 *   Positions are 0..T-1 (prefill always starts at position 0).
 *   Row (b, i, h) attends to keys j = 0..i of group h / (Hq/Hkv).
 *   Softmax scale is fixed to 1/sqrt(d).
 *   workspace: device scratch of at least q3a_prefill_workspace_size() bytes,
 *           256-byte aligned, owned by the caller, contents need not be
 *           initialised; it holds the normalised+rotated K, a table of the
 *           RoPE cos/sin of positions 0..T-1 and an error word (the query
 *           tiles are normalised and rotated in shared memory by the attention
 *           kernel itself). It must not be shared by two calls that run
 *           concurrently.
 *   B == 0 or T == 0: returns Q3A_OK and launches nothing.
 *   Limits: B*T*Hq <= 2^31 - 1 rows; Hq + Hkv <= 512.
 * ------------------------------------------------------------------------- */
size_t q3a_prefill_workspace_size(int B, int T, int Hq, int Hkv, int d);

q3a_status q3a_prefill(const q3a_bf16* q, const q3a_bf16* k, const q3a_bf16* v,
                       const q3a_bf16* q_gamma, const q3a_bf16* k_gamma,
                       q3a_bf16* out,
                       int B, int T, int Hq, int Hkv, int d,
                       double theta, float eps,
                       void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * The two halves of q3a_prefill, for callers that schedule them separately
 * (and for timing each kernel). q3a_prefill(...) is exactly
 * q3a_prefill_prologue(...) followed by q3a_prefill_attention(...) on the
 * same stream and workspace.
 *
 * q3a_prefill_prologue — steps 1-2 for the keys: normalises and rotates k
 *   (positions 0..T-1) into `workspace`, writes there the logit bound that
 *   QK-Norm implies (from q_gamma and k_gamma) and clears the workspace's
 *   error word. Same argument rules as q3a_prefill.
 * q3a_prefill_attention — steps 1-2 for the queries and step 3: the kernel
 *   loads each tile of q, normalises and rotates it in shared memory (q_gamma
 *   and eps as for q3a_prefill; the RoPE angles of each position come from a
 *   table the prologue leaves in the workspace), and computes the causal GQA
 *   attention against the keys that the last q3a_prefill_prologue with the
 *   same B, T, Hq, Hkv left in `workspace` and against v, into out. The
 *   workspace contents are only read. Calling it on a workspace that no
 *   prologue of these shapes has filled computes on whatever bytes are there
 *   (no fault, meaningless output).
 * Sources: as q3a_prefill.
 * ------------------------------------------------------------------------- */
q3a_status q3a_prefill_prologue(const q3a_bf16* k,
                                const q3a_bf16* q_gamma, const q3a_bf16* k_gamma,
                                int B, int T, int Hq, int Hkv, int d,
                                double theta, float eps,
                                void* workspace, size_t ws_bytes, void* stream);

q3a_status q3a_prefill_attention(const q3a_bf16* q, const q3a_bf16* v,
                                 const q3a_bf16* q_gamma, q3a_bf16* out,
                                 int B, int T, int Hq, int Hkv, int d, float eps,
                                 void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_prefill_chunk — prefill of a chunk of Tq new tokens per sequence
 * against a KV cache, appending the chunk to the cache.
 *
 *   q       [B, Tq, Hq, d]  bf16 projected queries of the chunk.
 *   k, v    [B, Tq, Hkv, d] bf16 projected keys / values of the chunk.
 *   k_cache, v_cache [B, Hkv, S_max, d] bf16: rows 0..start_pos[b]-1 hold the
 *           sequence's earlier keys (normalised and rotated, as this library
 *           writes them, with the same k_gamma) and values.
 *   start_pos HOST int32 [B]: position of the chunk's first token in
 *           sequence b; token t is at position start_pos[b] + t.
 *   out     [B, Tq, Hq, d] bf16: token t of sequence b attends to cache rows
 *           0..start_pos[b]-1 and the chunk's keys 0..t (causal).
 *   Side effect: k_cache[b, :, start_pos[b] + t] = bf16(RoPE(RMSNorm(k)))
 *   and v_cache[b, :, start_pos[b] + t] = v for t < Tq; other rows are
 *   neither read nor written.
 *   The softmax relies on the cached keys obeying the norm bound that keys
 *   normalised with this k_gamma obey (the precondition above); a cache that
 *   breaks it so far that a softmax sum overflows leaves those output rows
 *   undefined and q3a_last_device_error() returns Q3A_EINVAL.
 *   With start_pos[b] = 0 for all b this is q3a_prefill that also fills the
 *   cache; with Tq = 1 it computes what q3a_decode computes.
 *   Requires 0 <= start_pos[b] and start_pos[b] + Tq <= S_max for every b,
 *   else Q3A_ERANGE with the caches untouched. B <= 2048, S_max <= 2^30,
 *   Hq + 2 Hkv <= 512.
 *   workspace: at least q3a_prefill_chunk_workspace_size() bytes, 256-byte
 *   aligned, owned by the caller (normalised queries and an error word).
 *   B == 0 or Tq == 0: returns Q3A_OK and launches nothing.
 * Source: "Chapter 20, Qwen3 and Qwen3.5" (book.ozine.me), §20.3: a position
 * counter and a rectangular causal mask starting at pos_start; new keys are
 * rotated at their positions and concatenated to the cached ones; §20.9: the
 * chunked-cache check (chunks [0:2], [2:5], [5:6] against one forward).
 * ------------------------------------------------------------------------- */
size_t q3a_prefill_chunk_workspace_size(int B, int Tq, int Hq, int Hkv, int d);

q3a_status q3a_prefill_chunk(const q3a_bf16* q, const q3a_bf16* k, const q3a_bf16* v,
                             q3a_bf16* k_cache, q3a_bf16* v_cache,
                             const int32_t* start_pos,
                             const q3a_bf16* q_gamma, const q3a_bf16* k_gamma,
                             q3a_bf16* out,
                             int B, int Tq, int Hq, int Hkv, int d, int S_max,
                             double theta, float eps,
                             void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_decode — one new token per sequence against a KV cache.
 *
 *   q       [B, Hq, d]  bf16 projected query of the new token.
 *   k_new   [B, Hkv, d] bf16 projected key of the new token (NOT normalised).
 *   v_new   [B, Hkv, d] bf16 projected value of the new token.
 *   k_cache [B, Hkv, S_max, d] bf16, rows 0..start_pos[b]-1 hold keys that are
 *           already normalised and rotated (as this library writes them).
 *   v_cache [B, Hkv, S_max, d] bf16, rows 0..start_pos[b]-1 hold values.
 *   start_pos HOST int32 [B]: position of the new token of sequence b.
 *   out     [B, Hq, d] bf16 attention output of the new token.
 *   Side effect: k_cache[b, :, start_pos[b], :] = bf16(RoPE(RMSNorm(k_new)))
 *   and v_cache[b, :, start_pos[b], :] = v_new. Rows beyond start_pos[b] are
 *   neither read nor written.
 *   Requires 0 <= start_pos[b] and start_pos[b] + 1 <= S_max for every b,
 *   else Q3A_ERANGE with the caches untouched. B <= 2048, S_max <= 2^30.
 *   workspace: at least q3a_decode_workspace_size() bytes of device scratch,
 *   256-byte aligned, owned by the caller; holds split partials and an
 *   error word. Not shareable between concurrent calls.
 *   B == 0: returns Q3A_OK and launches nothing.
 * Source: §20.3 of the book.ozine.me chapter (the new K is rotated at
 * start_pos and concatenated; the old K is never rotated again) and the
 * cache update after RoPE in the quoted transformers forward.
 * ------------------------------------------------------------------------- */
size_t q3a_decode_workspace_size(int B, int Hq, int Hkv, int d, int S_max);

q3a_status q3a_decode(const q3a_bf16* q, const q3a_bf16* k_new, const q3a_bf16* v_new,
                      q3a_bf16* k_cache, q3a_bf16* v_cache,
                      const int32_t* start_pos,
                      const q3a_bf16* q_gamma, const q3a_bf16* k_gamma,
                      q3a_bf16* out,
                      int B, int Hq, int Hkv, int d, int S_max,
                      double theta, float eps,
                      void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_decode_device_pos — q3a_decode with the positions in DEVICE memory,
 * for decode loops captured into a CUDA graph (the positions change between
 * replays; the parameters of the captured launches do not).
 *
 *   Arguments as q3a_decode, except:
 *   start_pos DEVICE int32 [B], 4-byte aligned, read by the kernels when they
 *           run (the call never reads it on the host and never synchronises).
 *   Range check on the device: a one-block kernel checks
 *   0 <= start_pos[b] < S_max for every b before the decode kernels run; if
 *   any position is out of range, nothing is written (caches and out are
 *   left as they were) and the workspace's error word records it:
 *   q3a_last_device_error() then returns Q3A_ERANGE. Host-checkable argument
 *   errors return Q3A_EINVAL at the call as for q3a_decode.
 *   Work: every split a sequence could need at S_max is launched; splits past
 *   a sequence's length exit at once.
 *   workspace: q3a_decode_workspace_size() bytes (the same as q3a_decode).
 * Source: as q3a_decode; the pages have no counterpart for graph capture or
 * device-resident positions (a serving-loop concern).
 * ------------------------------------------------------------------------- */
q3a_status q3a_decode_device_pos(const q3a_bf16* q, const q3a_bf16* k_new,
                                 const q3a_bf16* v_new,
                                 q3a_bf16* k_cache, q3a_bf16* v_cache,
                                 const int32_t* start_pos,
                                 const q3a_bf16* q_gamma, const q3a_bf16* k_gamma,
                                 q3a_bf16* out,
                                 int B, int Hq, int Hkv, int d, int S_max,
                                 double theta, float eps,
                                 void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_decode_noalloc — q3a_decode for callers that cannot allocate device
 * memory for a workspace: a plugin whose host framework owns every device
 * allocation and hands it none, or a latency-critical loop that must not call
 * cudaMalloc because cudaMalloc can synchronise the device. The scratch that
 * q3a_decode keeps in the caller's workspace (split partials and the error
 * word) lives instead in one static device array of
 * Q3A_DECODE_NOALLOC_SCRATCH_BYTES bytes inside the library; every GPU that
 * loads the library holds that array until the process exits. The pages have
 * no counterpart of this entry point: it exists for callers of this library.
 *
 *   Arguments, results, the cache append and the error rules are those of
 *   q3a_decode, without workspace and ws_bytes.
 *   Size limit: it needs 256 + 4 * 130 * B * Hkv * g * S bytes, where
 *   S = max over b of ceil((start_pos[b] + 1) / 1024) and g = Hq / Hkv; a
 *   call that needs more than Q3A_DECODE_NOALLOC_SCRATCH_BYTES returns
 *   Q3A_EINVAL before anything is launched or written.
 *   Device-side errors: its kernels keep their error word at the start of the
 *   array; q3a_last_device_error(NULL, stream) reads it for the current
 *   device (Q3A_ETIMEOUT if a bounded wait of the last call gave up).
 *   No allocation: it calls no cudaMalloc, cudaFree or allocating routine.
 *   Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and keeps it. Under
 *   CUDA's default lazy module loading that first lookup also loads the
 *   library's device code on the device, which reserves the array and can
 *   synchronise: make one warm-up call outside any latency-critical loop, and
 *   before any stream capture on the device. The address is kept for the
 *   life of the process: do not use this entry point after cudaDeviceReset
 *   (or in a different primary context) of a device it has already run on.
 *   Sharing: every call on a device uses the same array, which keeps the last
 *   call's contents (the error word is cleared at the start of each call).
 *   Calls whose executions overlap on the GPU (different streams, or several
 *   host threads) race on the array and may return wrong results; order them
 *   on one stream or serialise them.
 * ------------------------------------------------------------------------- */
#define Q3A_DECODE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

q3a_status q3a_decode_noalloc(const q3a_bf16* q, const q3a_bf16* k_new, const q3a_bf16* v_new,
                              q3a_bf16* k_cache, q3a_bf16* v_cache,
                              const int32_t* start_pos,
                              const q3a_bf16* q_gamma, const q3a_bf16* k_gamma,
                              q3a_bf16* out,
                              int B, int Hq, int Hkv, int d, int S_max,
                              double theta, float eps, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_gated_prefill — causal prefill of the gated global-attention layer of
 * Qwen3-Next / Qwen3.5 ("Chapter 20, Qwen3 and Qwen3.5" §20.4; "14. The Qwen
 * family", Qwen3-Next section).
 *
 *   qg      [B, T, Hq, 2d] bf16, the query projection viewed per head: for head
 *           h, qg[b, t, h, 0 .. d-1] is the query and qg[b, t, h, d .. 2d-1]
 *           the output gate (the split is inside each head's 2d block).
 *   k, v    [B, T, Hkv, d] bf16 projected keys / values.
 *   q_w, k_w [d] bf16 zero-centred norm weights: the norm scales by 1 + w.
 *   out     [B, T, Hq, d] bf16, z = sigmoid(gate) * softmax(q k^T / sqrt(d)) v
 *           (the input of the output projection), one rounding.
 *   Per head, Q and K are RMS-normalised (fp32) and scaled by 1 + w, then the
 *   first d_rot coordinates are rotated (rotate-half pairs (i, i + d_rot/2),
 *   frequencies theta^(-2i/d_rot), positions 0..T-1); the others pass through.
 *   d must be 256; d_rot a multiple of 16 in 0..256 (Qwen3-Next / Qwen3.5: 64).
 *   Hq / Hkv any whole ratio up to 16 (e.g. 16/2, 24/4, 32/2; above 16
 *   returns Q3A_ENOTIMPL); Hq + Hkv <= 192; B*T*Hq <= 2^31 - 1.
 *   workspace: device scratch of at least q3a_gated_prefill_workspace_size()
 *           bytes, 256-byte aligned, caller-owned, not shared by concurrent
 *           calls; it holds the normalised+rotated Q and K and the error word.
 *   B == 0 or T == 0: returns Q3A_OK and launches nothing. Every argument is
 *   checked before anything is launched.
 * q3a_gated_prefill_prologue / q3a_gated_prefill_attention — the two kernels
 *   of q3a_gated_prefill separately (same arguments and workspace; the
 *   attention half reads what the last prologue of the same shapes wrote, and
 *   reads the gate from qg).
 * ------------------------------------------------------------------------- */
size_t q3a_gated_prefill_workspace_size(int B, int T, int Hq, int Hkv, int d);

q3a_status q3a_gated_prefill(const q3a_bf16* qg, const q3a_bf16* k, const q3a_bf16* v,
                             const q3a_bf16* q_w, const q3a_bf16* k_w, q3a_bf16* out,
                             int B, int T, int Hq, int Hkv, int d, int d_rot,
                             double theta, float eps,
                             void* workspace, size_t ws_bytes, void* stream);

q3a_status q3a_gated_prefill_prologue(const q3a_bf16* qg, const q3a_bf16* k,
                                      const q3a_bf16* q_w, const q3a_bf16* k_w,
                                      int B, int T, int Hq, int Hkv, int d, int d_rot,
                                      double theta, float eps,
                                      void* workspace, size_t ws_bytes, void* stream);

q3a_status q3a_gated_prefill_attention(const q3a_bf16* qg, const q3a_bf16* v, q3a_bf16* out,
                                       int B, int T, int Hq, int Hkv, int d,
                                       void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_gated_prefill_fill — q3a_gated_prefill of a prompt (positions 0..T-1)
 * that also fills the KV caches a later q3a_gated_decode continues from
 * ("Chapter 20" §20.3: the prompt is prefilled, then only new tokens pass):
 * rows 0..T-1 of k_cache [B, Hkv, S_max, 256] receive the normalised, rotated
 * keys (bf16, the same values the attention reads) and rows 0..T-1 of v_cache
 * the values. `out` equals q3a_gated_prefill's bit for bit. T <= S_max (else
 * Q3A_ERANGE, nothing written); Hq + 2*Hkv <= 192; other rules as
 * q3a_gated_prefill. The workspace holds only the normalised queries and the
 * error word: q3a_gated_prefill_fill_workspace_size() bytes.
 * ------------------------------------------------------------------------- */
size_t q3a_gated_prefill_fill_workspace_size(int B, int T, int Hq, int Hkv, int d);

q3a_status q3a_gated_prefill_fill(const q3a_bf16* qg, const q3a_bf16* k, const q3a_bf16* v,
                                  q3a_bf16* k_cache, q3a_bf16* v_cache,
                                  const q3a_bf16* q_w, const q3a_bf16* k_w, q3a_bf16* out,
                                  int B, int T, int Hq, int Hkv, int d, int d_rot, int S_max,
                                  double theta, float eps,
                                  void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_gated_prefill_chunk — a chunk of Tq new tokens per sequence of the
 * gated global-attention layer against its KV caches, appending the chunk.
 *
 *   qg      [B, Tq, Hq, 2d] bf16: per head, the query (first d) and the gate.
 *   k, v    [B, Tq, Hkv, d] bf16 projected keys / values of the chunk.
 *   k_cache, v_cache [B, Hkv, S_max, d] bf16: rows 0..start_pos[b]-1 hold the
 *           sequence's earlier keys (zero-centred-normalised with the same
 *           k_w and partially rotated, as this library writes them) and values.
 *   start_pos HOST int32 [B]: token t of sequence b sits at start_pos[b] + t.
 *   out     [B, Tq, Hq, d] bf16: token t attends to cache rows
 *           0..start_pos[b]-1 and the chunk's keys 0..t, and the result is
 *           multiplied by sigmoid(gate).
 *   Side effect: k_cache[b, :, start_pos[b] + t] = the chunk's normalised,
 *   rotated keys and v_cache[b, :, start_pos[b] + t] = v, for t < Tq; other
 *   rows are neither written nor, past start_pos[b] + Tq, used (the kernel
 *   reads them but gives them zero weight and zeroes their values on chip, so
 *   a NaN there does not reach the output).
 *   The softmax relies on the cached keys obeying the norm bound of keys
 *   normalised with this k_w; a cache that breaks it so far that a softmax
 *   sum overflows leaves those rows undefined and q3a_last_device_error()
 *   returns Q3A_EINVAL.
 *   With every start_pos[b] = 0 this is q3a_gated_prefill_fill; with Tq = 1
 *   it computes what q3a_gated_decode computes.
 *   Requires 0 <= start_pos[b] and start_pos[b] + Tq <= S_max for every b,
 *   else Q3A_ERANGE with the caches untouched. B <= 2048, S_max <= 2^30,
 *   Hq + 2 Hkv <= 192, d = 256, d_rot a multiple of 16 up to 256; groupings
 *   as q3a_gated_prefill.
 *   workspace: at least q3a_gated_prefill_chunk_workspace_size() bytes,
 *   256-byte aligned, owned by the caller (normalised queries, error word).
 *   B == 0 or Tq == 0: returns Q3A_OK and launches nothing.
 * Source: "Chapter 20, Qwen3 and Qwen3.5" §20.3 (position counter, cached
 * keys then new ones, rectangular causal mask starting at pos_start; chunks
 * [0:2], [2:5], [5:6] against one forward) applied to the §20.4 gated layer.
 * ------------------------------------------------------------------------- */
size_t q3a_gated_prefill_chunk_workspace_size(int B, int Tq, int Hq, int Hkv, int d);

q3a_status q3a_gated_prefill_chunk(const q3a_bf16* qg, const q3a_bf16* k, const q3a_bf16* v,
                                   q3a_bf16* k_cache, q3a_bf16* v_cache,
                                   const int32_t* start_pos,
                                   const q3a_bf16* q_w, const q3a_bf16* k_w, q3a_bf16* out,
                                   int B, int Tq, int Hq, int Hkv, int d, int d_rot, int S_max,
                                   double theta, float eps,
                                   void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_gated_decode — one decode step of the gated global-attention layer of
 * Qwen3-Next / Qwen3.5 against a KV cache, appending the new token
 * ("Chapter 20, Qwen3 and Qwen3.5" §20.3 cache protocol, §20.4 layer).
 *
 *   qg      [B, Hq, 2d] bf16: per head, the query (first d) and the gate (last d).
 *   k_new, v_new [B, Hkv, d] bf16: the new token's projected key and value.
 *   k_cache, v_cache [B, Hkv, S_max, d] bf16, caller-owned: rows
 *           0..start_pos[b]-1 are read as stored (normalised and rotated by
 *           earlier calls with the same k_w, d_rot and theta); row start_pos[b]
 *           receives the new token's normalised, rotated key and its value.
 *   start_pos [B] int32 on the HOST: position of each sequence's new token.
 *   q_w, k_w [d] bf16 zero-centred norm weights (scale 1 + w).
 *   out     [B, Hq, d] bf16: sigmoid(gate) * softmax(q k^T / sqrt(d)) v.
 *   d = 256; d_rot a multiple of 16 in 0..256; Hq / Hkv any whole ratio up
 *   to 16 (above 16 returns Q3A_ENOTIMPL); B <= 2048; S_max <= 2^30.
 *   workspace: at least q3a_gated_decode_workspace_size() bytes, 256-byte
 *           aligned, caller-owned, not shared by concurrent calls.
 *   Every argument is checked before anything is written; a start_pos[b] < 0
 *   or >= S_max returns Q3A_ERANGE with the caches untouched.
 * ------------------------------------------------------------------------- */
size_t q3a_gated_decode_workspace_size(int B, int Hq, int Hkv, int d, int S_max);

q3a_status q3a_gated_decode(const q3a_bf16* qg, const q3a_bf16* k_new, const q3a_bf16* v_new,
                            q3a_bf16* k_cache, q3a_bf16* v_cache,
                            const int32_t* start_pos,
                            const q3a_bf16* q_w, const q3a_bf16* k_w,
                            q3a_bf16* out,
                            int B, int Hq, int Hkv, int d, int d_rot, int S_max,
                            double theta, float eps,
                            void* workspace, size_t ws_bytes, void* stream);

/* q3a_gated_decode_device_pos — q3a_gated_decode with start_pos [B] int32 in
 * DEVICE memory (4-byte aligned), for steps captured in a CUDA graph: the
 * positions are checked on the device by a one-block pre-pass; if any
 * start_pos[b] is < 0 or >= S_max nothing is written and
 * q3a_last_device_error() returns Q3A_ERANGE. No host read or
 * synchronisation happens in the call; every split up to S_max is launched
 * (those past a sequence's length exit at once). Host-checkable argument
 * errors return as for q3a_gated_decode. */
q3a_status q3a_gated_decode_device_pos(const q3a_bf16* qg, const q3a_bf16* k_new,
                                       const q3a_bf16* v_new,
                                       q3a_bf16* k_cache, q3a_bf16* v_cache,
                                       const int32_t* start_pos,
                                       const q3a_bf16* q_w, const q3a_bf16* k_w,
                                       q3a_bf16* out,
                                       int B, int Hq, int Hkv, int d, int d_rot, int S_max,
                                       double theta, float eps,
                                       void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_selftest_bounded_wait — a diagnostic: one block of 32 threads waits on
 * an mbarrier through the bounded-wait routine that every kernel of this
 * library uses, with a wait limit of `limit_cycles` SM cycles
 * (1 .. about 2 s of cycles). With arrive == 0 nothing arrives: the wait gives
 * up, writes its timeout code into the error word at the start of `workspace`
 * (>= 256 bytes, 16-byte aligned, device memory) and the kernel returns, so
 * q3a_last_device_error(workspace) then reports Q3A_ETIMEOUT; with arrive != 0
 * the barrier completes and the word stays zero. It lets a caller check, on
 * its own GPU, that a device-side wait that runs out is reported as an error
 * and leaves the context usable (the clear-error rule of "Chapter 20, Qwen3
 * and Qwen3.5" §20.9), without faulting or hanging the device.
 * Returns Q3A_EINVAL for a bad workspace or limit (nothing launched).
 * ------------------------------------------------------------------------- */
q3a_status q3a_selftest_bounded_wait(void* workspace, size_t ws_bytes, long long limit_cycles,
                                     int arrive, void* stream);

/* ---------------------------------------------------------------------------
 * q3a_last_device_error — reads, synchronously on `stream`, the error word
 * that the kernels of the last call which used `workspace` left in its first
 * bytes (prefill and decode workspaces both keep it at offset 0).
 * With workspace == NULL it reads the error word of q3a_decode_noalloc (in
 * that entry point's static array) on the current device.
 * Returns Q3A_OK when the word is zero, Q3A_ERANGE when the device-side
 * position check of q3a_decode_device_pos failed, Q3A_ETIMEOUT when a bounded
 * device wait gave up, Q3A_EINVAL when a chunk's
 * cached keys broke their norm precondition so far that a softmax sum
 * overflowed, Q3A_ECUDA if the read failed. The prologue of each prefill or
 * chunk call clears the word.
 * ------------------------------------------------------------------------- */
q3a_status q3a_last_device_error(const void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* Q3A_H_ */
