/*
 * dllm_cache.h -- C ABI of the per-layer, per-denoising-step cached attention of a
 * masked diffusion LLM, for NVIDIA B300 (sm_103a).
 *
 * One step of one layer (the pipeline of "Flash-dLLM: IO-aware KV caching and
 * parallel decoding", paragraph 2: QKV projection -> rotary embedding -> cache write
 * -> attention) runs as two kernels on the caller's stream:
 *
 *   1. a fused tcgen05/TMEM GEMM that projects the active rows, applies the rotary
 *      embedding at their absolute positions and scatter-writes K/V straight into the
 *      flat cache (the intermediates never round-trip through HBM);
 *   2. bidirectional (non-causal) attention of the step's query rows over every
 *      visible cache slot ("LaCache: Exact Caching and Precision-Adaptive Inference
 *      for Diffusion Large Language Models", technical summary, Problem Statement).
 *
 * Conventions shared by every call:
 *   - Every tensor argument is a DEVICE pointer owned by the caller, unless stated.
 *     All tensors are dense row-major with the layout given beside them; base
 *     addresses must be 16-byte aligned.
 *   - D = n_heads * head_dim.  "act" is the activation type: fp32 for a DLLM_F32
 *     cache, bf16 for DLLM_BF16 and DLLM_E4M3 caches.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and never synchronise, except dllm_cache_alloc/free/status.  A cache
 *     owns small workspaces (split-KV partials and their arrival counters, the drift
 *     test's partial sums and arrival counters), so calls on one cache must be ordered
 *     (one stream, or events between streams).
 *   - A cache lives on the device that was current when dllm_cache_alloc created it;
 *     every call that launches work on it must be made with that device current,
 *     else it returns DLLM_EINVAL and launches nothing.
 *   - Every call returns a dllm_status.  Argument errors are detected on the host
 *     before anything is launched and leave all buffers untouched.  Range errors in
 *     device-resident index data (a position outside [0, max_pos), too many draft
 *     rows for the tail, an unknown view tag) cannot be seen by the host: the kernel
 *     skips the offending row and sets a bit in the cache's device status word, which
 *     dllm_cache_status() returns.  A pipeline wait that exceeds its time limit
 *     (about one second) also sets a bit there and ends the kernel cleanly instead of
 *     hanging.
 *   - Nothing here falls back to the CPU.  Without a usable sm_103a device every
 *     call that launches work returns DLLM_ECUDA.
 */
#ifndef DLLM_CACHE_H
#define DLLM_CACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DLLM_OK = 0,
  DLLM_EINVAL = 1,       /* bad argument (shape, null pointer, alignment, dtype) */
  DLLM_EOOM = 2,         /* device allocation failed */
  DLLM_ECUDA = 3,        /* a CUDA runtime/driver call failed (no device, bad launch) */
  DLLM_EDEVICE = 4,      /* dllm_cache_status only: the device status word is non-zero */
  DLLM_EUNSUPPORTED = 5  /* valid but not supported by these kernels (e.g. head_dim) */
} dllm_status;

/* Bits of the device status word (see dllm_cache_status). */
#define DLLM_DEV_BAD_POSITION 0x1 /* a row's position is outside [0, max_pos) */
#define DLLM_DEV_BAD_VIEW 0x2     /* a view tag is not BASE/DRAFT/MASK */
#define DLLM_DEV_TAIL_FULL 0x4    /* more DRAFT rows in a sequence than tail_slots */
#define DLLM_DEV_TIMEOUT 0x8      /* a pipeline wait ran out of time; the kernel quit */
#define DLLM_DEV_BAD_INDEX 0x10   /* a top-k / drift index is outside [0, max_pos) */

/* Cache storage types. */
#define DLLM_F32 0  /* fp32 K/V, fp32 activations (SIMT fp32 kernels) */
#define DLLM_BF16 1 /* bf16 K/V, bf16 activations (tcgen05 kernels) */
#define DLLM_E4M3 2 /* FP8-e4m3 K/V with one fp32 scale per (slot, K|V, head), bf16 activations */

/* Row view tags for Flash-Verify ("Flash-dLLM ...", paragraph 3).  A BASE row is an
 * ordinary block token.  A search-set token appears twice: as a MASK row (its own
 * position/slot, filled with the mask embedding) and as a DRAFT row (same absolute
 * position for the rotary embedding, but written to a tail slot).  Visibility: key j
 * is visible to query q iff view(j) is SHARED (any slot not written by a MASK or DRAFT
 * row of this step), or view(j) == view(q), or (view(q) == BASE and view(j) == MASK).
 * The r-th DRAFT row of a sequence (in row order) writes tail slot max_pos + r. */
#define DLLM_VIEW_BASE 0
#define DLLM_VIEW_DRAFT 1
#define DLLM_VIEW_MASK 2

typedef struct dllm_cache dllm_cache; /* opaque; owns or wraps one flat K/V buffer */

typedef struct {
  int n_layers;      /* layers held by the cache (>= 1) */
  int batch;         /* sequences B (>= 1) */
  int max_pos;       /* regular slots per sequence = positions 0..max_pos-1 (>= 1) */
  int tail_slots;    /* extra slots per sequence for Flash-Verify draft views (>= 0) */
  int n_heads;       /* H (>= 1) */
  int head_dim;      /* hd: 128 for DLLM_BF16/DLLM_E4M3; a multiple of 4, <= 256, for DLLM_F32 */
  int kv_dtype;      /* DLLM_F32 | DLLM_BF16 | DLLM_E4M3 */
  double rope_theta; /* rotary base (> 0), e.g. 10000 or 500000 */
  void* external_buf;    /* optional caller device buffer of >= dllm_cache_bytes() bytes,
                            256-byte aligned; NULL = the library allocates and owns it */
  size_t external_bytes; /* size of external_buf */
} dllm_cache_desc;

/* Layout of the flat buffer, for callers that read or fill the cache directly.
 *   kv:    [n_layers][batch][max_pos + tail_slots][2 (K,V)][n_heads][head_dim],
 *          element type fp32 / bf16 / e4m3 per kv_dtype; K is stored after the
 *          rotary embedding.
 *   scale: (DLLM_E4M3 only, else NULL) fp32 [n_layers][batch][max_pos + tail_slots][2][n_heads];
 *          the stored value of element i is e4m3(code_i) * scale.                    */
typedef struct {
  void* kv;
  float* scale;
  size_t kv_bytes;
  size_t scale_bytes;
  size_t layer_elems; /* elements of kv per layer */
  int slots;          /* max_pos + tail_slots */
  int elem_bytes;     /* 4, 2 or 1 */
} dllm_cache_layout;

/* Bytes of the flat K/V (+ scale) buffer that `desc` needs; 0 if `desc` is invalid.
 * Host only, no CUDA call.  Flash-dLLM paragraph 5: one flat, preallocated cache. */
size_t dllm_cache_bytes(const dllm_cache_desc* desc);

/* Create a cache for `desc` on the current device.  Allocates (or wraps
 * external_buf for) the K/V buffer, plus small library-owned buffers: the rotary
 * cos/sin table (fp32 from fp64, [max_pos][head_dim/2]), the device status word, a
 * split-KV workspace of a few MB with its arrival counts, and the drift test's partial
 * sums.  The K/V contents are left uninitialised.
 * Returns DLLM_EINVAL for a bad desc, DLLM_EUNSUPPORTED for an unsupported head_dim,
 * DLLM_EOOM / DLLM_ECUDA on device failure; *out is NULL on error. */
int dllm_cache_alloc(const dllm_cache_desc* desc, dllm_cache** out);

/* Release the cache and every library-owned buffer (not external_buf).  Waits for the
 * device to finish.  NULL is accepted. */
int dllm_cache_free(dllm_cache* cache);

/* Fill *out with the buffer layout of `cache`. */
int dllm_cache_get_layout(const dllm_cache* cache, dllm_cache_layout* out);

/* One denoising step of one layer (Flash-dLLM paragraph 2; LaCache Methodology 1:
 * the cached state is the projected, rotary-embedded K/V of each token).
 *
 *   layer         0 <= layer < n_layers
 *   x             act [batch][n_tok][D]: hidden states of the step's query rows
 *   w_qkv         act [3D][D]: row n holds output feature n; the mathematical projection
 *                 is [q|k|v] = x . W with W = transpose(w_qkv) of shape [D][3D]; features 0..D-1
 *                 are Q, D..2D-1 K, 2D..3D-1 V, head-major (h*head_dim + i); no bias
 *   positions     int32 [batch][n_tok]: absolute position of each row (rotary angle and,
 *                 for BASE/MASK rows, the cache slot); must be distinct within a
 *                 sequence among non-DRAFT rows
 *   view          uint8 [batch][n_tok] DLLM_VIEW_* tags, or NULL (all BASE, and the tail
 *                 slots are not attended)
 *   n_tok         query rows per sequence (>= 0)
 *   out           act [batch][n_tok][D]: attention output per head, heads concatenated
 *                 (before any output projection).  Also used as scratch for the rotated
 *                 Q during the call, so it must not alias x.
 *   kv_x          act [batch][n_kv][D] or NULL: K/V-only rows (no query, no output)
 *   kv_positions  int32 [batch][n_kv]: their absolute positions
 *   n_kv          K/V-only rows per sequence (>= 0)
 *   probe_kv      act [batch][n_kv][2][D] or NULL.  NULL: the K/V-only rows are written
 *                 into the cache at their positions (a refresh of those slots).  Non-NULL:
 *                 the cache is left alone and their rotated K (index 0) and V (index 1)
 *                 go here instead (probes for dllm_kv_drift).
 *   stream        cudaStream_t
 *
 * Order of effects: all cache writes of the step (K/V-only rows and query rows) happen
 * before any attention read, so the block attends to its own fresh K/V.  Each query
 * row then attends, per head, over slots 0..max_pos-1 and over the tail slots written
 * by this step's DRAFT rows, with the visibility rule given above, scores scaled by
 * 1/sqrt(head_dim) and an fp32 softmax. */
int dllm_cache_step(dllm_cache* cache, int layer,
                    const void* x, const void* w_qkv,
                    const int32_t* positions, const uint8_t* view, int n_tok,
                    void* out,
                    const void* kv_x, const int32_t* kv_positions, int n_kv,
                    void* probe_kv,
                    void* stream);

/* The two halves of dllm_cache_step, for callers that schedule or time them apart;
 * dllm_cache_step(...) is exactly dllm_cache_project(...) followed by
 * dllm_cache_attend(...) on the same stream with the same arguments.
 *
 * dllm_cache_project: the fused projection + rotary embedding + cache (or probe)
 *   write of dllm_cache_step; the rotated Q of the query rows is left in `out`
 *   (act [batch][n_tok][D]).  Arguments as for dllm_cache_step.
 * dllm_cache_attend: the attention half.  `out` must hold the rotated Q that
 *   dllm_cache_project left for the same positions / view / n_tok; it is overwritten
 *   with the attention output.  Errors as for dllm_cache_step.  How the work is split
 *   over the GPU (whole (sequence, head) units, keys split over CTAs, the partial
 *   states merged in the kernel or by a second launch) depends only on the shapes, so
 *   repeated calls on the same inputs give bit-identical outputs. */
int dllm_cache_project(dllm_cache* cache, int layer,
                       const void* x, const void* w_qkv,
                       const int32_t* positions, const uint8_t* view, int n_tok,
                       void* out,
                       const void* kv_x, const int32_t* kv_positions, int n_kv,
                       void* probe_kv,
                       void* stream);
int dllm_cache_attend(dllm_cache* cache, int layer,
                      const int32_t* positions, const uint8_t* view, int n_tok,
                      void* out, void* stream);

/* Attention over a ragged batch ("Elastic-Cache", Deployment notes: a batch built from
 * sequences of different lengths): as dllm_cache_attend without Flash-Verify views, but
 * sequence b attends only to its first key_len[b] slots (clamped to [0, max_pos]); cache
 * tiles past that length are not read.  A row whose sequence has key_len 0 gets zeros.
 *
 *   key_len   int32 [batch], device
 * DLLM_BF16 and DLLM_E4M3 caches (DLLM_EUNSUPPORTED for DLLM_F32). */
int dllm_cache_attend_ragged(dllm_cache* cache, int layer, const int32_t* positions, int n_tok,
                             const int32_t* key_len, void* out, void* stream);

/* Partial attention state over a slot range ("LaCache ...", Methodology 1, FACache: the
 * running maximum m, the normaliser l and the unnormalised accumulator O of online
 * softmax are cached for key blocks that do not change and combined with those of the
 * blocks that do, instead of re-reading the unchanged keys).  For every query row t,
 * head h and the keys j in [slot_lo, slot_hi):
 *   s_j = (q . k_j) / sqrt(hd) * log2(e),  m = max_j s_j,  l = sum_j 2^(s_j - m),
 *   O[i] = sum_j 2^(s_j - m) v_j[i]
 * (m = -inf, l = 0, O = 0 when the range holds no key).
 *
 *   q         bf16 [batch][n_tok][D]: rotated Q (dllm_cache_project's `out`); not modified,
 *             so several ranges can be evaluated from the same q
 *   state     fp32 [batch][n_tok][n_heads][head_dim + 2] out: O, then m, then l; 16-byte
 *             aligned
 *   0 <= slot_lo < slot_hi <= max_pos (regular slots; no Flash-Verify views)
 * DLLM_BF16 and DLLM_E4M3 caches. */
int dllm_cache_attend_partial(dllm_cache* cache, int layer, const int32_t* positions, int n_tok, const void* q,
                              int slot_lo, int slot_hi, float* state, void* stream);

/* FACache reuse in one call ("LaCache ...", Methodology 1, FACache): attention of the
 * query rows over the slots [slot_lo, slot_hi) that changed, merged in the same kernel
 * with a state the caller cached for all the other keys (dllm_cache_attend_partial
 * output of an earlier call, for the same rows and the same q), written as the
 * normalised output
 *   out = (2^(m_r - M) O_r + 2^(m_c - M) O_c) / (2^(m_r - M) l_r + 2^(m_c - M) l_c),
 * M = max(m_r, m_c), r = this range, c = the cached state (0 where both are empty).
 * Only the changed slots are read: a step that rewrote a few tiles reads those tiles,
 * not the whole cache.  The result equals the attention over both key sets when the
 * cached state's keys and q have not changed since it was computed; the caller decides
 * that.
 *
 *   q         bf16 [batch][n_tok][D]: rotated Q (not modified)
 *   state     fp32 [batch][n_tok][n_heads][head_dim + 2], 16-byte aligned: the cached state
 *   out       bf16 [batch][n_tok][D] out; must not alias q or state
 *   0 <= slot_lo < slot_hi <= max_pos (regular slots; no Flash-Verify views)
 * DLLM_BF16 and DLLM_E4M3 caches (DLLM_EUNSUPPORTED for DLLM_F32). */
int dllm_cache_attend_with_state(dllm_cache* cache, int layer, const int32_t* positions, int n_tok, const void* q,
                                 int slot_lo, int slot_hi, const float* state, void* out, void* stream);

/* Combine two partial states of the same rows (the key ranges must not overlap):
 *   M = max(m_a, m_b), w_a = 2^(m_a - M), w_b = 2^(m_b - M),
 *   O = w_a O_a + w_b O_b, l = w_a l_a + w_b l_b,
 * and write the attention output out = O / l (bf16 [batch][n_tok][n_heads * head_dim],
 * 0 where l = 0) and/or the combined state (same layout as the inputs; may alias
 * neither input).  Either output may be NULL, not both.  head_dim must be 128
 * (DLLM_EUNSUPPORTED otherwise).  States and `out` 16-byte aligned, batch * n_tok *
 * n_heads below 2^31 (DLLM_EINVAL otherwise). */
int dllm_attend_merge(const float* state_a, const float* state_b, int batch, int n_tok, int n_heads, int head_dim,
                      void* out, float* state_out, void* stream);

/* Attention mass of this step per cached position ("Flash-dLLM ...", paragraph 4 tracks
 * the most-attended tokens; "Elastic-Cache", Core idea tests the previous step's
 * most-attended tokens).  For sequence b and regular slot j < max_pos:
 *   mass[b][j] = sum over heads h and query rows t of softmax_j(q_{t,h} . k_{j,h} / sqrt(hd)),
 * with the same visibility rule as the attention (Flash-Verify views included; weights
 * of draft-view tail slots count in each softmax but are not reported).  The result is
 * what dllm_kv_topk reads in the next step.
 *
 *   q         bf16 [batch][n_tok][D]: the rotated Q that dllm_cache_project leaves in its
 *             `out` (call this before dllm_cache_attend overwrites it)
 *   mass      fp32 [batch][max_pos] out (zeroed and filled by the call)
 * Other arguments as for dllm_cache_attend.  DLLM_BF16 and DLLM_E4M3 caches (an e4m3
 * key is its codes times its group scale, as in the attention); DLLM_EUNSUPPORTED for
 * DLLM_F32.  Reads the layer's K twice per (sequence, head) unit; the second read
 * mostly hits L2. */
int dllm_attention_mass(dllm_cache* cache, int layer, const int32_t* positions, const uint8_t* view, int n_tok,
                        const void* q, float* mass, void* stream);

/* The conventional pipeline, for comparison with the fused step ("Flash-dLLM ...",
 * paragraph 2: QKV projection, rotary embedding, cache write and attention as four
 * kernels, each writing its intermediates to HBM for the next one).  Same arguments and
 * effects as dllm_cache_step, plus a caller-owned device workspace that receives the
 * projection output: [batch][n_tok][3D] for the query rows, then (at the next 256-byte
 * boundary) [batch][n_kv][2D] for the K/V-only rows.  The workspace holds bf16 values
 * for DLLM_BF16 caches, which are rounded to bf16 before the rotation and the cache
 * store (results differ from dllm_cache_step by that extra rounding), and fp32 values
 * for DLLM_E4M3 caches, which are quantised from the unrounded rotated value as
 * dllm_cache_step does (the codes differ only where fp32 sums in another order cross a
 * rounding boundary).
 *
 *   workspace        device buffer of >= dllm_unfused_workspace_bytes() bytes, 256-byte
 *                    aligned (DLLM_EINVAL otherwise)
 * Returns DLLM_EUNSUPPORTED for DLLM_F32 caches. */
size_t dllm_unfused_workspace_bytes(const dllm_cache* cache, int n_tok, int n_kv);
int dllm_cache_step_unfused(dllm_cache* cache, int layer,
                            const void* x, const void* w_qkv,
                            const int32_t* positions, const uint8_t* view, int n_tok,
                            void* out,
                            const void* kv_x, const int32_t* kv_positions, int n_kv,
                            void* probe_kv, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Top-k most-attended positions ("Flash-dLLM ...", paragraph 4: a fixed budget of the
 * top 32 most-attended tokens; "Elastic-Cache", Core idea: the previous step's
 * most-attended tokens).
 *
 *   mass      fp32 [batch][n_pos]: previous-step attention mass per position (finite)
 *   block_lo  int32 [batch]: first position of each sequence's active block; positions
 *             block_lo .. block_lo+block_len-1 are not candidates
 *   idx       int32 [batch][k] out: candidate positions ordered by mass descending, ties
 *             to the lower position; k <= n_pos - block_len, n_pos <= 16384 */
int dllm_kv_topk(const float* mass, int batch, int n_pos, const int32_t* block_lo, int block_len,
                 int k, int32_t* idx, void* stream);

/* Hidden states of the tracked tokens ("Elastic-Cache", Core idea: the drift test
 * recomputes K/V of the previous step's most-attended tokens from this step's states;
 * "Flash-dLLM ...", paragraph 4: 32 tracked tokens): a row gather on the device, so
 * that top-k, gather, probe projection and drift test run back to back on the stream
 * without a host round trip.
 *
 *   x_all     act [batch][n_pos][D]: this step's hidden states of every position
 *   idx       int32 [batch][k]: positions to gather (dllm_kv_topk's output)
 *   x_rows    act [batch][k][D] out: x_rows[b][j] = x_all[b][idx[b][j]]
 * batch and D are the cache's (the cache supplies them and the status word); act as
 * for dllm_cache_step.  A position outside [0, n_pos) gives a zero row and sets
 * DLLM_DEV_BAD_INDEX.  x_all and x_rows 16-byte aligned, k >= 1, n_pos >= 1. */
int dllm_gather_rows(dllm_cache* cache, const void* x_all, int n_pos, const int32_t* idx, int k, void* x_rows,
                     void* stream);

/* dllm_kv_topk followed by dllm_gather_rows of the selected positions, with the batch
 * taken from the cache: for k <= 32 one launch, whose block per sequence copies the
 * rows right after it has selected them (for larger k, the two launches).
 *   mass, n_pos, block_lo, block_len, k, idx   as for dllm_kv_topk (batch = the cache's)
 *   x_all, x_rows                             as for dllm_gather_rows
 * Same results as the two calls; argument errors as for either. */
int dllm_kv_topk_gather(dllm_cache* cache, const float* mass, int n_pos, const int32_t* block_lo, int block_len,
                        int k, int32_t* idx, const void* x_all, void* x_rows, void* stream);

/* Attention-aware drift test ("Elastic-Cache", Core idea and Algorithm knobs).
 *
 *   idx       int32 [batch][k]: tracked positions (slots) in `layer`
 *   probe_kv  act [batch][k][2][D]: freshly computed K/V of the same tokens
 *             (dllm_cache_step with probe_kv)
 *   cos       fp32 [batch][k][2] out: cosine similarity between cached and probe
 *             K (index 0) and V (index 1), each over the full D-vector of the token
 *             (FP8 caches are dequantised first)
 *   refresh   int32 [batch] out, or NULL: 1 where min over that sequence's cos < gamma
 *             (the layer's cache has drifted and deeper layers should be recomputed),
 *             else 0 */
int dllm_kv_drift(const dllm_cache* cache, int layer, const int32_t* idx, int k,
                  const void* probe_kv, float gamma, float* cos, int32_t* refresh, void* stream);

/* The projection half with the drift test fused into it ("Elastic-Cache", Core idea and
 * Algorithm knobs; "Flash-dLLM ...", paragraph 4).  Same effects as
 *   dllm_cache_project(cache, layer, x, w_qkv, positions, view, n_tok, out,
 *                      kv_x, idx, k, probe, stream)
 *   dllm_kv_drift(cache, layer, idx, k, probe, gamma, cos, refresh, stream)
 * without the probe buffer: the projection's epilogue compares each tracked token's
 * recomputed K and V (fp32, before any rounding) with the cached ones at its position
 * and writes only the cosines and the flags, so the probe K/V never go to HBM.
 *
 *   kv_x      act [batch][k][D]: this step's hidden states of the tracked tokens
 *   idx       int32 [batch][k]: their positions, which are also the compared slots; they
 *             must not be slots that this call's query rows write (dllm_kv_topk leaves
 *             the active block out), else a cosine may see either the old or the new K/V
 *   k         tracked tokens per sequence, 1 <= k <= 256 (DLLM_EUNSUPPORTED above)
 *   gamma, cos, refresh   as for dllm_kv_drift
 * Other arguments as for dllm_cache_project.  DLLM_BF16 and DLLM_E4M3 caches
 * (DLLM_EUNSUPPORTED for DLLM_F32).  A position outside [0, max_pos) gives NaN cosines
 * for that token (the flag's minimum skips them) and sets DLLM_DEV_BAD_POSITION.  Uses
 * a small workspace of the cache, so calls on one cache must be ordered. */
int dllm_cache_project_drift(dllm_cache* cache, int layer, const void* x, const void* w_qkv,
                             const int32_t* positions, const uint8_t* view, int n_tok, void* out,
                             const void* kv_x, const int32_t* idx, int k, float gamma,
                             float* cos, int32_t* refresh, void* stream);

/* dllm_cache_project_drift followed by dllm_cache_attend on the same stream: one
 * denoising step of one layer with the drift test of its tracked tokens. */
int dllm_cache_step_drift(dllm_cache* cache, int layer, const void* x, const void* w_qkv,
                          const int32_t* positions, const uint8_t* view, int n_tok, void* out,
                          const void* kv_x, const int32_t* idx, int k, float gamma,
                          float* cos, int32_t* refresh, void* stream);

/* One denoising step over layers 0 .. n_layers-1 of the cache with the depth-wise
 * refresh of "Elastic-Cache ..." (Core idea: when the drift test of the most-attended
 * tokens fails at layer l, the layers after l are recomputed, shallow layers keep their
 * caches; Algorithm knobs: threshold gamma, window size beta).  Per layer l, in order,
 * on one stream and without host synchronisation:
 *   1. (l > 0) for every sequence b with flags[j][b] set for some j < l: K and V of
 *      every regular slot 0 .. max_pos-1 are recomputed from x_all[l] (fused
 *      projection, rotary embedding, cache store); other sequences' slots are untouched;
 *   2. idx = the k most-attended positions of mass[l] outside the window (dllm_kv_topk);
 *   3. the window rows win_lo[b] .. win_lo[b]+beta-1 of x_all[l] are projected (Q, K, V)
 *      and their K/V written to their slots; the tracked rows x_all[l][b][idx] are
 *      projected and compared with their cached K/V: the drift test -> cos[l],
 *      flags[l] (dllm_cache_project_drift);
 *   4. (mass_out != NULL) the window's attention mass per slot -> mass_out[l]
 *      (dllm_attention_mass), the next step's mass input;
 *   5. the window attends over the cache -> out[l] (dllm_cache_attend).
 * A layer whose own test fails is not recomputed in this step; the layers after it are.
 *
 *   x_all       host array of n_layers device pointers, each bf16 [batch][max_pos][D]:
 *               this step's hidden states of every position at that layer
 *   w_qkv       host array of n_layers device pointers, bf16 [3D][D] each
 *   win_lo      int32 [batch] device: first position of each sequence's window;
 *               0 <= win_lo[b] <= max_pos - beta (else the window's rows are zero and
 *               DLLM_DEV_BAD_POSITION is raised)
 *   mass        fp32 [n_layers][batch][max_pos] device: previous step's attention mass
 *   k, gamma    tracked tokens per sequence (1 <= k <= max_pos - beta, k <= 256), drift
 *               threshold
 *   out         bf16 [n_layers][batch][beta][D] device out: attention output per layer
 *   cos         fp32 [n_layers][batch][k][2] device out
 *   flags       int32 [n_layers][batch] device out: the drift test's refresh flags
 *   mass_out    fp32 [n_layers][batch][max_pos] device out, or NULL
 *   workspace   device, 256-byte aligned, >= dllm_elastic_workspace_bytes(cache, beta, k)
 * Uses the cache's own workspaces: calls on one cache must be ordered.  DLLM_F32 caches:
 * DLLM_EUNSUPPORTED.  max_pos <= 16384. */
size_t dllm_elastic_workspace_bytes(const dllm_cache* cache, int beta, int k);
int dllm_elastic_step(dllm_cache* cache, int n_layers, const void* const* x_all, const void* const* w_qkv,
                      const int32_t* win_lo, int beta, const float* mass, int k, float gamma,
                      void* out, float* cos, int32_t* flags, float* mass_out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Scratch capacity of dllm_cache_attend_noalloc, in bytes (16 MiB). */
#define DLLM_NOALLOC_SCRATCH_BYTES (16u << 20)

/* dllm_cache_attend for callers that cannot allocate device memory.  The pages have
 * no counterpart to this call; it exists for how the library is hosted, not for the
 * method.  Some callers must not call cudaMalloc at all: a serving engine that has
 * already handed its whole device memory budget to its own pool (a new allocation
 * would fail or break that budget), or a latency-critical decode loop that cannot
 * take the device-wide synchronisation cudaMalloc may cause.  This call allocates
 * nothing: when the work is split over keys, the partial softmax states go to one
 * fixed array of DLLM_NOALLOC_SCRATCH_BYTES in the library's own device memory, which
 * every device that loads the library holds until the process exits.
 *
 * Arguments, results and errors are those of dllm_cache_attend, plus:
 *   - DLLM_EUNSUPPORTED when the split partial states of this call would need more
 *     than DLLM_NOALLOC_SCRATCH_BYTES (one slot of 64 query rows * 130 floats per
 *     piece); nothing is launched then.  Both entry points cut units into pieces only
 *     as far as the pieces' states fit this size, so with the current kernels the case
 *     does not arise.  The arrival counts that say which CTA completes a split unit are
 *     the cache's own (allocated with it, back at zero after every call).
 *   - The first call on each device looks up the device address of that array (with
 *     the device current) and remembers it; make this first call before any stream
 *     capture begins.  cudaDeviceReset() discards the array with the rest of the
 *     device's memory and leaves the remembered address stale: do not call this entry
 *     point on a device after resetting it.
 *   - It launches exactly the kernels dllm_cache_attend launches, with the same work
 *     split, so its output is bit-identical to dllm_cache_attend's.
 *   - Every call on a device shares the same array and leaves its contents behind.
 *     Nothing in it needs to start at zero.  Calls whose kernels overlap on the GPU
 *     (different streams without ordering between them) race on it and give wrong
 *     results; order them on one stream or with events. */
int dllm_cache_attend_noalloc(dllm_cache* cache, int layer,
                              const int32_t* positions, const uint8_t* view, int n_tok,
                              void* out, void* stream);

/* Self-test of the failure handling: launches one CTA that waits, with the library's
 * bounded wait, on an mbarrier that nothing arrives at.  The wait gives up after its
 * time limit (about one second), the kernel sets DLLM_DEV_TIMEOUT in the cache's status
 * word and ends; dllm_cache_status() then returns DLLM_EDEVICE with that bit and clears
 * it, and the context stays usable.  Not part of the pages' method. */
int dllm_selftest_wait_timeout(dllm_cache* cache, void* stream);

/* Self-test of the allocation-failure paths: the nth device allocation the library
 * makes from now on (1 = the next one) fails as if the device were out of memory; 0
 * cancels a pending failure.  Process-wide; allocations by the caller are unaffected.
 * dllm_cache_alloc then returns DLLM_EOOM with *out NULL, having released whatever it
 * had allocated before the failure.  DLLM_EINVAL for nth < 0.  Host only, no CUDA call.
 * Not part of the pages' method. */
int dllm_selftest_fail_alloc(int nth);

/* Synchronise the device, read the cache's device status word into *device_bits (may
 * be NULL) and clear it.  Returns DLLM_EDEVICE if any bit was set, else DLLM_OK.  With
 * DLLM_DEV_TIMEOUT set it also zeroes the cache's arrival counters (drift test, split
 * attention), which a kernel that gave up may have left part-way. */
int dllm_cache_status(dllm_cache* cache, int* device_bits);

/* Static, human-readable name of a dllm_status. */
const char* dllm_strerror(int status);

/* Page-locked HOST memory for a step's inputs and results when they live on the host
 * (a serving loop that receives hidden states and returns outputs): `bytes` bytes
 * from the CUDA runtime's own page-locked allocator, which the GPU's copy engines read
 * and write directly, at the link rate, with no staging copy.  Not part of the pages'
 * method: the end-to-end path's host-side buffers.
 *   - *out receives the host address (16-byte aligned or better), or NULL on error or
 *     when bytes == 0 (which returns DLLM_OK).  The contents are uninitialised.
 *   - The caller owns the block and releases it with dllm_host_free; it stays valid for
 *     every device and context of the process until then.
 *   - Errors: DLLM_EINVAL if out is NULL; DLLM_EOOM if the memory cannot be locked;
 *     DLLM_ECUDA if no CUDA device is usable.  Synchronous; launches nothing. */
int dllm_host_alloc(size_t bytes, void** out);

/* Release a block from dllm_host_alloc (NULL: no-op, DLLM_OK).  The caller first makes
 * sure no copy that reads or writes it is still pending.  Returns DLLM_ECUDA if the
 * runtime rejects the address (not a dllm_host_alloc block). */
int dllm_host_free(void* ptr);

/* Copy `bytes` bytes of host memory from src to dst (normally a dllm_host_alloc block
 * that a host-to-device copy will read next) with streaming stores, which leave no
 * dirty copies of dst in the CPU caches.  A device copy that reads host lines still
 * dirty in those caches has to fetch each one out of them, and on the B300 hosts
 * measured that cut host-to-device copies from about 54 GB/s to about 12 GB/s; a
 * buffer written with this call is read at the full rate.  Not part of the pages'
 * method: staging of the end-to-end path.
 *   - Host pointers, any alignment; the ranges must not overlap (DLLM_EINVAL), nor
 *     may dst or src be NULL unless bytes == 0 (which does nothing, DLLM_OK).
 *   - Synchronous, on the calling thread; no CUDA call, no GPU needed.  The result is
 *     a plain byte copy (memcpy semantics). */
int dllm_host_stage(void* dst, const void* src, size_t bytes);

#ifdef __cplusplus
}
#endif
#endif /* DLLM_CACHE_H */
