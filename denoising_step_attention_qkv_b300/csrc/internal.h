// Host/device shared definitions of the library (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "../../include/dllm_cache.h"

struct dllm_cache {
  dllm_cache_desc desc;
  int device;
  int sm_count;
  int pair_clusters;  // clusters of two projection CTAs resident at once (0 = none)
  int* drift_cnt;     // [batch] block arrivals of dllm_kv_drift; zero between calls
  // Fused drift test (dllm_cache_project_drift), zero between calls: per tracked row
  // partial sums [batch * kMaxDriftRows][2 (K,V)][3 (dot, |cache|^2, |probe|^2)].
  float* drift_acc;
  void* kv;
  float* scale;
  bool owns_kv;
  size_t kv_bytes, scale_bytes;
  size_t layer_elems;   // K/V elements per layer
  size_t layer_scales;  // scales per layer (e4m3)
  int slots;            // max_pos + tail_slots
  int elem_bytes;
  float2* rope;  // [max_pos][head_dim/2] (cos, sin), fp32 rounded from fp64
  int* status;   // device status word
  float* ws;     // split-KV partials
  size_t ws_floats;
  int* merge_cnt;  // [2 * sm_count] arrival counts of the tail units' pieces; zero between calls
  size_t drift_acc_bytes;
};

namespace dllm {

// Raise `kernel`'s dynamic shared-memory limit to at least `bytes` on the current
// device, calling the driver only the first time (per device and kernel) a larger size
// is needed, so that launches (and stream capture) do no extra driver work.
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

// Programmatic dependent launch.  A kernel launched this way may start (its prologue:
// barrier setup, TMEM allocation, descriptor prefetch) while the previous kernel on the
// stream is still running; each such kernel lets its own dependents launch early
// (griddepcontrol.launch_dependents) and, in every thread, waits for the previous grid
// to complete (griddepcontrol.wait) before it reads or writes anything that grid may
// touch.  Since every CTA passes that wait before it exits, completion stays ordered
// along the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kHd = 128;         // head_dim of the tensor-core path
constexpr int kMaxDriftRows = 256;  // tracked rows per sequence of the fused drift test
constexpr int kQChunk = 64;      // query rows per attention work unit (tensor-core path)
constexpr int kKeyTile = 128;    // keys per attention tile
constexpr int kMaxPieces = 4;    // pieces a tail unit of the attention may be cut into

// ---------------------------------------------------------------- fused projection
struct ProjParams {
  int D, H;
  int n_tok, n_kv;    // rows per sequence: query rows, K/V-only rows
  int m_q, m_kv;      // total rows
  int mt_q, mt_kv;    // 128-row tiles
  int nt_q, nt_kv;    // column tiles per row tile (3D/BN, 2D/BN)
  int tiles_q, tiles_total;
  int whole_items;    // tiles computed whole (the first ones)
  int items_total;    // whole_items + 2 * (tiles_total - whole_items): the rest in 128-column halves
  int pmt_q, pmt_kv;  // CTA-pair kernel: 256-row tiles of the query rows, of the K/V-only rows
  int k_blocks;       // D / 64
  int m_fastest;      // tile raster: row tiles vary fastest
  const int32_t* positions;
  const uint8_t* view;
  const int32_t* kv_positions;  // [m_kv], or null: row i of a sequence is position i
  // Optional selection of the K/V-only rows by sequence: rows of sequence b are computed
  // and stored only when kv_seq_flags[j * batch + b] != 0 for some j < n_flag_sets
  // (device flags, e.g. the drift test's refresh flags of the layers above).
  const int32_t* kv_seq_flags;
  int n_flag_sets, batch;
  void* q_out;        // act [m_q][D]
  void* cache_kv;     // this layer: [B][slots][2][H][hd]
  float* cache_scale; // this layer: [B][slots][2][H] (e4m3)
  void* probe;        // act [m_kv][2][D] or null
  int kv_dtype;
  int max_pos, tail, slots;
  const float2* rope;
  int* status;
  // Unfused pipeline only (else null): the GEMM stores its plain output here,
  // [m_q][3D] for query rows and [m_kv][2D] (K|V) for K/V-only rows, with no rotation;
  // fp32 when raw_f32 (e4m3 caches, which quantise the unrounded rotated value), else bf16.
  void* raw_q;
  void* raw_kv;
  bool raw_f32;
  // Fused drift test (else drift_acc is null): the K/V-only rows are probes, compared in
  // the epilogue with the cached K/V at their positions instead of being stored; the
  // epilogue adds each row's dot product and squared norms into drift_acc, and
  // launch_drift_finalize (after the projection) writes the cosines drift_cos[m][2] (K, V)
  // and drift_refresh[b] = (min cosine < drift_gamma), if not null.
  float* drift_acc;   // [m_kv][2][3], zero on entry and on exit
  float* drift_cos;
  int32_t* drift_refresh;
  float drift_gamma;
};

// ------------------------------------------------------------------------ attention
struct AttnParams {
  int B, H, D, n_tok;
  int max_pos, tail, slots;
  int nq_pad;        // query columns per unit (multiple of 16, <= kQChunk)
  int n_qchunks;
  int key_tiles;     // 128-key tiles covering the attended slot range
  int n_splits, tiles_per_split;
  int units;         // B * H * n_qchunks * n_splits
  const uint8_t* view;
  const int32_t* positions;
  void* out;         // act [B][n_tok][D]: rotated Q in, attention output out
  float* ws;         // split partials: [units][nq_pad][hd] O, then [units][nq_pad][2] (m, l)
  float scale_log2;  // log2(e) / sqrt(hd)
  const float* kv_scale;  // this layer, e4m3 only
  int kv_dtype;
  // Key range (regular slots only; the defaults cover every slot): keys j with
  // key_lo <= j < min(key_hi, key_len[b]) are attended.  tile_lo = key_lo / 128; the
  // units cover key_tiles tiles from there.  key_len (device, [B]) or null.
  int key_lo, key_hi, tile_lo;
  const int32_t* key_len;
  bool ranged;       // key_lo > 0, key_hi < max_pos or key_len given
  // Partial-state output instead of `out` (no key splits then):
  // fp32 [B][n_tok][H][hd + 2] = (unnormalised O, m, l), m in base-2 units.
  float* state;
  // A cached state of the keys outside the range, same layout (no key splits then): the
  // finish merges it with the range's and writes the normalised output to `out`.
  const float* state_in;
  // Balanced schedule (tail_pieces > 0; n_splits = 1): dp_waves rounds of whole units
  // over the grid, then the last tail_units units (fewer than the grid) cut into
  // tail_pieces pieces of piece_tiles key tiles; the CTA that completes a tail unit
  // merges its pieces' partial states (ws: tail_units * tail_pieces slots of kQChunk rows,
  // O then (m, l)) into the output.  merge_cnt: [2 * tail_units] arrival counts, zero on
  // entry and on exit.
  int dp_waves, tail_units, tail_pieces, piece_tiles;
  int* merge_cnt;
  // Rows loaded of a key tile that runs past the sequence's slots (a multiple of 8,
  // through a tensor map with that box height); 0: every tile loads 128 rows.
  int tail_rows;
  int* status;
};

// Launchers (return a cudaError_t cast to int, 0 on success).
int launch_proj_tc(const ProjParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_xkv,
                   const CUtensorMap& tm_w, const CUtensorMap& tm_w_half, int bn, int grid, cudaStream_t s);
// CTA-pair variant (256 x 256 output tiles on two SMs, cta_group::2); grid = 2 x pairs.
// tm_w / tm_w_half: W boxes of 128 / 64 rows (each CTA's half of a 256 / 128-wide tile).
int launch_proj_pair(const ProjParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_xkv,
                     const CUtensorMap& tm_w, const CUtensorMap& tm_w_half, int grid, cudaStream_t s);
int proj_pair_max_clusters(int* clusters);
// The fused drift test's cosines and refresh flags from the partial sums (one block per
// sequence); launched after the projection on the same stream.
int launch_drift_finalize(const ProjParams& p, cudaStream_t s);
// tm_kv_tail: the same cache with boxes of tail_rows rows, for a tile that runs past the
// sequence's slots (used only when p.tail_rows != 0).
int launch_attn_tc(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                   const CUtensorMap& tm_kv_tail, int grid, cudaStream_t s);
int launch_attn_combine(const AttnParams& p, cudaStream_t s);
// Merge two partial softmax states (rows x heads, [hd + 2] each) into a normalised bf16
// output and/or a merged state.
int launch_state_merge(const float* a, const float* b, int rows, int H, void* out, float* state_out, cudaStream_t s);
int launch_attn_mass(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv, float* mass, int grid,
                     cudaStream_t s);

int launch_proj_f32(const ProjParams& p, const float* x, const float* xkv, const float* w, int hd,
                    cudaStream_t s);
int launch_attn_f32(const AttnParams& p, const float* kv_layer, int hd, cudaStream_t s);

int launch_topk(const float* mass, int batch, int n_pos, const int32_t* block_lo, int block_len, int k,
                int32_t* idx, cudaStream_t s);
// k <= 32: the top-k and, in the same launch, the selected rows (row_vecs 16-byte
// vectors each) of x_all[batch][n_pos] copied into x_rows[batch][k].
int launch_topk_gather(const float* mass, int batch, int n_pos, const int32_t* block_lo, int block_len, int k,
                       int32_t* idx, const void* x_all, int row_vecs, void* x_rows, cudaStream_t s);
int launch_drift(const void* kv_layer, const float* scale_layer, int kv_dtype, int B, int slots, int max_pos,
                 int H, int hd, const int32_t* idx, int k, const void* probe, float gamma, float* cos,
                 int32_t* refresh, int* counters, int sm_count, int* status, cudaStream_t s);

// The conventional pipeline's separate stages (unfused comparison): rotate Q (into
// q_out) and K (in place) of the raw GEMM output, then write K/V to their slots.
int launch_rope_rows(const ProjParams& p, cudaStream_t s);
int launch_cache_write(const ProjParams& p, cudaStream_t s);

// Multi-layer refresh step: gather one layer's window rows (and their positions) and
// tracked rows from its hidden states x_all [B][S][D] (bf16).
int launch_gather_rows(const void* x_all, int B, int S, int D, const int32_t* win_lo, int beta, const int32_t* idx,
                       int k, void* x_win, void* x_trk, int32_t* pos_win, int* status, cudaStream_t s);

size_t proj_tc_smem_bytes(int bn);
size_t attn_tc_smem_bytes();

}  // namespace dllm
