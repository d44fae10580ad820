// Host side of the C ABI: argument checks, the flat cache allocator, the rotary
// table, TMA descriptors, tile/split selection and kernel launches.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"

using namespace dllm;

namespace dllm {

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  struct Entry {
    int device;
    const void* kernel;
    int bytes;
  };
  static std::mutex mu;
  static std::vector<Entry> table;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (Entry& en : table) {
    if (en.device == dev && en.kernel == kernel) {
      if (en.bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) en.bytes = bytes;
      return e;
    }
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) table.push_back(Entry{dev, kernel, bytes});
  return e;
}

}  // namespace dllm

namespace {

// Device allocations of the library go through dev_alloc, which a test can make fail on
// purpose (dllm_selftest_fail_alloc) to exercise the error paths without a GPU fault.
std::mutex g_alloc_mu;
int g_fail_alloc_in = 0;  // > 0: the g_fail_alloc_in-th allocation from now fails

cudaError_t dev_alloc(void** p, size_t bytes) {
  {
    std::lock_guard<std::mutex> lock(g_alloc_mu);
    if (g_fail_alloc_in > 0 && --g_fail_alloc_in == 0) {
      *p = nullptr;
      return cudaErrorMemoryAllocation;
    }
  }
  return cudaMalloc(p, bytes);
}
template <typename T>
cudaError_t dev_alloc(T** p, size_t bytes) {
  void* v = nullptr;
  const cudaError_t e = dev_alloc(&v, bytes);
  *p = static_cast<T*>(v);
  return e;
}

int from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return DLLM_OK;
  if (e == cudaErrorMemoryAllocation) return DLLM_EOOM;
  return DLLM_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes_of(int kv_dtype) { return kv_dtype == DLLM_F32 ? 4 : (kv_dtype == DLLM_BF16 ? 2 : 1); }

// Shape checks shared by dllm_cache_bytes and dllm_cache_alloc.
int check_desc(const dllm_cache_desc* d) {
  if (!d) return DLLM_EINVAL;
  if (d->n_layers < 1 || d->batch < 1 || d->max_pos < 1 || d->tail_slots < 0 || d->n_heads < 1 || d->head_dim < 2)
    return DLLM_EINVAL;
  if (d->kv_dtype != DLLM_F32 && d->kv_dtype != DLLM_BF16 && d->kv_dtype != DLLM_E4M3) return DLLM_EINVAL;
  if (!(d->rope_theta > 0.0) || !std::isfinite(d->rope_theta)) return DLLM_EINVAL;
  if ((long long)d->max_pos + d->tail_slots > (1 << 24)) return DLLM_EINVAL;
  if ((long long)d->n_heads * d->head_dim > 65536) return DLLM_EINVAL;
  if (d->kv_dtype == DLLM_F32) {
    if (d->head_dim % 4 != 0 || d->head_dim > 256) return DLLM_EUNSUPPORTED;
  } else {
    if (d->head_dim != kHd) return DLLM_EUNSUPPORTED;
  }
  return DLLM_OK;
}

size_t kv_bytes_of(const dllm_cache_desc* d) {
  return (size_t)d->n_layers * d->batch * (size_t)(d->max_pos + d->tail_slots) * 2 * d->n_heads * d->head_dim *
         elem_bytes_of(d->kv_dtype);
}
size_t scale_bytes_of(const dllm_cache_desc* d) {
  if (d->kv_dtype != DLLM_E4M3) return 0;
  return (size_t)d->n_layers * d->batch * (size_t)(d->max_pos + d->tail_slots) * 2 * d->n_heads * sizeof(float);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D tile map over a row-major [rows][cols] bf16 matrix with 128-byte swizzle.
bool map_2d_bf16(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D tile map over one layer of the cache viewed as [B*slots][2H][hd].
bool map_cache(CUtensorMap* m, const void* layer, int kv_dtype, int hd, int H, uint64_t rows,
               uint32_t box_rows = kKeyTile) {
  auto enc = encode_fn();
  if (!enc) return false;
  const uint32_t eb = kv_dtype == DLLM_E4M3 ? 1 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)(2 * H), rows};
  cuuint64_t strides[2] = {(cuuint64_t)hd * eb, (cuuint64_t)2 * H * hd * eb};
  cuuint32_t box[3] = {128u / eb, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  const CUtensorMapDataType dt = kv_dtype == DLLM_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return enc(m, dt, 3, const_cast<void*>(layer), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

}  // namespace

extern "C" {

size_t dllm_cache_bytes(const dllm_cache_desc* desc) {
  if (check_desc(desc) != DLLM_OK) return 0;
  return kv_bytes_of(desc) + scale_bytes_of(desc);
}

int dllm_cache_alloc(const dllm_cache_desc* desc, dllm_cache** out) {
  if (!out) return DLLM_EINVAL;
  *out = nullptr;
  int rc = check_desc(desc);
  if (rc != DLLM_OK) return rc;
  const size_t kvb = kv_bytes_of(desc), scb = scale_bytes_of(desc);
  if (desc->external_buf) {
    if (desc->external_bytes < kvb + scb) return DLLM_EINVAL;
    if (reinterpret_cast<uintptr_t>(desc->external_buf) & 255u) return DLLM_EINVAL;
  }
  dllm_cache* c = new (std::nothrow) dllm_cache();
  if (!c) return DLLM_EOOM;
  c->desc = *desc;
  c->slots = desc->max_pos + desc->tail_slots;
  c->elem_bytes = elem_bytes_of(desc->kv_dtype);
  c->kv_bytes = kvb;
  c->scale_bytes = scb;
  c->layer_elems = (size_t)desc->batch * c->slots * 2 * desc->n_heads * desc->head_dim;
  c->layer_scales = desc->kv_dtype == DLLM_E4M3 ? (size_t)desc->batch * c->slots * 2 * desc->n_heads : 0;

  auto fail = [&](int code) {
    dllm_cache_free(c);
    return code;
  };
  cudaError_t e = cudaGetDevice(&c->device);
  if (e != cudaSuccess) return fail(from_cuda(e));
  e = cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device);
  if (e != cudaSuccess) return fail(from_cuda(e));
  if (desc->kv_dtype != DLLM_F32) {
    // CTA pairs the projection can keep resident at once (0: use single-CTA tiles)
    int clusters = 0;
    if (proj_pair_max_clusters(&clusters) != 0) clusters = 0;
    (void)cudaGetLastError();
    c->pair_clusters = clusters < c->sm_count / 2 ? clusters : c->sm_count / 2;
  }

  if (desc->external_buf) {
    c->kv = desc->external_buf;
    c->owns_kv = false;
  } else {
    e = dev_alloc(&c->kv, kvb + scb);
    if (e != cudaSuccess) return fail(from_cuda(e));
    c->owns_kv = true;
  }
  c->scale = scb ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(c->kv) + kvb) : nullptr;

  // rotary table: angle p * theta^(-2i/hd) in fp64, cos/sin rounded to fp32
  const int half = desc->head_dim / 2;
  std::vector<float2> tab((size_t)desc->max_pos * half);
  for (int p = 0; p < desc->max_pos; ++p)
    for (int i = 0; i < half; ++i) {
      const double a = (double)p * std::pow(desc->rope_theta, -2.0 * i / desc->head_dim);
      tab[(size_t)p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
  e = dev_alloc(&c->rope, tab.size() * sizeof(float2));
  if (e != cudaSuccess) return fail(from_cuda(e));
  e = cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(from_cuda(e));

  e = dev_alloc(&c->status, sizeof(int));
  if (e != cudaSuccess) return fail(from_cuda(e));
  e = cudaMemset(c->status, 0, sizeof(int));
  if (e != cudaSuccess) return fail(from_cuda(e));
  e = dev_alloc(&c->drift_cnt, (size_t)desc->batch * sizeof(int));
  if (e != cudaSuccess) return fail(from_cuda(e));
  e = cudaMemset(c->drift_cnt, 0, (size_t)desc->batch * sizeof(int));
  if (e != cudaSuccess) return fail(from_cuda(e));
  {
    // fused drift test: the partial sums (zeroed; the finalize kernel zeroes them again)
    const size_t rows = (size_t)desc->batch * kMaxDriftRows;
    const size_t bytes = rows * 6 * sizeof(float);
    e = dev_alloc(&c->drift_acc, bytes);
    if (e != cudaSuccess) return fail(from_cuda(e));
    c->drift_acc_bytes = bytes;
    e = cudaMemset(c->drift_acc, 0, bytes);
    if (e != cudaSuccess) return fail(from_cuda(e));
  }

  // split-KV partials: at most 4 * SMs slots of kQChunk rows (the key splits of few
  // units, or the tail pieces of the balanced schedule), and the tail units' arrival
  // counts (zeroed)
  if (desc->kv_dtype != DLLM_F32) {
    c->ws_floats = (size_t)4 * c->sm_count * kQChunk * (kHd + 2);
    e = dev_alloc(&c->ws, c->ws_floats * sizeof(float));
    if (e != cudaSuccess) return fail(from_cuda(e));
    e = dev_alloc(&c->merge_cnt, (size_t)2 * c->sm_count * sizeof(int));
    if (e != cudaSuccess) return fail(from_cuda(e));
    e = cudaMemset(c->merge_cnt, 0, (size_t)2 * c->sm_count * sizeof(int));
    if (e != cudaSuccess) return fail(from_cuda(e));
  }
  *out = c;
  return DLLM_OK;
}

int dllm_cache_free(dllm_cache* c) {
  if (!c) return DLLM_OK;
  cudaDeviceSynchronize();
  if (c->owns_kv && c->kv) cudaFree(c->kv);
  if (c->rope) cudaFree(c->rope);
  if (c->status) cudaFree(c->status);
  if (c->drift_cnt) cudaFree(c->drift_cnt);
  if (c->drift_acc) cudaFree(c->drift_acc);
  if (c->ws) cudaFree(c->ws);
  if (c->merge_cnt) cudaFree(c->merge_cnt);
  delete c;
  return DLLM_OK;
}

int dllm_cache_get_layout(const dllm_cache* c, dllm_cache_layout* out) {
  if (!c || !out) return DLLM_EINVAL;
  out->kv = c->kv;
  out->scale = c->scale;
  out->kv_bytes = c->kv_bytes;
  out->scale_bytes = c->scale_bytes;
  out->layer_elems = c->layer_elems;
  out->slots = c->slots;
  out->elem_bytes = c->elem_bytes;
  return DLLM_OK;
}

}  // extern "C"

namespace {

struct StepArgs {
  int layer;
  const void* x;
  const void* w_qkv;
  const int32_t* positions;
  const uint8_t* view;
  int n_tok;
  void* out;
  const void* kv_x;
  const int32_t* kv_positions;
  int n_kv;
  void* probe_kv;
  cudaStream_t s;
  // K/V-only rows of sequence b only where one of flags[j][b], j < n_flag_sets, is set
  const int32_t* kv_seq_flags = nullptr;
  int n_flag_sets = 0;
  // fused drift test: the K/V-only rows are probes compared with the cache (cos set)
  float* drift_cos = nullptr;
  int32_t* drift_refresh = nullptr;
  float drift_gamma = 0.0f;
};

void* layer_kv(dllm_cache* c, int layer) {
  return reinterpret_cast<uint8_t*>(c->kv) + (size_t)layer * c->layer_elems * c->elem_bytes;
}
float* layer_scale(dllm_cache* c, int layer) {
  return c->scale ? c->scale + (size_t)layer * c->layer_scales : nullptr;
}

// The calls launch on the current device; the cache's buffers live on the device that
// was current when it was created.  A call made with another device current would run
// kernels against another GPU's memory, so it is rejected.
bool on_cache_device(const dllm_cache* c) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return d == c->device;
}

int check_common(dllm_cache* c, int layer, int n_tok, const int32_t* positions, void* out) {
  if (!c || layer < 0 || layer >= c->desc.n_layers || n_tok < 0) return DLLM_EINVAL;
  if (!on_cache_device(c)) return DLLM_EINVAL;
  if (n_tok > 0 && (!positions || !out)) return DLLM_EINVAL;
  if (!aligned16(out)) return DLLM_EINVAL;
  if ((long long)c->desc.batch * n_tok > (1ll << 30)) return DLLM_EINVAL;
  return DLLM_OK;
}

int check_project(dllm_cache* c, const StepArgs& a) {
  int rc = check_common(c, a.layer, a.n_tok, a.positions, a.out);
  if (rc) return rc;
  if (a.n_kv < 0 || !a.w_qkv) return DLLM_EINVAL;
  if (a.n_tok > 0 && !a.x) return DLLM_EINVAL;
  if (a.n_kv > 0 && (!a.kv_x || !a.kv_positions)) return DLLM_EINVAL;
  if (!aligned16(a.x) || !aligned16(a.w_qkv) || !aligned16(a.kv_x) || !aligned16(a.probe_kv)) return DLLM_EINVAL;
  if (a.n_tok > 0 && a.x == a.out) return DLLM_EINVAL;
  if ((long long)c->desc.batch * a.n_kv > (1ll << 30)) return DLLM_EINVAL;
  if (c->desc.kv_dtype != DLLM_F32 && (c->desc.n_heads * c->desc.head_dim) % kHd != 0) return DLLM_EUNSUPPORTED;
  return DLLM_OK;
}

int check_attend(dllm_cache* c, int layer, int n_tok, const int32_t* positions, const uint8_t* view, void* out) {
  int rc = check_common(c, layer, n_tok, positions, out);
  if (rc) return rc;
  const dllm_cache_desc& d = c->desc;
  if (view && d.max_pos > 32 * 512) return DLLM_EUNSUPPORTED;
  if (d.kv_dtype == DLLM_F32 && (size_t)(d.max_pos + d.tail_slots + d.head_dim + 32) * 4 > 200 * 1024)
    return DLLM_EUNSUPPORTED;
  return DLLM_OK;
}

ProjParams make_proj(dllm_cache* c, const StepArgs& a) {
  const dllm_cache_desc& d = c->desc;
  ProjParams p{};
  p.D = d.n_heads * d.head_dim;
  p.H = d.n_heads;
  p.n_tok = a.n_tok;
  p.n_kv = a.n_kv;
  p.m_q = d.batch * a.n_tok;
  p.m_kv = d.batch * a.n_kv;
  p.positions = a.positions;
  p.view = a.view;
  p.kv_positions = a.kv_positions;
  p.kv_seq_flags = a.kv_seq_flags;
  p.n_flag_sets = a.n_flag_sets;
  p.batch = d.batch;
  p.q_out = a.out;
  p.cache_kv = layer_kv(c, a.layer);
  p.cache_scale = layer_scale(c, a.layer);
  p.probe = a.probe_kv;
  p.kv_dtype = d.kv_dtype;
  p.max_pos = d.max_pos;
  p.tail = d.tail_slots;
  p.slots = c->slots;
  p.rope = c->rope;
  p.status = c->status;
  if (a.drift_cos != nullptr) {
    p.probe = nullptr;
    p.drift_acc = c->drift_acc;
    p.drift_cos = a.drift_cos;
    p.drift_refresh = a.drift_refresh;
    p.drift_gamma = a.drift_gamma;
  }
  return p;
}

int do_project(dllm_cache* c, const StepArgs& a, void* raw_q = nullptr, void* raw_kv = nullptr) {
  if (a.n_tok == 0 && a.n_kv == 0) return DLLM_OK;
  const dllm_cache_desc& d = c->desc;
  ProjParams p = make_proj(c, a);
  p.raw_q = raw_q;
  p.raw_kv = raw_kv;
  p.raw_f32 = d.kv_dtype == DLLM_E4M3;
  const int D = p.D;
  int rc;
  if (d.kv_dtype == DLLM_F32) {
    rc = launch_proj_f32(p, (const float*)a.x, (const float*)a.kv_x, (const float*)a.w_qkv, d.head_dim, a.s);
    return rc ? from_cuda((cudaError_t)rc) : DLLM_OK;
  }
  int bn = (D % 256 == 0) ? 256 : 128;
  auto tiles_for = [&](int bnv) {
    return (long long)ceil_div(p.m_q, 128) * (3 * D / bnv) + (long long)ceil_div(p.m_kv, 128) * (2 * D / bnv);
  };
  if (bn == 256 && tiles_for(256) < c->sm_count) bn = 128;
  p.k_blocks = D / 64;
  p.m_fastest = ((size_t)(p.m_q + p.m_kv) * D * 2 <= ((size_t)48 << 20)) ? 1 : 0;

  // Tiles beyond the last full round: when they would leave at least half the workers
  // (CTAs, or CTA pairs) idle, each is done as two 128-column halves spread over them.
  auto split_tail = [&](int tiles, int workers) {
    p.tiles_total = tiles;
    p.whole_items = tiles;
    const int rem = tiles % workers;
    if (rem > 0 && 2 * rem <= workers) p.whole_items = tiles - rem;
    p.items_total = p.whole_items + 2 * (tiles - p.whole_items);
  };

  CUtensorMap tm_w, tm_w_half, tm_x, tm_xkv;
  if (p.m_q > 0) {
    if (!map_2d_bf16(&tm_x, a.x, D, p.m_q, 64, 128)) return DLLM_ECUDA;
  }
  if (p.m_kv > 0) {
    if (!map_2d_bf16(&tm_xkv, a.kv_x, D, p.m_kv, 64, 128)) return DLLM_ECUDA;
  }
  if (bn == 256 && c->pair_clusters >= 1) {
    // 256 x 256 tiles on CTA pairs (cta_group::2); each CTA loads 128 (or 64) W rows
    if (!map_2d_bf16(&tm_w, a.w_qkv, D, 3 * (uint64_t)D, 64, 128)) return DLLM_ECUDA;
    if (!map_2d_bf16(&tm_w_half, a.w_qkv, D, 3 * (uint64_t)D, 64, 64)) return DLLM_ECUDA;
    if (p.m_q == 0) tm_x = tm_w;
    if (p.m_kv == 0) tm_xkv = tm_w;
    p.pmt_q = ceil_div(p.m_q, 256);
    p.pmt_kv = ceil_div(p.m_kv, 256);
    const int pairs = c->pair_clusters;
    split_tail(p.pmt_q * (3 * D / 256) + p.pmt_kv * (2 * D / 256), pairs);
    const int grid = 2 * (p.items_total < pairs ? p.items_total : pairs);
    rc = launch_proj_pair(p, tm_x, tm_xkv, tm_w, tm_w_half, grid, a.s);
    if (!rc && p.drift_acc) rc = launch_drift_finalize(p, a.s);
    return rc ? from_cuda((cudaError_t)rc) : DLLM_OK;
  }
  p.mt_q = ceil_div(p.m_q, 128);
  p.mt_kv = ceil_div(p.m_kv, 128);
  p.nt_q = 3 * D / bn;
  p.nt_kv = 2 * D / bn;
  p.tiles_q = p.mt_q * p.nt_q;
  split_tail(p.tiles_q + p.mt_kv * p.nt_kv, c->sm_count);
  if (bn != 256) {  // 128-wide tiles have no halves
    p.whole_items = p.tiles_total;
    p.items_total = p.tiles_total;
  }
  if (!map_2d_bf16(&tm_w, a.w_qkv, D, 3 * (uint64_t)D, 64, bn)) return DLLM_ECUDA;
  if (!map_2d_bf16(&tm_w_half, a.w_qkv, D, 3 * (uint64_t)D, 64, 128)) return DLLM_ECUDA;
  if (p.m_q == 0) tm_x = tm_w;
  if (p.m_kv == 0) tm_xkv = tm_w;
  const int grid = p.items_total < c->sm_count ? p.items_total : c->sm_count;
  rc = launch_proj_tc(p, tm_x, tm_xkv, tm_w, tm_w_half, bn, grid, a.s);
  if (!rc && p.drift_acc) rc = launch_drift_finalize(p, a.s);
  return rc ? from_cuda((cudaError_t)rc) : DLLM_OK;
}

// Key range of an attention launch: regular slots [lo, hi) of every sequence, further
// limited to the first key_len[b] slots of sequence b when key_len is given; state
// (partial softmax state per row and head) replaces the normalised output when given.
struct KeyRange {
  int lo = 0, hi = -1;  // hi < 0: every slot (and the Flash-Verify tail)
  const int32_t* key_len = nullptr;
  float* state = nullptr;
  const float* state_in = nullptr;  // cached state of the other keys, merged into the output
  const void* q = nullptr;          // rotated Q, when it is not in `out`
};

// Where the split-KV partial states go: the cache's own workspace, unless `get` is set,
// in which case it is called (only when the keys are split) for a buffer of `floats`.
struct SplitScratch {
  int (*get)(float** out) = nullptr;
  size_t floats = 0;
};

// Tensor maps of an attention launch: Q (a.nq_pad rows a box), the layer's cache (128
// rows a box), and, when the launch's last key tile runs past the sequence's slots, the
// cache with boxes of only that tile's rows (sets a.tail_rows; else a copy of tm_kv).
int attn_maps(dllm_cache* c, int layer, const void* q, int n_tok, AttnParams& a, CUtensorMap* tm_q, CUtensorMap* tm_kv,
              CUtensorMap* tm_kv_tail) {
  const dllm_cache_desc& d = c->desc;
  const int H = d.n_heads, hd = d.head_dim, D = H * hd;
  if (!map_2d_bf16(tm_q, q, D, (uint64_t)d.batch * n_tok, 64, a.nq_pad)) return DLLM_ECUDA;
  const uint64_t rows = (uint64_t)d.batch * c->slots;
  if (!map_cache(tm_kv, layer_kv(c, layer), d.kv_dtype, hd, H, rows)) return DLLM_ECUDA;
  a.tail_rows = 0;
  *tm_kv_tail = *tm_kv;
  const int last = a.tile_lo + a.key_tiles - 1;  // the launch's last key tile
  const int valid = c->slots - last * kKeyTile;   // slots of the sequence in that tile
  if (valid > 0 && valid < kKeyTile) {
    a.tail_rows = std::min(kKeyTile, (valid + 7) / 8 * 8);
    if (a.tail_rows < kKeyTile &&
        !map_cache(tm_kv_tail, layer_kv(c, layer), d.kv_dtype, hd, H, rows, (uint32_t)a.tail_rows))
      return DLLM_ECUDA;
    if (a.tail_rows == kKeyTile) a.tail_rows = 0;
  }
  return DLLM_OK;
}

int do_attend(dllm_cache* c, int layer, const int32_t* positions, const uint8_t* view, int n_tok, void* out,
              cudaStream_t s, const KeyRange& kr = KeyRange(), const SplitScratch& scratch = SplitScratch()) {
  if (n_tok == 0) return DLLM_OK;
  const dllm_cache_desc& d = c->desc;
  const int B = d.batch, H = d.n_heads, hd = d.head_dim, D = H * hd;
  AttnParams a{};
  a.B = B;
  a.H = H;
  a.D = D;
  a.n_tok = n_tok;
  a.max_pos = d.max_pos;
  a.tail = d.tail_slots;
  a.slots = c->slots;
  a.view = view;
  a.positions = positions;
  a.out = out;
  a.ws = scratch.get ? nullptr : c->ws;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)hd));
  a.kv_scale = layer_scale(c, layer);
  a.kv_dtype = d.kv_dtype;
  a.status = c->status;
  a.key_lo = 0;
  a.key_hi = d.max_pos;
  a.tile_lo = 0;
  a.key_len = kr.key_len;
  a.state = kr.state;
  a.state_in = kr.state_in;
  a.ranged = kr.hi >= 0 || kr.key_len != nullptr;
  if (kr.hi >= 0) {
    a.key_lo = kr.lo;
    a.key_hi = kr.hi;
    a.tile_lo = kr.lo / kKeyTile;
  }
  int rc;
  if (d.kv_dtype == DLLM_F32) {
    if (a.ranged || a.state) return DLLM_EUNSUPPORTED;
    rc = launch_attn_f32(a, (const float*)layer_kv(c, layer), hd, s);
    return rc ? from_cuda((cudaError_t)rc) : DLLM_OK;
  }
  a.nq_pad = n_tok <= 32 ? 32 : (n_tok <= 48 ? 48 : 64);
  a.n_qchunks = ceil_div(n_tok, kQChunk);
  a.key_tiles = kr.hi >= 0 ? ceil_div(a.key_hi, kKeyTile) - a.tile_lo
                           : ceil_div(d.max_pos + (view ? d.tail_slots : 0), kKeyTile);
  const int base = B * H * a.n_qchunks;
  const size_t scratch_floats = scratch.get ? scratch.floats : c->ws_floats;
  // Balanced schedule: full waves of whole units, then the remaining units (fewer than
  // the SMs) cut into equal pieces that all SMs share, merged in the kernel by whichever
  // CTA completes a unit.  The piece count minimises the largest number of key tiles a
  // CTA runs, counting a merge as one tile; ties go to fewer pieces, and one piece is
  // the plain round-robin.  Only with at least one full wave: with fewer units than SMs
  // the merge would sit on every CTA's path, and the key split below with its second
  // kernel measured faster (batch 1: 16.5 against 18.4 us).  Not for ragged batches
  // (unequal units) or partial-state launches (one unit per row), nor e4m3 caches, whose
  // tiles are bound by the per-tile conversion chain: there a piece's extra boundary (the
  // Q split, the merge) cost more than the balance gained (86 against 80 us on the
  // batch-8, 3072-slot cache).  The same rule holds for every scratch, so that each
  // entry point makes the same choice.
  if (d.kv_dtype == DLLM_BF16 && !kr.key_len && !a.state && !a.state_in && base >= c->sm_count) {
    const int sm = c->sm_count, kt = a.key_tiles;
    const int waves = base / sm, tail = base - waves * sm;
    const size_t slot_floats = (size_t)kQChunk * (kHd + 2);
    const size_t max_slots = std::min(c->ws_floats, (size_t)DLLM_NOALLOC_SCRATCH_BYTES / sizeof(float)) / slot_floats;
    int best_k = 1, best_tps = kt;
    long long best = -1;
    for (int k = 1; tail > 0 && k <= kMaxPieces && k <= kt; ++k) {
      const int tps = ceil_div(kt, k), kk = ceil_div(kt, tps);
      if (kk != k || (size_t)tail * kk > max_slots) continue;
      const long long items = (long long)tail * kk;
      const long long grid_k = waves ? sm : std::min<long long>(items, sm);
      const long long cost = (long long)waves * kt + (items + grid_k - 1) / grid_k * tps + (kk > 1 ? 1 : 0);
      if (best < 0 || cost < best) {
        best = cost;
        best_k = kk;
        best_tps = tps;
      }
    }
    if (best_k > 1) {
      a.n_splits = 1;
      a.tiles_per_split = kt;
      a.units = base;
      a.dp_waves = waves;
      a.tail_units = tail;
      a.tail_pieces = best_k;
      a.piece_tiles = best_tps;
      a.merge_cnt = c->merge_cnt;
      if ((size_t)tail * best_k * slot_floats > scratch_floats) return DLLM_EUNSUPPORTED;
      if (scratch.get) {
        rc = scratch.get(&a.ws);
        if (rc) return rc;
      }
      const int grid = waves ? sm : std::min(tail * best_k, sm);
      CUtensorMap tm_q, tm_kv, tm_kv_tail;
      rc = attn_maps(c, layer, kr.q ? kr.q : out, n_tok, a, &tm_q, &tm_kv, &tm_kv_tail);
      if (rc) return rc;
      rc = launch_attn_tc(a, tm_q, tm_kv, tm_kv_tail, grid, s);
      return rc ? from_cuda((cudaError_t)rc) : DLLM_OK;
    }
  }
  // Fewer units than SMs where the balanced schedule does not apply (ragged batches,
  // e4m3 caches): the keys split evenly, partial states merged by a second kernel.
  int splits = 1;
  if (base < c->sm_count && !a.state && !a.state_in) {  // states are per row: one unit per row
    splits = ceil_div(c->sm_count, base);
    if (splits > a.key_tiles) splits = a.key_tiles;
  }
  a.tiles_per_split = ceil_div(a.key_tiles, splits);
  a.n_splits = ceil_div(a.key_tiles, a.tiles_per_split);
  a.units = base * a.n_splits;
  if (a.n_splits > 1) {
    const size_t need = (size_t)a.units * kQChunk * (kHd + 2);
    if (need > (scratch.get ? scratch.floats : c->ws_floats)) return DLLM_EUNSUPPORTED;
    if (scratch.get) {
      rc = scratch.get(&a.ws);
      if (rc) return rc;
    }
  }

  CUtensorMap tm_q, tm_kv, tm_kv_tail;
  rc = attn_maps(c, layer, kr.q ? kr.q : out, n_tok, a, &tm_q, &tm_kv, &tm_kv_tail);
  if (rc) return rc;
  const int grid = a.units < c->sm_count ? a.units : c->sm_count;
  rc = launch_attn_tc(a, tm_q, tm_kv, tm_kv_tail, grid, s);
  if (rc) return from_cuda((cudaError_t)rc);
  if (a.n_splits > 1) {
    rc = launch_attn_combine(a, s);
    if (rc) return from_cuda((cudaError_t)rc);
  }
  return DLLM_OK;
}

}  // namespace

extern "C" {

int dllm_cache_project(dllm_cache* c, int layer, const void* x, const void* w_qkv, const int32_t* positions,
                       const uint8_t* view, int n_tok, void* out, const void* kv_x, const int32_t* kv_positions,
                       int n_kv, void* probe_kv, void* stream) {
  StepArgs a{layer, x, w_qkv, positions, view, n_tok, out, kv_x, kv_positions, n_kv, probe_kv,
             reinterpret_cast<cudaStream_t>(stream)};
  int rc = check_project(c, a);
  if (rc) return rc;
  return do_project(c, a);
}

int dllm_cache_attend(dllm_cache* c, int layer, const int32_t* positions, const uint8_t* view, int n_tok, void* out,
                      void* stream) {
  int rc = check_attend(c, layer, n_tok, positions, view, out);
  if (rc) return rc;
  return do_attend(c, layer, positions, view, n_tok, out, reinterpret_cast<cudaStream_t>(stream));
}

int dllm_cache_step(dllm_cache* c, int layer, const void* x, const void* w_qkv, const int32_t* positions,
                    const uint8_t* view, int n_tok, void* out, const void* kv_x, const int32_t* kv_positions, int n_kv,
                    void* probe_kv, void* stream) {
  StepArgs a{layer, x, w_qkv, positions, view, n_tok, out, kv_x, kv_positions, n_kv, probe_kv,
             reinterpret_cast<cudaStream_t>(stream)};
  int rc = check_project(c, a);
  if (rc) return rc;
  if (n_tok > 0) {
    rc = check_attend(c, layer, n_tok, positions, view, out);
    if (rc) return rc;
  }
  rc = do_project(c, a);
  if (rc) return rc;
  return do_attend(c, layer, positions, view, n_tok, out, a.s);
}

namespace {
int project_drift_args(dllm_cache* c, StepArgs& a, int k, float gamma, float* cos, int32_t* refresh) {
  if (!c) return DLLM_EINVAL;
  if (k < 1 || !a.kv_x || !a.kv_positions || !cos) return DLLM_EINVAL;
  if (c->desc.kv_dtype == DLLM_F32) return DLLM_EUNSUPPORTED;
  if (k > kMaxDriftRows) return DLLM_EUNSUPPORTED;
  a.drift_cos = cos;
  a.drift_refresh = refresh;
  a.drift_gamma = gamma;
  return check_project(c, a);
}
}  // namespace

int dllm_cache_project_drift(dllm_cache* c, int layer, const void* x, const void* w_qkv, const int32_t* positions,
                             const uint8_t* view, int n_tok, void* out, const void* kv_x, const int32_t* idx, int k,
                             float gamma, float* cos, int32_t* refresh, void* stream) {
  StepArgs a{layer, x, w_qkv, positions, view, n_tok, out, kv_x, idx, k, nullptr,
             reinterpret_cast<cudaStream_t>(stream)};
  int rc = project_drift_args(c, a, k, gamma, cos, refresh);
  if (rc) return rc;
  return do_project(c, a);
}

int dllm_cache_step_drift(dllm_cache* c, int layer, const void* x, const void* w_qkv, const int32_t* positions,
                          const uint8_t* view, int n_tok, void* out, const void* kv_x, const int32_t* idx, int k,
                          float gamma, float* cos, int32_t* refresh, void* stream) {
  StepArgs a{layer, x, w_qkv, positions, view, n_tok, out, kv_x, idx, k, nullptr,
             reinterpret_cast<cudaStream_t>(stream)};
  int rc = project_drift_args(c, a, k, gamma, cos, refresh);
  if (rc) return rc;
  if (n_tok > 0) {
    rc = check_attend(c, layer, n_tok, positions, view, out);
    if (rc) return rc;
  }
  rc = do_project(c, a);
  if (rc) return rc;
  return do_attend(c, layer, positions, view, n_tok, out, a.s);
}

int dllm_cache_attend_ragged(dllm_cache* c, int layer, const int32_t* positions, int n_tok, const int32_t* key_len,
                             void* out, void* stream) {
  int rc = check_attend(c, layer, n_tok, positions, nullptr, out);
  if (rc) return rc;
  if (!key_len) return DLLM_EINVAL;
  KeyRange kr;
  kr.key_len = key_len;
  return do_attend(c, layer, positions, nullptr, n_tok, out, reinterpret_cast<cudaStream_t>(stream), kr);
}

int dllm_cache_attend_partial(dllm_cache* c, int layer, const int32_t* positions, int n_tok, const void* q,
                              int slot_lo, int slot_hi, float* state, void* stream) {
  int rc = check_attend(c, layer, n_tok, positions, nullptr, const_cast<void*>(q));
  if (rc) return rc;
  if (!state || !aligned16(state) || slot_lo < 0 || slot_hi <= slot_lo || slot_hi > c->desc.max_pos)
    return DLLM_EINVAL;
  KeyRange kr;
  kr.lo = slot_lo;
  kr.hi = slot_hi;
  kr.state = state;
  return do_attend(c, layer, positions, nullptr, n_tok, const_cast<void*>(q), reinterpret_cast<cudaStream_t>(stream),
                   kr);
}

int dllm_cache_attend_with_state(dllm_cache* c, int layer, const int32_t* positions, int n_tok, const void* q,
                                 int slot_lo, int slot_hi, const float* state, void* out, void* stream) {
  int rc = check_attend(c, layer, n_tok, positions, nullptr, out);
  if (rc) return rc;
  if (n_tok > 0 && (!q || !state)) return DLLM_EINVAL;
  if (!aligned16(q) || !aligned16(state) || slot_lo < 0 || slot_hi <= slot_lo || slot_hi > c->desc.max_pos)
    return DLLM_EINVAL;
  if (c->desc.kv_dtype == DLLM_F32) return DLLM_EUNSUPPORTED;
  KeyRange kr;
  kr.lo = slot_lo;
  kr.hi = slot_hi;
  kr.state_in = state;
  kr.q = q;
  return do_attend(c, layer, positions, nullptr, n_tok, out, reinterpret_cast<cudaStream_t>(stream), kr);
}

int dllm_attend_merge(const float* state_a, const float* state_b, int batch, int n_tok, int n_heads, int head_dim,
                      void* out, float* state_out, void* stream) {
  if (!state_a || !state_b || (!out && !state_out) || batch < 1 || n_tok < 0 || n_heads < 1) return DLLM_EINVAL;
  if (!aligned16(state_a) || !aligned16(state_b) || !aligned16(out) || !aligned16(state_out)) return DLLM_EINVAL;
  if ((long long)batch * n_tok * n_heads >= (1ll << 31)) return DLLM_EINVAL;
  if (head_dim != kHd) return DLLM_EUNSUPPORTED;
  if (n_tok == 0) return DLLM_OK;
  const int rc = launch_state_merge(state_a, state_b, batch * n_tok, n_heads, out, state_out,
                                    reinterpret_cast<cudaStream_t>(stream));
  return rc ? from_cuda((cudaError_t)rc) : DLLM_OK;
}

int dllm_attention_mass(dllm_cache* c, int layer, const int32_t* positions, const uint8_t* view, int n_tok,
                        const void* q, float* mass, void* stream) {
  int rc = check_attend(c, layer, n_tok, positions, view, const_cast<void*>(q));
  if (rc) return rc;
  if (!mass) return DLLM_EINVAL;
  if (c->desc.kv_dtype == DLLM_F32) return DLLM_EUNSUPPORTED;
  const dllm_cache_desc& d = c->desc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(mass, 0, (size_t)d.batch * d.max_pos * sizeof(float), s);
  if (e != cudaSuccess) return from_cuda(e);
  if (n_tok == 0) return DLLM_OK;
  const int B = d.batch, H = d.n_heads, hd = d.head_dim, D = H * hd;
  AttnParams a{};
  a.B = B;
  a.H = H;
  a.D = D;
  a.n_tok = n_tok;
  a.max_pos = d.max_pos;
  a.tail = d.tail_slots;
  a.slots = c->slots;
  a.view = view;
  a.positions = positions;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)hd));
  a.kv_scale = layer_scale(c, layer);
  a.kv_dtype = d.kv_dtype;
  a.status = c->status;
  a.nq_pad = n_tok <= 32 ? 32 : 64;
  a.n_qchunks = ceil_div(n_tok, kQChunk);
  a.key_tiles = ceil_div(d.max_pos + (view ? d.tail_slots : 0), kKeyTile);
  a.n_splits = 1;
  a.tiles_per_split = a.key_tiles;
  a.units = B * H * a.n_qchunks;
  CUtensorMap tm_q, tm_kv;
  if (!map_2d_bf16(&tm_q, q, D, (uint64_t)B * n_tok, 64, a.nq_pad)) return DLLM_ECUDA;
  if (!map_cache(&tm_kv, layer_kv(c, layer), d.kv_dtype, hd, H, (uint64_t)B * c->slots)) return DLLM_ECUDA;
  const int grid = a.units < c->sm_count ? a.units : c->sm_count;
  rc = launch_attn_mass(a, tm_q, tm_kv, mass, grid, s);
  return rc ? from_cuda((cudaError_t)rc) : DLLM_OK;
}

namespace {
// Bytes per raw projection value in the unfused pipeline's workspace: fp32 for e4m3
// caches (quantised from the unrounded value), bf16 otherwise.
size_t unfused_raw_bytes(const dllm_cache* c) { return c->desc.kv_dtype == DLLM_E4M3 ? 4 : 2; }
size_t unfused_q_bytes(const dllm_cache* c, int n_tok) {
  const size_t D = (size_t)c->desc.n_heads * c->desc.head_dim;
  return (((size_t)c->desc.batch * n_tok * 3 * D * unfused_raw_bytes(c) + 255) / 256) * 256;
}
}  // namespace

size_t dllm_unfused_workspace_bytes(const dllm_cache* c, int n_tok, int n_kv) {
  if (!c || n_tok < 0 || n_kv < 0) return 0;
  const size_t D = (size_t)c->desc.n_heads * c->desc.head_dim;
  return unfused_q_bytes(c, n_tok) + (size_t)c->desc.batch * n_kv * 2 * D * unfused_raw_bytes(c);
}

int dllm_cache_step_unfused(dllm_cache* c, int layer, const void* x, const void* w_qkv, const int32_t* positions,
                            const uint8_t* view, int n_tok, void* out, const void* kv_x, const int32_t* kv_positions,
                            int n_kv, void* probe_kv, void* workspace, size_t workspace_bytes, void* stream) {
  StepArgs a{layer, x, w_qkv, positions, view, n_tok, out, kv_x, kv_positions, n_kv, probe_kv,
             reinterpret_cast<cudaStream_t>(stream)};
  int rc = check_project(c, a);
  if (rc) return rc;
  if (c->desc.kv_dtype == DLLM_F32) return DLLM_EUNSUPPORTED;
  if (n_tok > 0) {
    rc = check_attend(c, layer, n_tok, positions, view, out);
    if (rc) return rc;
  }
  const size_t need = dllm_unfused_workspace_bytes(c, n_tok, n_kv);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return DLLM_EINVAL;
  if (n_tok == 0 && n_kv == 0) return DLLM_OK;
  void* raw_q = workspace;
  void* raw_kv = reinterpret_cast<uint8_t*>(workspace) + unfused_q_bytes(c, n_tok);
  // 1. projection GEMM, plain output to the workspace
  rc = do_project(c, a, raw_q, raw_kv);
  if (rc) return rc;
  // 2. rotary embedding (Q into `out`, K in place), 3. cache (or probe) write
  ProjParams p = make_proj(c, a);
  p.raw_q = raw_q;
  p.raw_kv = raw_kv;
  p.raw_f32 = c->desc.kv_dtype == DLLM_E4M3;
  rc = launch_rope_rows(p, a.s);
  if (rc) return from_cuda((cudaError_t)rc);
  rc = launch_cache_write(p, a.s);
  if (rc) return from_cuda((cudaError_t)rc);
  // 4. attention
  return do_attend(c, layer, positions, view, n_tok, out, a.s);
}

int dllm_kv_topk(const float* mass, int batch, int n_pos, const int32_t* block_lo, int block_len, int k, int32_t* idx,
                 void* stream) {
  if (!mass || !block_lo || !idx || batch < 1 || n_pos < 1 || n_pos > 16384 || block_len < 0 || k < 1 ||
      k > n_pos - block_len)
    return DLLM_EINVAL;
  return from_cuda((cudaError_t)launch_topk(mass, batch, n_pos, block_lo, block_len, k, idx,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

int dllm_kv_drift(const dllm_cache* c, int layer, const int32_t* idx, int k, const void* probe_kv, float gamma,
                  float* cos, int32_t* refresh, void* stream) {
  if (!c || layer < 0 || layer >= c->desc.n_layers || !idx || k < 1 || !probe_kv || !cos) return DLLM_EINVAL;
  if (!on_cache_device(c)) return DLLM_EINVAL;
  if (!aligned16(probe_kv)) return DLLM_EINVAL;
  const dllm_cache_desc& d = c->desc;
  const void* kvl = reinterpret_cast<const uint8_t*>(c->kv) + (size_t)layer * c->layer_elems * c->elem_bytes;
  const float* scl = c->scale ? c->scale + (size_t)layer * c->layer_scales : nullptr;
  return from_cuda((cudaError_t)launch_drift(kvl, scl, d.kv_dtype, d.batch, c->slots, d.max_pos, d.n_heads, d.head_dim,
                                             idx, k, probe_kv, gamma, cos, refresh, c->drift_cnt, c->sm_count,
                                             c->status, reinterpret_cast<cudaStream_t>(stream)));
}

int dllm_gather_rows(dllm_cache* c, const void* x_all, int n_pos, const int32_t* idx, int k, void* x_rows,
                     void* stream) {
  if (!c || !x_all || !idx || !x_rows || n_pos < 1 || k < 1) return DLLM_EINVAL;
  if (!on_cache_device(c)) return DLLM_EINVAL;
  if (!aligned16(x_all) || !aligned16(x_rows)) return DLLM_EINVAL;
  const dllm_cache_desc& d = c->desc;
  if ((long long)d.batch * k > (1ll << 30) || (long long)d.batch * n_pos > (1ll << 40)) return DLLM_EINVAL;
  // the kernel copies rows as 16-byte vectors of bf16 elements: D * elt bytes per row
  const int D = d.n_heads * d.head_dim;
  const int row_bf16 = d.kv_dtype == DLLM_F32 ? 2 * D : D;  // fp32 rows are twice as long
  if (row_bf16 % 8 != 0) return DLLM_EUNSUPPORTED;
  return from_cuda((cudaError_t)launch_gather_rows(x_all, d.batch, n_pos, row_bf16, nullptr, 0, idx, k, nullptr,
                                                   x_rows, nullptr, c->status, reinterpret_cast<cudaStream_t>(stream)));
}

int dllm_kv_topk_gather(dllm_cache* c, const float* mass, int n_pos, const int32_t* block_lo, int block_len, int k,
                        int32_t* idx, const void* x_all, void* x_rows, void* stream) {
  if (!c || !mass || !block_lo || !idx || !x_all || !x_rows || n_pos < 1 || n_pos > 16384 || block_len < 0 || k < 1 ||
      k > n_pos - block_len)
    return DLLM_EINVAL;
  if (!on_cache_device(c)) return DLLM_EINVAL;
  if (!aligned16(x_all) || !aligned16(x_rows)) return DLLM_EINVAL;
  const dllm_cache_desc& d = c->desc;
  if ((long long)d.batch * n_pos > (1ll << 40)) return DLLM_EINVAL;
  const int D = d.n_heads * d.head_dim;
  const int row_bf16 = d.kv_dtype == DLLM_F32 ? 2 * D : D;  // fp32 rows are twice as long
  if (row_bf16 % 8 != 0) return DLLM_EUNSUPPORTED;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (k <= 32)  // one launch: the selection, then the rows, per sequence
    return from_cuda((cudaError_t)launch_topk_gather(mass, d.batch, n_pos, block_lo, block_len, k, idx, x_all,
                                                     row_bf16 / 8, x_rows, s));
  int rc = launch_topk(mass, d.batch, n_pos, block_lo, block_len, k, idx, s);
  if (rc) return from_cuda((cudaError_t)rc);
  return from_cuda((cudaError_t)launch_gather_rows(x_all, d.batch, n_pos, row_bf16, nullptr, 0, idx, k, nullptr,
                                                   x_rows, nullptr, c->status, s));
}

// Multi-layer refresh step: workspace layout (each part at a 256-byte boundary).
struct ElasticWs {
  void *x_win, *x_trk;
  int32_t *pos_win, *idx;
  size_t bytes;
};

static ElasticWs elastic_ws(const dllm_cache* c, int beta, int k, void* base) {
  const size_t B = c->desc.batch, D = (size_t)c->desc.n_heads * c->desc.head_dim;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  size_t off = 0;
  ElasticWs w{};
  uint8_t* p = static_cast<uint8_t*>(base);
  w.x_win = p ? p + off : nullptr;
  off += up(B * beta * D * 2);
  w.x_trk = p ? p + off : nullptr;
  off += up(B * k * D * 2);
  w.pos_win = p ? reinterpret_cast<int32_t*>(p + off) : nullptr;
  off += up(B * beta * 4);
  w.idx = p ? reinterpret_cast<int32_t*>(p + off) : nullptr;
  off += up(B * k * 4);
  w.bytes = off;
  return w;
}

size_t dllm_elastic_workspace_bytes(const dllm_cache* c, int beta, int k) {
  if (!c || beta < 1 || k < 1) return 0;
  return elastic_ws(c, beta, k, nullptr).bytes;
}

int dllm_elastic_step(dllm_cache* c, int n_layers, const void* const* x_all, const void* const* w_qkv,
                      const int32_t* win_lo, int beta, const float* mass, int k, float gamma, void* out, float* cos,
                      int32_t* flags, float* mass_out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!c || n_layers < 1 || n_layers > c->desc.n_layers || !x_all || !w_qkv || !win_lo || !mass || !out || !cos ||
      !flags || !workspace)
    return DLLM_EINVAL;
  if (!on_cache_device(c)) return DLLM_EINVAL;
  const dllm_cache_desc& d = c->desc;
  const int B = d.batch, S = d.max_pos, D = d.n_heads * d.head_dim;
  if (beta < 1 || beta > S || k < 1 || k > S - beta || S > 16384) return DLLM_EINVAL;
  if (k > kMaxDriftRows) return DLLM_EUNSUPPORTED;
  if (d.kv_dtype == DLLM_F32 || D % kHd != 0) return DLLM_EUNSUPPORTED;
  if (!aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DLLM_EINVAL;
  const ElasticWs ws = elastic_ws(c, beta, k, workspace);
  if (workspace_bytes < ws.bytes) return DLLM_EINVAL;
  for (int l = 0; l < n_layers; ++l)
    if (!x_all[l] || !w_qkv[l] || !aligned16(x_all[l]) || !aligned16(w_qkv[l])) return DLLM_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t out_layer = (size_t)B * beta * D * 2;
  int rc;
  for (int l = 0; l < n_layers; ++l) {
    void* out_l = static_cast<uint8_t*>(out) + l * out_layer;
    // 1. recompute every slot of this layer for the sequences whose drift test failed in
    //    a layer above (flags of layers 0 .. l-1, written by the launches before this one)
    if (l > 0) {
      StepArgs r{l, nullptr, w_qkv[l], nullptr, nullptr, 0, nullptr, x_all[l], nullptr, S, nullptr, s};
      r.kv_seq_flags = flags;
      r.n_flag_sets = l;
      rc = do_project(c, r);
      if (rc) return rc;
    }
    // 2. the tracked tokens: top-k of the previous step's mass outside the window
    rc = from_cuda((cudaError_t)launch_topk(mass + (size_t)l * B * S, B, S, win_lo, beta, k, ws.idx, s));
    if (rc) return rc;
    // 3. the rows the projection reads
    rc = from_cuda((cudaError_t)launch_gather_rows(x_all[l], B, S, D, win_lo, beta, ws.idx, k, ws.x_win, ws.x_trk,
                                                   ws.pos_win, c->status, s));
    if (rc) return rc;
    // 4. window rows -> cache slots and Q; tracked rows -> the drift test of this layer
    //    (fused into the projection: cosines and refresh flags, no probe buffer)
    StepArgs a{l, ws.x_win, w_qkv[l], ws.pos_win, nullptr, beta, out_l, ws.x_trk, ws.idx, k, nullptr, s};
    a.drift_cos = cos + (size_t)l * B * k * 2;
    a.drift_refresh = flags + (size_t)l * B;
    a.drift_gamma = gamma;
    rc = do_project(c, a);
    if (rc) return rc;
    // 5. this step's attention mass (the next step's top-k input), then the attention
    if (mass_out) {
      rc = dllm_attention_mass(c, l, ws.pos_win, nullptr, beta, out_l, mass_out + (size_t)l * B * S, stream);
      if (rc) return rc;
    }
    rc = do_attend(c, l, ws.pos_win, nullptr, beta, out_l, s);
    if (rc) return rc;
  }
  return DLLM_OK;
}

int dllm_selftest_fail_alloc(int nth) {
  if (nth < 0) return DLLM_EINVAL;
  std::lock_guard<std::mutex> lock(g_alloc_mu);
  g_fail_alloc_in = nth;
  return DLLM_OK;
}

int dllm_cache_status(dllm_cache* c, int* device_bits) {
  if (!c) return DLLM_EINVAL;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return from_cuda(e);
  int bits = 0;
  e = cudaMemcpy(&bits, c->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return from_cuda(e);
  e = cudaMemset(c->status, 0, sizeof(int));
  if (e != cudaSuccess) return from_cuda(e);
  if (bits & DLLM_DEV_TIMEOUT) {
    // a kernel that gave up may have left its arrival counters part-way: start them over
    e = cudaMemset(c->drift_cnt, 0, (size_t)c->desc.batch * sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(c->drift_acc, 0, c->drift_acc_bytes);
    if (e == cudaSuccess && c->merge_cnt) e = cudaMemset(c->merge_cnt, 0, (size_t)2 * c->sm_count * sizeof(int));
    if (e != cudaSuccess) return from_cuda(e);
  }
  if (device_bits) *device_bits = bits;
  return bits ? DLLM_EDEVICE : DLLM_OK;
}

const char* dllm_strerror(int s) {
  switch (s) {
    case DLLM_OK: return "ok";
    case DLLM_EINVAL: return "invalid argument";
    case DLLM_EOOM: return "out of device memory";
    case DLLM_ECUDA: return "CUDA error";
    case DLLM_EDEVICE: return "device-side range error or timeout (see status bits)";
    case DLLM_EUNSUPPORTED: return "unsupported configuration";
    default: return "unknown status";
  }
}

}  // extern "C"

// ------------------------------------------------------------------------------------
// dllm_cache_attend_noalloc: the attention half with its split-KV scratch in a static
// device array instead of the cache's workspace, so the call itself never allocates.
// ------------------------------------------------------------------------------------
namespace {

// Partial (O, m, l) states of the key splits.  One copy per device that loads this
// library, kept until the process exits.  Every call shares it: calls whose kernels
// overlap on the GPU race on it.  Nothing here has to start at zero, because the merge
// only reads partials that the same call wrote just before (the arrival counts that
// tell which CTA merges are the cache's own).
static __device__ __align__(256) float g_noalloc_scratch[DLLM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

constexpr int kMaxDevices = 256;
std::mutex g_noalloc_mu;
float* g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  Host code cannot use
// the symbol itself (it names a host-side shadow), so the address is looked up once
// per device, with that device current, and remembered.  A cudaDeviceReset() of the
// device discards the array with the rest of its memory and makes the remembered
// address stale; the public header tells callers not to use the entry point after one.
int noalloc_scratch_address(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return DLLM_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return from_cuda(e);
    g_noalloc_addr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_addr[dev];
  return DLLM_OK;
}

}  // namespace

// The same launches as dllm_cache_attend (same work split, so the same results), with
// the split-KV partials in g_noalloc_scratch instead of the cache's workspace.
extern "C" int dllm_cache_attend_noalloc(dllm_cache* c, int layer, const int32_t* positions, const uint8_t* view,
                                         int n_tok, void* out, void* stream) {
  int rc = check_attend(c, layer, n_tok, positions, view, out);
  if (rc) return rc;
  SplitScratch scratch;
  scratch.get = noalloc_scratch_address;
  scratch.floats = DLLM_NOALLOC_SCRATCH_BYTES / sizeof(float);
  return do_attend(c, layer, positions, view, n_tok, out, reinterpret_cast<cudaStream_t>(stream), KeyRange(),
                   scratch);
}
