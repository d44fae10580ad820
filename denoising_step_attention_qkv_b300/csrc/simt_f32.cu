// fp32 path (DLLM_F32 caches): the same step with CUDA-core fp32 arithmetic.
//
// The tensor-core kinds that accept fp32 operands round them to a 10-bit mantissa,
// which does not meet a 1e-4 relative bound, so the fp32 step runs on the FMA pipes.
// It serves small layers (the tiny fp32 workload has a 256-wide model); the pipeline
// order and the slot/visibility rules are those of the tensor-core path
// ("Flash-dLLM ...", paragraphs 2 and 3).
#include "internal.h"

namespace dllm {
namespace {

// One block per (row, part, head); one thread per rotary pair index i (< hd/2): the
// thread computes features i and i + hd/2 of that head, so the pair is rotated in
// registers before the store.
__global__ void proj_rope_store_f32(const ProjParams p, const float* __restrict__ x, const float* __restrict__ xkv,
                                    const float* __restrict__ w, int hd) {
  const int m_all = blockIdx.x;  // query rows first, then K/V-only rows
  const int grp = m_all >= p.m_q;
  const int m = grp ? m_all - p.m_q : m_all;
  const int parts = grp ? 2 : 3;
  const int ph = blockIdx.y;
  if (ph >= parts * p.H) return;
  const int part = (grp ? 1 : 0) + ph / p.H;
  const int h = ph % p.H;
  const int i = threadIdx.x;
  const int half = hd / 2;
  if (i >= half) return;

  int b, pos, slot = 0;
  bool valid = true;
  if (!grp) {
    b = m / p.n_tok;
    pos = p.positions[m];
    slot = pos;
    const int v = p.view ? p.view[m] : DLLM_VIEW_BASE;
    if (v > DLLM_VIEW_MASK) {
      if (ph == 0 && i == 0) atomicOr(p.status, DLLM_DEV_BAD_VIEW);
      valid = false;
    } else if (v == DLLM_VIEW_DRAFT) {
      int rank = 0;
      for (int t = b * p.n_tok; t < m; ++t) rank += (p.view[t] == DLLM_VIEW_DRAFT);
      if (rank >= p.tail) {
        if (ph == 0 && i == 0) atomicOr(p.status, DLLM_DEV_TAIL_FULL);
        valid = false;
      }
      slot = p.max_pos + rank;
    }
  } else {
    b = m / p.n_kv;
    pos = p.kv_positions[m];
    slot = pos;
  }
  if (valid && (pos < 0 || pos >= p.max_pos)) {
    if (ph == 0 && i == 0) atomicOr(p.status, DLLM_DEV_BAD_POSITION);
    valid = false;
  }
  if (!valid) return;

  const float* xr = (grp ? xkv : x) + static_cast<size_t>(m) * p.D;
  const size_t n_lo = static_cast<size_t>(part) * p.D + h * hd + i;
  const float* w_lo = w + n_lo * p.D;
  const float* w_hi = w + (n_lo + half) * p.D;
  float lo = 0.0f, hi = 0.0f;
  for (int c = 0; c < p.D; ++c) {
    const float xv = __ldg(xr + c);
    lo = fmaf(xv, __ldg(w_lo + c), lo);
    hi = fmaf(xv, __ldg(w_hi + c), hi);
  }
  if (part < 2) {
    const float2 cs = p.rope[static_cast<size_t>(pos) * half + i];
    const float a = lo, bb = hi;
    lo = a * cs.x - bb * cs.y;
    hi = bb * cs.x + a * cs.y;
  }
  float* dst;
  if (part == 0) {
    dst = reinterpret_cast<float*>(p.q_out) + static_cast<size_t>(m) * p.D + h * hd;
  } else if (grp && p.probe) {
    dst = reinterpret_cast<float*>(p.probe) + (static_cast<size_t>(m) * 2 + (part - 1)) * p.D + h * hd;
  } else {
    dst = reinterpret_cast<float*>(p.cache_kv) + ((static_cast<size_t>(b) * p.slots + slot) * 2 + (part - 1)) * p.D + h * hd;
  }
  dst[i] = lo;
  dst[i + half] = hi;
}

// One block per (query row, head).  Scores of every slot go to shared memory; the
// softmax is the two-pass form (max, then exp and sum) in fp32.
__global__ void attn_f32(const AttnParams p, const float* __restrict__ kv, int hd) {
  extern __shared__ float sm[];
  const int row = blockIdx.x;  // b * n_tok + t
  const int h = blockIdx.y;
  const int b = row / p.n_tok;
  const int row0 = b * p.n_tok;
  const int n_keys = p.max_pos + (p.view ? p.tail : 0);
  float* q = sm;            // [hd]
  float* sc = sm + hd;      // [n_keys]
  float* red = sc + n_keys; // [32]
  float* out = reinterpret_cast<float*>(p.out) + static_cast<size_t>(row) * p.D + h * hd;
  for (int i = threadIdx.x; i < hd; i += blockDim.x) q[i] = out[i];

  int qview = DLLM_VIEW_BASE, n_draft = 0;
  if (p.view) {
    qview = p.view[row];
    for (int t = 0; t < p.n_tok; ++t) n_draft += (p.view[row0 + t] == DLLM_VIEW_DRAFT);
    n_draft = min(n_draft, p.tail);
  }
  __syncthreads();

  const float scale = rsqrtf(static_cast<float>(hd));
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < n_keys; j += blockDim.x) {
    bool vis;
    if (j < p.max_pos) {
      bool is_mask = false;
      if (p.view) {
        for (int t = 0; t < p.n_tok; ++t)
          if (p.view[row0 + t] == DLLM_VIEW_MASK && p.positions[row0 + t] == j) is_mask = true;
      }
      vis = !is_mask || qview != DLLM_VIEW_DRAFT;
    } else {
      vis = (j < p.max_pos + n_draft) && qview == DLLM_VIEW_DRAFT;
    }
    float s = -INFINITY;
    if (vis) {
      const float* k = kv + ((static_cast<size_t>(b) * p.slots + j) * 2) * p.D + h * hd;
      float acc = 0.0f;
      for (int i = 0; i < hd; ++i) acc = fmaf(q[i], k[i], acc);
      s = acc * scale;
    }
    sc[j] = s;
    mx = fmaxf(mx, s);
  }
  // block max
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : -INFINITY;
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float m = red[0];
  __syncthreads();
  float sum = 0.0f;
  for (int j = threadIdx.x; j < n_keys; j += blockDim.x) {
    const float e = (sc[j] == -INFINITY) ? 0.0f : expf(sc[j] - m);
    sc[j] = e;
    sum += e;
  }
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float l = red[0];
  for (int i = threadIdx.x; i < hd; i += blockDim.x) {
    float acc = 0.0f;
    for (int j = 0; j < n_keys; ++j) {
      const float e = sc[j];
      if (e != 0.0f) acc = fmaf(e, kv[((static_cast<size_t>(b) * p.slots + j) * 2 + 1) * p.D + h * hd + i], acc);
    }
    out[i] = l > 0.0f ? acc / l : 0.0f;
  }
}

}  // namespace

int launch_proj_f32(const ProjParams& p, const float* x, const float* xkv, const float* w, int hd, cudaStream_t s) {
  const int rows = p.m_q + p.m_kv;
  if (rows == 0) return 0;
  dim3 grid(rows, 3 * p.H);
  proj_rope_store_f32<<<grid, hd / 2, 0, s>>>(p, x, xkv, w, hd);
  return (int)cudaGetLastError();
}

int launch_attn_f32(const AttnParams& p, const float* kv_layer, int hd, cudaStream_t s) {
  const int n_keys = p.max_pos + (p.view ? p.tail : 0);
  const size_t smem = (static_cast<size_t>(hd) + n_keys + 32) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(attn_f32), (int)(smem));
    if (e != cudaSuccess) return (int)e;
  }
  dim3 grid(p.B * p.n_tok, p.H);
  attn_f32<<<grid, 128, smem, s>>>(p, kv_layer, hd);
  return (int)cudaGetLastError();
}

}  // namespace dllm
