// Top-k most-attended positions and the K/V cosine-drift reduction.
//
// "Flash-dLLM ...", paragraph 4: a fixed budget of the 32 most-attended tokens carries
// about half of the attention mass in middle layers.  "Elastic-Cache", Core idea: the
// cosine similarity between the cached and the recomputed K/V of the previous step's
// most-attended tokens decides whether deeper layers are refreshed (gamma = 0.9 in
// Algorithm knobs).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace dllm {
namespace {

// Total order on candidates: mass first (order-preserving bits of the float), then the
// lower position (inverted index in the low word).  0 marks "no candidate".
__device__ __forceinline__ unsigned long long cand_key(float mass, int i) {
  const uint32_t u = __float_as_uint(mass);
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(ord) << 32) | static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(i));
}
__device__ __forceinline__ int cand_pos(unsigned long long key) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull));
}

__device__ __forceinline__ unsigned long long shfl_xor64(unsigned long long v, int m) {
  return __shfl_xor_sync(0xffffffffu, v, m);
}

// Sort one key per lane across the warp, descending (lane 0 largest): bitonic network.
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long v, int lane) {
#pragma unroll
  for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
      const unsigned long long o = shfl_xor64(v, j);
      const bool lower = (lane & j) == 0;       // this lane holds the first of the pair
      const bool desc = (lane & kk) == 0 || kk == 32;  // direction of this subsequence
      const bool keep_max = (lower == desc);
      v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// a: this warp's descending top-32 list; b: another descending list.  Returns the
// descending top 32 of their union (lane i gets max(a[i], b[31-i]), a bitonic
// sequence holding the top 32, then sorts it with the half-cleaner steps).
__device__ __forceinline__ unsigned long long warp_merge_top32(unsigned long long a, unsigned long long b_rev,
                                                               int lane) {
  unsigned long long v = a > b_rev ? a : b_rev;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const unsigned long long o = shfl_xor64(v, j);
    const bool lower = (lane & j) == 0;
    v = lower ? (v > o ? v : o) : (v < o ? v : o);
  }
  return v;
}

// k <= 32: blocks of 32 warps, `per_seq` of them per sequence.  Each warp keeps a
// descending top-32 list of its share of the positions (one key per lane), merging in 32
// new keys at a time; the 32 lists are then merged pairwise in shared memory.  The first
// block of a sequence writes its indices.  With x_all, each block then copies its share
// (every per_seq-th row) of the selected tokens' rows (row_vecs 16-byte vectors each)
// of the sequence's hidden states x_all[b][n_pos] into x_rows[b][k]; the selection is
// cheap, so the blocks of a sequence each make it rather than wait for one another.
__global__ void __launch_bounds__(1024) kv_topk32_kernel(const float* __restrict__ mass, int n_pos,
                                                         const int32_t* __restrict__ block_lo, int block_len, int k,
                                                         int32_t* __restrict__ idx, const uint4* __restrict__ x_all,
                                                         int row_vecs, uint4* __restrict__ x_rows, int per_seq) {
  __shared__ unsigned long long lists[32][32];
  __shared__ int sel[32];
  grid_dep_launch();
  grid_dep_wait();
  const int b = blockIdx.x / per_seq, part = blockIdx.x - b * per_seq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lo = block_lo[b];
  const float* mrow = mass + static_cast<size_t>(b) * n_pos;
  unsigned long long best = 0ull;
  for (int base = warp * 32; base < n_pos; base += 1024) {
    const int i = base + lane;
    unsigned long long key = 0ull;
    if (i < n_pos && !(i >= lo && i < lo + block_len)) key = cand_key(__ldg(mrow + i), i);
    key = warp_sort_desc(key, lane);
    best = warp_merge_top32(best, __shfl_sync(0xffffffffu, key, 31 - lane), lane);
  }
  lists[warp][lane] = best;
  __syncthreads();
  for (int step = 1; step < 32; step <<= 1) {
    if ((warp & (2 * step - 1)) == 0) {
      const unsigned long long other = lists[warp + step][31 - lane];
      best = warp_merge_top32(best, other, lane);
    }
    __syncthreads();
    if ((warp & (2 * step - 1)) == 0) lists[warp][lane] = best;
    __syncthreads();
  }
  if (warp == 0 && lane < k) {
    const int pos = cand_pos(best);
    if (part == 0) idx[static_cast<size_t>(b) * k + lane] = pos;
    sel[lane] = pos;
  }
  if (x_all == nullptr) return;
  __syncthreads();
  // this block's rows (j = part, part + per_seq, ...): eight 16-byte loads in flight per
  // thread before their stores
  const int my_rows = (k - part + per_seq - 1) / per_seq;
  const int total = my_rows * row_vecs;
  const uint4* src = x_all + static_cast<size_t>(b) * n_pos * row_vecs;
  uint4* dst = x_rows + static_cast<size_t>(b) * k * row_vecs;
  for (int i0 = threadIdx.x; i0 < total; i0 += 8 * blockDim.x) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < total) {
        const int row = part + (i / row_vecs) * per_seq, c = i % row_vecs;
        v[u] = __ldg(src + static_cast<size_t>(sel[row]) * row_vecs + c);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < total) {
        const int row = part + (i / row_vecs) * per_seq, c = i % row_vecs;
        dst[static_cast<size_t>(row) * row_vecs + c] = v[u];
      }
    }
  }
}

// General k: one block per sequence, bitonic sort (descending) of all keys in shared
// memory; positions inside the active block get key 0 and sink to the end.
__global__ void __launch_bounds__(1024) kv_topk_kernel(const float* __restrict__ mass, int n_pos,
                                                       const int32_t* __restrict__ block_lo, int block_len, int k,
                                                       int n, int32_t* __restrict__ idx) {
  extern __shared__ unsigned long long keys[];
  grid_dep_launch();
  grid_dep_wait();
  const int b = blockIdx.x;
  const int lo = block_lo[b];
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    unsigned long long key = 0ull;
    if (i < n_pos && !(i >= lo && i < lo + block_len)) key = cand_key(mass[static_cast<size_t>(b) * n_pos + i], i);
    keys[i] = key;
  }
  __syncthreads();
  for (int kk = 2; kk <= n; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = keys[i], c = keys[ixj];
          const bool desc = (i & kk) == 0;
          if (desc ? (a < c) : (a > c)) {
            keys[i] = c;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < k; i += blockDim.x) idx[static_cast<size_t>(b) * k + i] = cand_pos(keys[i]);
}

// ------------------------------------------------------------------------------ drift
constexpr int kDriftWarps = 16;  // warps per block; one tracked row (token, K|V) per warp at a time
// 8-element units a lane loads before reducing them (fp32 units take twice the registers)
template <int KV>
constexpr int drift_batch() { return KV == DLLM_F32 ? 4 : 8; }

// 8 consecutive elements of a cache row (dequantised) and of a probe row, as fp32.
template <int KV>
struct Unit8 {
  uint4 c0, c1;  // cache: bf16 (c0) / fp32 (c0, c1) / e4m3 (c0.x, c0.y)
  uint4 p0, p1;  // probe: bf16 (p0) / fp32 (p0, p1)
};

template <int KV>
__device__ __forceinline__ void load_unit(Unit8<KV>& u, const void* crow, const void* prow, int e) {
  if (KV == DLLM_BF16) {
    u.c0 = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(crow) + e));
    u.p0 = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(prow) + e));
  } else if (KV == DLLM_F32) {
    const uint4* c = reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(crow) + e);
    const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(prow) + e);
    u.c0 = __ldg(c);
    u.c1 = __ldg(c + 1);
    u.p0 = __ldg(q);
    u.p1 = __ldg(q + 1);
  } else {
    const uint2 c = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(crow) + e));
    u.c0 = make_uint4(c.x, c.y, 0u, 0u);
    u.p0 = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(prow) + e));
  }
}

__device__ __forceinline__ void bf16x8(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

template <int KV>
__device__ __forceinline__ void accumulate(const Unit8<KV>& u, float scale, float& dot, float& nc, float& np) {
  float c[8], q[8];
  if (KV == DLLM_BF16) {
    bf16x8(u.c0, c);
    bf16x8(u.p0, q);
  } else if (KV == DLLM_F32) {
    c[0] = __uint_as_float(u.c0.x); c[1] = __uint_as_float(u.c0.y);
    c[2] = __uint_as_float(u.c0.z); c[3] = __uint_as_float(u.c0.w);
    c[4] = __uint_as_float(u.c1.x); c[5] = __uint_as_float(u.c1.y);
    c[6] = __uint_as_float(u.c1.z); c[7] = __uint_as_float(u.c1.w);
    q[0] = __uint_as_float(u.p0.x); q[1] = __uint_as_float(u.p0.y);
    q[2] = __uint_as_float(u.p0.z); q[3] = __uint_as_float(u.p0.w);
    q[4] = __uint_as_float(u.p1.x); q[5] = __uint_as_float(u.p1.y);
    q[6] = __uint_as_float(u.p1.z); q[7] = __uint_as_float(u.p1.w);
  } else {
    const uint8_t* bytes = reinterpret_cast<const uint8_t*>(&u.c0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(bytes[i]), __NV_E4M3);
      c[i] = __half2float(__half(hr)) * scale;
    }
    bf16x8(u.p0, q);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    dot = fmaf(c[i], q[i], dot);
    nc = fmaf(c[i], c[i], nc);
    np = fmaf(q[i], q[i], np);
  }
}

// Grid (blocks_per_seq, B).  Warp w of block x handles tracked rows r = (x * 16 + w),
// r + 16 * blocks_per_seq, ... of its sequence (row r = token r / 2, K if r is even
// else V): fp32 dot product and norms over the full D-vector, many loads in flight.
// The last block of a sequence to finish (arrival counter) takes the minimum over the
// sequence's cosines and writes the refresh flag, then resets the counter.
template <int KV>
__global__ void __launch_bounds__(kDriftWarps * 32) kv_drift_kernel(
    const void* __restrict__ kv, const float* __restrict__ scale, int slots, int max_pos, int H, int hd, int D,
    const int32_t* __restrict__ idx, int k, const void* __restrict__ probe, float gamma, float* __restrict__ cos,
    int32_t* __restrict__ refresh, int* __restrict__ counters, int* status) {
  grid_dep_launch();
  grid_dep_wait();
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int eb = KV == DLLM_F32 ? 4 : (KV == DLLM_BF16 ? 2 : 1);
  const int n_units = D / 8;
  for (int row = blockIdx.x * kDriftWarps + warp; row < 2 * k; row += gridDim.x * kDriftWarps) {
    const int j = row >> 1, which = row & 1;
    const int slot = idx[static_cast<size_t>(b) * k + j];
    const size_t prow_i = (static_cast<size_t>(b) * k + j) * 2 + which;
    if (slot < 0 || slot >= max_pos) {
      if (lane == 0) {
        atomicOr(status, DLLM_DEV_BAD_INDEX);
        cos[prow_i] = __int_as_float(0x7fc00000);
      }
      continue;
    }
    const size_t crow_i = (static_cast<size_t>(b) * slots + slot) * 2 + which;
    const void* crow = reinterpret_cast<const uint8_t*>(kv) + crow_i * D * eb;
    const void* prow = reinterpret_cast<const uint8_t*>(probe) + prow_i * D * (KV == DLLM_F32 ? 4 : 2);
    float dot = 0.0f, nc = 0.0f, np = 0.0f;
    constexpr int NB = drift_batch<KV>();
    for (int u0 = 0; u0 < n_units; u0 += 32 * NB) {
      Unit8<KV> un[NB];
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int unit = u0 + i * 32 + lane;
        if (unit < n_units) load_unit<KV>(un[i], crow, prow, unit * 8);
      }
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int unit = u0 + i * 32 + lane;
        if (unit < n_units) {
          const float sc = KV == DLLM_E4M3 ? __ldg(scale + crow_i * H + (unit * 8) / hd) : 1.0f;
          accumulate<KV>(un[i], sc, dot, nc, np);
        }
      }
    }
    if (KV == DLLM_F32) {  // D % 8 == 4 leaves a tail of 4 elements
      const float* c = reinterpret_cast<const float*>(crow);
      const float* q = reinterpret_cast<const float*>(prow);
      for (int e = n_units * 8 + lane; e < D; e += 32) {
        const float cv = __ldg(c + e), qv = __ldg(q + e);
        dot = fmaf(cv, qv, dot);
        nc = fmaf(cv, cv, nc);
        np = fmaf(qv, qv, np);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      dot += __shfl_xor_sync(0xffffffffu, dot, o);
      nc += __shfl_xor_sync(0xffffffffu, nc, o);
      np += __shfl_xor_sync(0xffffffffu, np, o);
    }
    if (lane == 0) {
      const float den = sqrtf(nc) * sqrtf(np);
      cos[prow_i] = den > 0.0f ? dot / den : 0.0f;
      __threadfence();  // visible to the block of this sequence that sets the flag
    }
  }
  if (refresh == nullptr) return;
  // ---- the sequence's last block sets the refresh flag (min cos < gamma)
  __shared__ int last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(counters + b, 1);
    last = (old == static_cast<int>(gridDim.x) - 1);
    if (last) {
      atomicExch(counters + b, 0);
      __threadfence();
    }
  }
  __syncthreads();
  if (last && warp == 0) {
    float mn = INFINITY;
    for (int i = lane; i < 2 * k; i += 32) mn = fminf(mn, __ldcg(cos + static_cast<size_t>(b) * 2 * k + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    if (lane == 0) refresh[b] = (mn < gamma) ? 1 : 0;
  }
}

}  // namespace

int launch_topk(const float* mass, int batch, int n_pos, const int32_t* block_lo, int block_len, int k, int32_t* idx,
                cudaStream_t s) {
  if (k <= 32) {
    return (int)launch_pdl(kv_topk32_kernel, dim3(batch), dim3(1024), 0, s, mass, n_pos, block_lo, block_len, k, idx,
                           static_cast<const uint4*>(nullptr), 0, static_cast<uint4*>(nullptr), 1);
  }
  int n = 1;
  while (n < n_pos) n <<= 1;
  const size_t smem = static_cast<size_t>(n) * 8;
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kv_topk_kernel), (int)(smem));
    if (e != cudaSuccess) return (int)e;
  }
  const int threads = n < 1024 ? (n < 32 ? 32 : n) : 1024;
  return (int)launch_pdl(kv_topk_kernel, dim3(batch), dim3(threads), smem, s, mass, n_pos, block_lo, block_len, k, n,
                         idx);
}

int launch_topk_gather(const float* mass, int batch, int n_pos, const int32_t* block_lo, int block_len, int k,
                       int32_t* idx, const void* x_all, int row_vecs, void* x_rows, cudaStream_t s) {
  // four blocks per sequence (each makes the selection and copies a quarter of the rows),
  // so the copy spreads over four times as many SMs
  const int per_seq = k < 4 ? k : 4;
  return (int)launch_pdl(kv_topk32_kernel, dim3(batch * per_seq), dim3(1024), 0, s, mass, n_pos, block_lo, block_len,
                         k, idx, static_cast<const uint4*>(x_all), row_vecs, static_cast<uint4*>(x_rows), per_seq);
}

int launch_drift(const void* kv_layer, const float* scale_layer, int kv_dtype, int B, int slots, int max_pos, int H,
                 int hd, const int32_t* idx, int k, const void* probe, float gamma, float* cos, int32_t* refresh,
                 int* counters, int sm_count, int* status, cudaStream_t s) {
  const int D = H * hd;
  // spread each sequence's 2k rows over enough blocks to keep most SMs streaming
  int per_seq = (sm_count + B - 1) / B;
  const int max_per_seq = (2 * k + kDriftWarps - 1) / kDriftWarps;
  if (per_seq > max_per_seq) per_seq = max_per_seq;
  if (per_seq < 1) per_seq = 1;
  dim3 grid(per_seq, B);
  constexpr int threads = kDriftWarps * 32;
  auto kern = kv_drift_kernel<DLLM_F32>;
  if (kv_dtype == DLLM_BF16) kern = kv_drift_kernel<DLLM_BF16>;
  else if (kv_dtype == DLLM_E4M3) kern = kv_drift_kernel<DLLM_E4M3>;
  return (int)launch_pdl(kern, grid, dim3(threads), 0, s, kv_layer, scale_layer, slots, max_pos, H, hd, D, idx, k,
                         probe, gamma, cos, refresh, counters, status);
}

}  // namespace dllm
