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

namespace dllm {
namespace {

__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One block per sequence: bitonic sort (descending) of 64-bit keys
// (order-preserving mass bits, inverted position) in shared memory; positions inside
// the active block get key 0 and sink to the end.
__global__ void __launch_bounds__(1024) kv_topk_kernel(const float* __restrict__ mass, int n_pos,
                                                       const int32_t* __restrict__ block_lo, int block_len, int k,
                                                       int n, int32_t* __restrict__ idx) {
  extern __shared__ unsigned long long keys[];
  const int b = blockIdx.x;
  const int lo = block_lo[b];
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    unsigned long long key = 0ull;
    if (i < n_pos && !(i >= lo && i < lo + block_len)) {
      key = (static_cast<unsigned long long>(ordered_bits(mass[static_cast<size_t>(b) * n_pos + i])) << 32) |
            static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(i));
    }
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
  for (int i = threadIdx.x; i < k; i += blockDim.x)
    idx[static_cast<size_t>(b) * k + i] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(keys[i] & 0xFFFFFFFFull));
}

template <int KV>
__device__ __forceinline__ void load8(const void* base, size_t e, float (&f)[16], int& n) {
  if (KV == DLLM_BF16) {
    const uint4 v = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + e);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
    n = 8;
  } else if (KV == DLLM_F32) {
    const float4 v = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + e);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    n = 4;
  }
}

// One warp per (sequence, tracked token, K|V): fp32 dot product and norms over the
// full D-vector of the cached row and the probe row.
template <int KV>
__global__ void __launch_bounds__(256) kv_drift_kernel(const void* __restrict__ kv, const float* __restrict__ scale,
                                                       int slots, int max_pos, int H, int hd, int D,
                                                       const int32_t* __restrict__ idx, int k,
                                                       const void* __restrict__ probe, float* __restrict__ cos,
                                                       int* status) {
  const int b = blockIdx.y;
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= 2 * k) return;
  const int j = wid >> 1, which = wid & 1;
  const int slot = idx[static_cast<size_t>(b) * k + j];
  if (slot < 0 || slot >= max_pos) {
    if (lane == 0) {
      atomicOr(status, DLLM_DEV_BAD_INDEX);
      cos[(static_cast<size_t>(b) * k + j) * 2 + which] = __int_as_float(0x7fc00000);
    }
    return;
  }
  const size_t crow = (static_cast<size_t>(b) * slots + slot) * 2 + which;
  const size_t prow = (static_cast<size_t>(b) * k + j) * 2 + which;
  float dot = 0.0f, nc = 0.0f, np = 0.0f;
  if (KV == DLLM_E4M3) {
    // 16 codes per lane per step; probe is bf16
    const uint8_t* c8 = reinterpret_cast<const uint8_t*>(kv) + crow * D;
    const __nv_bfloat16* pb = reinterpret_cast<const __nv_bfloat16*>(probe) + prow * D;
    for (int e = lane * 16; e < D; e += 32 * 16) {
      const float sc = scale[crow * H + e / hd];
      const uint4 raw = *reinterpret_cast<const uint4*>(c8 + e);
      const uint8_t* bytes = reinterpret_cast<const uint8_t*>(&raw);
      const uint4 p0 = *reinterpret_cast<const uint4*>(pb + e);
      const uint4 p1 = *reinterpret_cast<const uint4*>(pb + e + 8);
      const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&p0);
      const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&p1);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(bytes[i]), __NV_E4M3);
        const float c = __half2float(__half(hr)) * sc;
        const float2 pp = __bfloat1622float2(i < 8 ? h0[i >> 1] : h1[(i - 8) >> 1]);
        const float pv = (i & 1) ? pp.y : pp.x;
        dot = fmaf(c, pv, dot);
        nc = fmaf(c, c, nc);
        np = fmaf(pv, pv, np);
      }
    }
  } else {
    constexpr int V = (KV == DLLM_BF16) ? 8 : 4;
    for (int e = lane * V; e < D; e += 32 * V) {
      float c[16], pv[16];
      int n;
      load8<KV>(kv, crow * D + e, c, n);
      load8<KV>(probe, prow * D + e, pv, n);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        dot = fmaf(c[i], pv[i], dot);
        nc = fmaf(c[i], c[i], nc);
        np = fmaf(pv[i], pv[i], np);
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    dot += __shfl_xor_sync(0xffffffffu, dot, o);
    nc += __shfl_xor_sync(0xffffffffu, nc, o);
    np += __shfl_xor_sync(0xffffffffu, np, o);
  }
  if (lane == 0) {
    const float den = sqrtf(nc) * sqrtf(np);
    cos[prow] = den > 0.0f ? dot / den : 0.0f;
  }
}

__global__ void refresh_kernel(const float* __restrict__ cos, int k, float gamma, int32_t* __restrict__ refresh) {
  const int b = blockIdx.x;
  float mn = INFINITY;
  for (int i = threadIdx.x; i < 2 * k; i += 32) mn = fminf(mn, cos[static_cast<size_t>(b) * 2 * k + i]);
  for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  if (threadIdx.x == 0) refresh[b] = (mn < gamma) ? 1 : 0;
}

}  // namespace

int launch_topk(const float* mass, int batch, int n_pos, const int32_t* block_lo, int block_len, int k, int32_t* idx,
                cudaStream_t s) {
  int n = 1;
  while (n < n_pos) n <<= 1;
  const size_t smem = static_cast<size_t>(n) * 8;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kv_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
  }
  const int threads = n < 1024 ? (n < 32 ? 32 : n) : 1024;
  kv_topk_kernel<<<batch, threads, smem, s>>>(mass, n_pos, block_lo, block_len, k, n, idx);
  return (int)cudaGetLastError();
}

int launch_drift(const void* kv_layer, const float* scale_layer, int kv_dtype, int B, int slots, int max_pos, int H,
                 int hd, const int32_t* idx, int k, const void* probe, float gamma, float* cos, int32_t* refresh,
                 int* status, cudaStream_t s) {
  const int D = H * hd;
  dim3 grid((2 * k + 7) / 8, B);
  if (kv_dtype == DLLM_BF16)
    kv_drift_kernel<DLLM_BF16><<<grid, 256, 0, s>>>(kv_layer, scale_layer, slots, max_pos, H, hd, D, idx, k, probe, cos, status);
  else if (kv_dtype == DLLM_E4M3)
    kv_drift_kernel<DLLM_E4M3><<<grid, 256, 0, s>>>(kv_layer, scale_layer, slots, max_pos, H, hd, D, idx, k, probe, cos, status);
  else
    kv_drift_kernel<DLLM_F32><<<grid, 256, 0, s>>>(kv_layer, scale_layer, slots, max_pos, H, hd, D, idx, k, probe, cos, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  if (refresh) {
    refresh_kernel<<<B, 32, 0, s>>>(cos, k, gamma, refresh);
    e = cudaGetLastError();
  }
  return (int)e;
}

}  // namespace dllm
