// The conventional per-layer cache pipeline, kept as a comparison for the fused
// kernel ("Flash-dLLM ...", paragraph 2: QKV projection, rotary embedding, cache write
// and attention as four kernels, each writing its intermediates to HBM for the next).
// Stage 1 is the projection GEMM storing its plain output (bf16; fp32 for an e4m3
// cache, which is quantised from the unrounded rotated value as in the fused kernel);
// the two kernels here are stages 2 and 3; stage 4 is the same attention kernel as the
// fused path.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace dllm {
namespace {

// Raw projection values: T is float (fp32 workspace) or __nv_bfloat16.
DEVI float to_f(float v) { return v; }
DEVI float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
DEVI void from_f(float& d, float v) { d = v; }
DEVI void from_f(__nv_bfloat16& d, float v) { d = __float2bfloat16_rn(v); }

// Stage 2: one block per (row, head), one thread per rotary pair.  Query rows: rotate
// Q into q_out (bf16) and K in place; K/V-only rows: rotate K in place.  Rows whose
// position is out of range are left alone (stage 3 reports them).
template <typename T>
__global__ void __launch_bounds__(kHd / 2) rope_rows_kernel(const ProjParams p) {
  const int row = blockIdx.x;
  const int h = blockIdx.y;
  const int i = threadIdx.x;
  const bool q_row = row < p.m_q;
  const int m = q_row ? row : row - p.m_q;
  const int pos = q_row ? p.positions[m] : p.kv_positions[m];
  if (pos < 0 || pos >= p.max_pos) return;
  const float2 cs = p.rope[static_cast<size_t>(pos) * (kHd / 2) + i];
  auto rotate = [&](const T* src, auto* dst) {
    const float a = to_f(src[i]), b = to_f(src[i + kHd / 2]);
    from_f(dst[i], a * cs.x - b * cs.y);
    from_f(dst[i + kHd / 2], b * cs.x + a * cs.y);
  };
  if (q_row) {
    T* rowp = static_cast<T*>(p.raw_q) + static_cast<size_t>(m) * 3 * p.D;
    rotate(rowp + h * kHd, reinterpret_cast<__nv_bfloat16*>(p.q_out) + static_cast<size_t>(m) * p.D + h * kHd);
    rotate(rowp + p.D + h * kHd, rowp + p.D + h * kHd);
  } else {
    T* rowp = static_cast<T*>(p.raw_kv) + static_cast<size_t>(m) * 2 * p.D;
    rotate(rowp + h * kHd, rowp + h * kHd);
  }
}

// Four consecutive raw values of a head, as floats (16-byte fp32 or 8-byte bf16 load).
DEVI float4 load4(const float* src) { return *reinterpret_cast<const float4*>(src); }
DEVI float4 load4(const __nv_bfloat16* src) {
  const uint2 raw = *reinterpret_cast<const uint2*>(src);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

DEVI uint2 pack_bf16x4(float4 f) {
  __nv_bfloat162 a = __floats2bfloat162_rn(f.x, f.y), b = __floats2bfloat162_rn(f.z, f.w);
  return make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}

// Stage 3: one warp per (row, K|V, head): copy the rotated K (or V) head to the row's
// cache slot (bf16, or e4m3 with scale amax/448), or to the probe rows (bf16).
template <typename T>
__global__ void __launch_bounds__(256) cache_write_kernel(const ProjParams p) {
  const int warp_global = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int per_row = 2 * p.H;
  const int row = warp_global / per_row;
  if (row >= p.m_q + p.m_kv) return;
  const int part = (warp_global % per_row) / p.H;  // 0 K, 1 V
  const int h = warp_global % p.H;
  const bool q_row = row < p.m_q;
  const int m = q_row ? row : row - p.m_q;
  int b, pos, slot;
  bool valid = true;
  if (q_row) {
    b = m / p.n_tok;
    pos = p.positions[m];
    slot = pos;
    const int v = p.view ? static_cast<int>(p.view[m]) : DLLM_VIEW_BASE;
    if (v > DLLM_VIEW_MASK) {
      if (part == 0 && h == 0 && lane == 0) atomicOr(p.status, DLLM_DEV_BAD_VIEW);
      valid = false;
    } else if (v == DLLM_VIEW_DRAFT) {
      int rank = 0;
      for (int t = b * p.n_tok; t < m; ++t) rank += (p.view[t] == DLLM_VIEW_DRAFT);
      if (rank >= p.tail) {
        if (part == 0 && h == 0 && lane == 0) atomicOr(p.status, DLLM_DEV_TAIL_FULL);
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
    if (part == 0 && h == 0 && lane == 0) atomicOr(p.status, DLLM_DEV_BAD_POSITION);
    valid = false;
  }
  if (!valid) return;
  const T* src = q_row ? static_cast<const T*>(p.raw_q) + static_cast<size_t>(m) * 3 * p.D + (1 + part) * p.D + h * kHd
                       : static_cast<const T*>(p.raw_kv) + static_cast<size_t>(m) * 2 * p.D + part * p.D + h * kHd;
  // each lane holds 4 consecutive values
  const float4 f = load4(src + 4 * lane);
  if (!q_row && p.probe != nullptr) {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.probe) + (static_cast<size_t>(m) * 2 + part) * p.D + h * kHd;
    reinterpret_cast<uint2*>(dst)[lane] = pack_bf16x4(f);
    return;
  }
  const size_t crow = (static_cast<size_t>(b) * p.slots + slot) * 2 + part;
  if (p.kv_dtype == DLLM_E4M3) {
    float amax = fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w)));
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    const __nv_fp8x2_storage_t q0 =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t q1 =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(f.z, scale), __fdiv_rn(f.w, scale)), __NV_SATFINITE, __NV_E4M3);
    uint8_t* dst = reinterpret_cast<uint8_t*>(p.cache_kv) + crow * p.D + h * kHd;
    reinterpret_cast<uint32_t*>(dst)[lane] = static_cast<uint32_t>(q0) | (static_cast<uint32_t>(q1) << 16);
    if (lane == 0) p.cache_scale[crow * p.H + h] = scale;
  } else {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.cache_kv) + crow * p.D + h * kHd;
    reinterpret_cast<uint2*>(dst)[lane] = pack_bf16x4(f);
  }
}

}  // namespace

int launch_rope_rows(const ProjParams& p, cudaStream_t s) {
  const int rows = p.m_q + p.m_kv;
  if (rows == 0) return 0;
  if (p.raw_f32)
    rope_rows_kernel<float><<<dim3(rows, p.H), kHd / 2, 0, s>>>(p);
  else
    rope_rows_kernel<__nv_bfloat16><<<dim3(rows, p.H), kHd / 2, 0, s>>>(p);
  return (int)cudaGetLastError();
}

int launch_cache_write(const ProjParams& p, cudaStream_t s) {
  const long long warps = static_cast<long long>(p.m_q + p.m_kv) * 2 * p.H;
  if (warps == 0) return 0;
  if (p.raw_f32)
    cache_write_kernel<float><<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(p);
  else
    cache_write_kernel<__nv_bfloat16><<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace dllm
