// Host-side buffers of the end-to-end path: page-locked blocks that the copy engines
// read and write directly, and the staging copy that fills them with streaming stores.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#if defined(__x86_64__)
#include <emmintrin.h>
#endif

#include "../../include/dllm_cache.h"

namespace {

// Copy n bytes with 16-byte non-temporal stores (x86-64 SSE2), ordered by a store
// fence at the end; the unaligned head and tail of dst go through memcpy.
void stream_copy(char* dst, const char* src, size_t n) {
#if defined(__x86_64__)
  size_t head = (16 - (reinterpret_cast<uintptr_t>(dst) & 15u)) & 15u;
  if (head > n) head = n;
  std::memcpy(dst, src, head);
  dst += head;
  src += head;
  n -= head;
  const size_t vecs = n / 16;
  __m128i* d = reinterpret_cast<__m128i*>(dst);
  const __m128i* s = reinterpret_cast<const __m128i*>(src);
  size_t i = 0;
  for (; i + 4 <= vecs; i += 4) {
    const __m128i a = _mm_loadu_si128(s + i), b = _mm_loadu_si128(s + i + 1);
    const __m128i c = _mm_loadu_si128(s + i + 2), e = _mm_loadu_si128(s + i + 3);
    _mm_stream_si128(d + i, a);
    _mm_stream_si128(d + i + 1, b);
    _mm_stream_si128(d + i + 2, c);
    _mm_stream_si128(d + i + 3, e);
  }
  for (; i < vecs; ++i) _mm_stream_si128(d + i, _mm_loadu_si128(s + i));
  std::memcpy(dst + vecs * 16, src + vecs * 16, n - vecs * 16);
  _mm_sfence();
#else
  std::memcpy(dst, src, n);
#endif
}

}  // namespace

extern "C" {

int dllm_host_alloc(size_t bytes, void** out) {
  if (!out) return DLLM_EINVAL;
  *out = nullptr;
  if (bytes == 0) return DLLM_OK;
  void* p = nullptr;
  const cudaError_t e = cudaHostAlloc(&p, bytes, cudaHostAllocPortable);
  if (e != cudaSuccess) {
    cudaGetLastError();  // not sticky: clear it so that later calls do not see it
    return e == cudaErrorMemoryAllocation ? DLLM_EOOM : DLLM_ECUDA;
  }
  *out = p;
  return DLLM_OK;
}

int dllm_host_free(void* ptr) {
  if (!ptr) return DLLM_OK;
  if (cudaFreeHost(ptr) != cudaSuccess) {
    cudaGetLastError();
    return DLLM_ECUDA;
  }
  return DLLM_OK;
}

int dllm_host_stage(void* dst, const void* src, size_t bytes) {
  if (bytes == 0) return DLLM_OK;
  if (!dst || !src) return DLLM_EINVAL;
  const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
  if (d + bytes < d || s + bytes < s) return DLLM_EINVAL;  // wraps the address space
  if (d < s + bytes && s < d + bytes) return DLLM_EINVAL;  // overlapping ranges
  stream_copy(static_cast<char*>(dst), static_cast<const char*>(src), bytes);
  return DLLM_OK;
}

}  // extern "C"
