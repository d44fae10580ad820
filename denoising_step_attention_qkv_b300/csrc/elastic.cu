// Row gather of the multi-layer refresh step ("Elastic-Cache ...", Core idea: a
// sliding window of active tokens decodes while the most-attended tokens outside it
// are tracked for drift).  Given one layer's hidden states of every position this
// step, it collects the rows the fused projection reads: the window rows (which also
// get their positions) and the tracked rows chosen by the top-k.  A pure copy: 16-byte
// loads and stores, one block per row.
#include "internal.h"
#include "ptx.cuh"

namespace dllm {
namespace {

__device__ __forceinline__ void raise_bits(int* status, int bits) { atomicOr(status, bits); }

// Block r < B * beta copies window row (b, t) = (r / beta, r % beta); the next B * k
// blocks copy tracked row (b, j).  A window that does not fit the sequence gives zero
// rows and raises DLLM_DEV_BAD_POSITION; a tracked position outside it, a zero row and
// DLLM_DEV_BAD_INDEX.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x_all, int S, int row_vecs,
                                                           const int32_t* __restrict__ win_lo, int beta,
                                                           const int32_t* __restrict__ idx, int k, int B,
                                                           uint4* __restrict__ x_win, uint4* __restrict__ x_trk,
                                                           int32_t* __restrict__ pos_win, int* status) {
  grid_dep_launch();
  grid_dep_wait();
  const int r = blockIdx.x;
  int b, pos, bad_bit;
  uint4* dst;
  if (r < B * beta) {
    b = r / beta;
    const int t = r - b * beta;
    pos = __ldg(win_lo + b) + t;
    dst = x_win + static_cast<size_t>(r) * row_vecs;
    bad_bit = DLLM_DEV_BAD_POSITION;
    if (threadIdx.x == 0) pos_win[r] = pos;
  } else {
    const int j = r - B * beta;
    b = j / k;
    pos = __ldg(idx + j);
    dst = x_trk + static_cast<size_t>(j) * row_vecs;
    bad_bit = DLLM_DEV_BAD_INDEX;
  }
  const bool ok = pos >= 0 && pos < S;
  if (!ok && threadIdx.x == 0) raise_bits(status, bad_bit);
  const uint4* src = x_all + (static_cast<size_t>(b) * S + (ok ? pos : 0)) * row_vecs;
  for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) dst[i] = ok ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
}

}  // namespace

int launch_gather_rows(const void* x_all, int B, int S, int D, const int32_t* win_lo, int beta, const int32_t* idx,
                       int k, void* x_win, void* x_trk, int32_t* pos_win, int* status, cudaStream_t s) {
  const int rows = B * (beta + k);
  if (rows == 0) return 0;
  return (int)launch_pdl(gather_rows_kernel, dim3(rows), dim3(256), 0, s, static_cast<const uint4*>(x_all), S,
                         D * 2 / 16, win_lo, beta, idx, k, B, static_cast<uint4*>(x_win), static_cast<uint4*>(x_trk),
                         pos_win, status);
}

}  // namespace dllm
