// Attention mass per cached position: for every sequence and regular slot j, the sum
// over heads and query rows of the softmax weight that key j receives in this step.
// "Flash-dLLM ...", paragraph 4 keeps the 32 most-attended tokens; "Elastic-Cache",
// Core idea tests the drift of the previous step's most-attended tokens.  This kernel
// produces the mass that the next step's top-k reads.
//
// Design (sm_103a).  A work unit is (sequence, head, chunk of <= NQ query rows) on a
// persistent CTA.  The MMA warp computes S^T = K Q^T per 128-key tile with tcgen05
// (M = 128 keys, N = NQ queries) into TMEM, twice over the unit's tiles: pass 1 gives
// each query's running maximum (redux.sync per query, 4-warp exchange) and row sum
// (kept per thread, reduced once); pass 2 recomputes the scores and adds
// sum_q exp2(s - m_q) / l_q for the thread's key into mass[b][j] (one atomic add per
// key and unit).  The second pass re-reads the unit's K tiles, mostly from L2.
//
// FP8-e4m3 caches: TMA stages the e4m3 K tiles and four converter warps turn each into
// an f16 operand tile holding the bare codes (exact in f16); the softmax multiplies a
// key's scores by its K group scale, as the attention kernel does.  The converters also
// turn each unit's Q chunk from bf16 to f16 in place, so the MMAs of this path are f16.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace dllm {
namespace {

constexpr uint32_t kKTileBytes = kKeyTile * kHd * 2;  // 32 KB
constexpr uint32_t kK8TileBytes = kKeyTile * kHd;     // 16 KB (e4m3 codes)
constexpr int kMaskWords = 512;                        // MASK-slot bitmap: max_pos <= 16384

template <int NQ, bool FP8>
struct MassSmem {
  static constexpr int KST = FP8 ? 2 : 4;  // K operand ring (bf16 from TMA, or f16 from the converters)
  static constexpr int SST = FP8 ? 2 : 1;  // e4m3 staging ring
  static constexpr int kThreads = FP8 ? 320 : 192;
  uint8_t q[2][NQ * kHd * 2];
  uint8_t k[KST][kKTileBytes];
  uint8_t sk[SST][FP8 ? kK8TileBytes : 1024];
  float red[4][NQ];
  float m_run[NQ];
  float m_use[NQ];
  float alpha[NQ];
  float inv_l[NQ];
  uint32_t mask_bits[kMaskWords];
  uint32_t draft_qmask[2];
  int n_draft;
  uint64_t q_full[2], q_empty[2];
  uint64_t q_conv[2];  // e4m3: the Q chunk has been converted to f16 in place
  uint64_t k_full[KST], k_empty[KST];
  uint64_t sk_full[SST], sk_empty[SST];
  uint64_t s_full[2], s_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(MassSmem<64, false>) + 1024 <= 232448, "shared memory budget");
static_assert(sizeof(MassSmem<64, true>) + 1024 <= 232448, "shared memory budget (e4m3)");

// 16 e4m3 codes to f16, unscaled (exact: every e4m3 value is an f16 value).
DEVI void codes16_to_f16(const uint4 in, uint4& lo, uint4& hi) {
  const __nv_fp8x2_storage_t* pr = reinterpret_cast<const __nv_fp8x2_storage_t*>(&in);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 h = __half2(__nv_cvt_fp8x2_to_halfraw2(pr[i], __NV_E4M3));
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
}

// bf16 -> f16 of 8 values (a Q chunk of the e4m3 path).
DEVI uint4 q_bf16x8_to_f16x8(uint4 v) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
    const __half2 h = __floats2half2_rn(lo, hi);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return v;
}

DEVI void mass_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

DEVI float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

DEVI float exp2_approx(float x) {  // PTX ex2.approx.ftz.f32, 2^-inf = +0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int NQ, bool FP8>
__global__ void __launch_bounds__(MassSmem<NQ, FP8>::kThreads, 1)
    attn_mass_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                 const AttnParams p, float* __restrict__ mass) {
  using Sm = MassSmem<NQ, FP8>;
  constexpr int KST = Sm::KST, SST = Sm::SST;
  constexpr uint32_t kQBox = NQ * 128;
  constexpr uint32_t kTmemCols = (2 * NQ < 32) ? 32 : 2 * NQ;
  extern __shared__ uint8_t smem_raw[];
  Sm& S = *reinterpret_cast<Sm*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  volatile int* abort_flag = &S.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = p.B * p.H * p.n_qchunks;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.q_full[i], 1);
      mbar_init(&S.q_empty[i], 1);
      mbar_init(&S.q_conv[i], 4);  // the four converter warps (e4m3 caches)
      mbar_init(&S.s_full[i], 1);
      mbar_init(&S.s_free[i], 4);
    }
    // bf16: K tiles filled by TMA (one arrival + bytes); e4m3: by the 4 converter warps
    for (int i = 0; i < KST; ++i) {
      mbar_init(&S.k_full[i], FP8 ? 4 : 1);
      mbar_init(&S.k_empty[i], 1);
    }
    for (int i = 0; i < SST; ++i) {
      mbar_init(&S.sk_full[i], 1);
      mbar_init(&S.sk_empty[i], 4);
    }
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_kv);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  // unit u -> (b, h, query chunk)
  auto decode = [&](int u, int& b, int& h, int& qc) {
    qc = u % p.n_qchunks;
    u /= p.n_qchunks;
    h = u % p.H;
    b = u / p.H;
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_q = policy_evict_last();
    const uint64_t pol_k = policy_evict_normal();  // read twice per unit
    int ks = 0, uu = 0;  // K ring (bf16) or staging ring (e4m3) position
    uint32_t kph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uu) {
      int b, h, qc;
      decode(u, b, h, qc);
      const int qb = uu & 1;
      if (!mbar_wait(&S.q_empty[qb], ((uu >> 1) & 1) ^ 1u, abort_flag)) { ok = false; break; }
      mbar_arrive_expect_tx(&S.q_full[qb], 2 * kQBox);
      const int qrow = b * p.n_tok + qc * kQChunk;
      tma_load_2d(S.q[qb], &tm_q, &S.q_full[qb], h * kHd, qrow, pol_q);
      tma_load_2d(S.q[qb] + kQBox, &tm_q, &S.q_full[qb], h * kHd + 64, qrow, pol_q);
      for (int i = 0; i < 2 * p.key_tiles && ok; ++i) {
        const int t = i % p.key_tiles;
        const int key0 = b * p.slots + t * kKeyTile;
        if constexpr (FP8) {
          if (!mbar_wait(&S.sk_empty[ks], kph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.sk_full[ks], kK8TileBytes);
          tma_load_3d(S.sk[ks], &tm_kv, &S.sk_full[ks], 0, h, key0, pol_k);
          if (++ks == SST) { ks = 0; kph ^= 1u; }
        } else {
          if (!mbar_wait(&S.k_empty[ks], kph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.k_full[ks], kKTileBytes);
          tma_load_3d(S.k[ks], &tm_kv, &S.k_full[ks], 0, h, key0, pol_k);
          tma_load_3d(S.k[ks] + kKTileBytes / 2, &tm_kv, &S.k_full[ks], 64, h, key0, pol_k);
          if (++ks == KST) { ks = 0; kph ^= 1u; }
        }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.status, DLLM_DEV_TIMEOUT);
    }
    volatile int never = 0;
    const int qn = uu & 1;
    const uint32_t qph = (uu >> 1) & 1u;
    for (int i = 0; i < 2; ++i) mbar_wait(&S.q_full[i], (i < qn) ? qph : (qph ^ 1u), &never);
    if constexpr (FP8) {
      for (int i = 0; i < SST; ++i) mbar_wait(&S.sk_full[i], (i < ks) ? kph : (kph ^ 1u), &never);
    } else {
      for (int i = 0; i < KST; ++i) mbar_wait(&S.k_full[i], (i < ks) ? kph : (kph ^ 1u), &never);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = FP8 ? idesc_f16(128, NQ, false, false) : idesc_bf16(128, NQ, false, false);
    int ks = 0, uu = 0;
    uint32_t kph = 0, s_cnt = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uu) {
      const int qb = uu & 1;
      if (!mbar_wait(FP8 ? &S.q_conv[qb] : &S.q_full[qb], (uu >> 1) & 1u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t q0 = smem_u32(S.q[qb]);
      for (int i = 0; i < 2 * p.key_tiles; ++i) {
        const uint32_t sb = s_cnt & 1u, sph = (s_cnt >> 1) & 1u;
        if (!mbar_wait(&S.s_free[sb], sph ^ 1u, abort_flag)) { ok = false; break; }
        if (!mbar_wait(&S.k_full[ks], kph, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k0 = smem_u32(S.k[ks]);
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kKTileBytes / 2) + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * kQBox + (kk & 3) * 32;
          tc_mma_f16(tmem + sb * NQ, sdesc_sw128(k0 + off, 16, 1024), sdesc_sw128(q0 + qoff, 16, 1024), idesc_s,
                     kk != 0);
        }
        tc_commit(&S.k_empty[ks]);
        tc_commit(&S.s_full[sb]);
        if (++ks == KST) { ks = 0; kph ^= 1u; }
        ++s_cnt;
      }
      if (!ok) break;
      tc_commit(&S.q_empty[qb]);
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.status, DLLM_DEV_TIMEOUT);
    }
    tc_commit(&S.drain);
    volatile int never = 0;
    mbar_wait(&S.drain, 0, &never);
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ softmax warps
    // Thread r owns key r of every S^T tile.  The four warps run the same barrier
    // sequence; a failed wait is recorded and the sequence continues.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const bool has_view = p.view != nullptr;
    const int mask_words = (p.max_pos + 31) >> 5;
    uint32_t s_cnt = 0;
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t par) {
      if (!mbar_wait(bar, par, abort_flag)) {
        ok = false;
        *abort_flag = 1;
      }
    };
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      int b, h, qc;
      decode(u, b, h, qc);
      const int row0 = b * p.n_tok;
      const int nrows = min(kQChunk, p.n_tok - qc * kQChunk);
      // padded query columns take no part
      const uint64_t qmask = nrows >= 64 ? ~0ull : ((1ull << nrows) - 1ull);
      if (r < NQ) S.m_run[r] = -INFINITY;
      if (has_view) {
        for (int w = r; w < mask_words; w += 128) S.mask_bits[w] = 0u;
        if (r == 0) S.n_draft = 0;
        mass_sync();
        int my_draft = 0;
        for (int t = r; t < p.n_tok; t += 128) {
          const int v = p.view[row0 + t];
          if (v == DLLM_VIEW_MASK) {
            const int pos = p.positions[row0 + t];
            if (pos >= 0 && pos < p.max_pos) atomicOr(&S.mask_bits[pos >> 5], 1u << (pos & 31));
          } else if (v == DLLM_VIEW_DRAFT) {
            ++my_draft;
          }
        }
        if (my_draft) atomicAdd(&S.n_draft, my_draft);
        if (quarter < 2) {
          const bool is_draft = r < nrows && p.view[row0 + qc * kQChunk + r] == DLLM_VIEW_DRAFT;
          const uint32_t bal = __ballot_sync(0xffffffffu, is_draft);
          if (lane == 0) S.draft_qmask[quarter] = bal;
        }
      }
      mass_sync();
      const int n_draft = has_view ? min(S.n_draft, p.tail) : 0;
      const uint64_t dmask = has_view ? (static_cast<uint64_t>(S.draft_qmask[1]) << 32) | S.draft_qmask[0] : 0ull;
      float l_part[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) l_part[q] = 0.0f;

      for (int i = 0; i < 2 * p.key_tiles; ++i) {
        const bool pass2 = i >= p.key_tiles;
        const int t = pass2 ? i - p.key_tiles : i;
        const uint32_t sb = s_cnt & 1u, sph = (s_cnt >> 1) & 1u;
        wait(&S.s_full[sb], sph);
        tc_fence_after();
        float s[NQ];
#pragma unroll
        for (int c = 0; c < NQ; c += 32) tmem_ld32(tmem + lane_base + sb * NQ + c, *reinterpret_cast<float(*)[32]>(s + c));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.s_free[sb]);
        ++s_cnt;
        const int j = t * kKeyTile + r;
        uint64_t vis;
        if (!has_view) {
          vis = (j < p.max_pos) ? ~0ull : 0ull;
        } else if (j < p.max_pos) {
          vis = ((S.mask_bits[j >> 5] >> (j & 31)) & 1u) ? ~dmask : ~0ull;
        } else {
          vis = (j < p.max_pos + n_draft) ? dmask : 0ull;
        }
        vis &= qmask;
        // e4m3: the K operand holds the bare code; the key's K group scale multiplies
        // its scores
        const float sc = FP8 ? (vis ? p.scale_log2 * __ldg(p.kv_scale + (static_cast<size_t>(b) * p.slots + j) * 2 * p.H + h)
                                    : 0.0f)
                             : p.scale_log2;
#pragma unroll
        for (int q = 0; q < NQ; ++q) s[q] = ((vis >> q) & 1ull) ? s[q] * sc : -INFINITY;
        if (!pass2) {
          // ---- pass 1: running max per query, this thread's share of the row sums
          float mx[NQ];
#pragma unroll
          for (int q = 0; q < NQ; ++q) mx[q] = warp_max_f32(s[q]);
          if (lane == 0) {
            float4* dst = reinterpret_cast<float4*>(S.red[quarter]);
#pragma unroll
            for (int q = 0; q < NQ; q += 4) dst[q / 4] = make_float4(mx[q], mx[q + 1], mx[q + 2], mx[q + 3]);
          }
          mass_sync();
          if (r < NQ) {
            const float mt = fmaxf(fmaxf(S.red[0][r], S.red[1][r]), fmaxf(S.red[2][r], S.red[3][r]));
            const float m_old = S.m_run[r];
            const float m_new = fmaxf(m_old, mt);
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            S.m_run[r] = m_new;
            S.m_use[r] = m_use;
            S.alpha[r] = exp2_approx(m_old - m_use);
          }
          mass_sync();
#pragma unroll
          for (int q = 0; q < NQ; ++q) l_part[q] = l_part[q] * S.alpha[q] + exp2_approx(s[q] - S.m_use[q]);
          if (t == p.key_tiles - 1) {
            // end of pass 1: reduce the row sums over the 128 threads
#pragma unroll
            for (int c = 0; c < NQ; c += 32) {
              float tmp[32];
#pragma unroll
              for (int k = 0; k < 32; ++k) tmp[k] = l_part[c + k];
              // lane i ends with column c + i summed over the warp
#pragma unroll
              for (int w = 16; w >= 1; w >>= 1) {
                const bool upper = (lane & w) != 0;
#pragma unroll
                for (int k = 0; k < w; ++k) {
                  const float send = upper ? tmp[k] : tmp[k + w];
                  const float keep = upper ? tmp[k + w] : tmp[k];
                  tmp[k] = keep + __shfl_xor_sync(0xffffffffu, send, w);
                }
              }
              mass_sync();  // every thread has read red / alpha of this tile
              S.red[quarter][c + lane] = tmp[0];
              mass_sync();
              if (r < 32) {
                const float lt = S.red[0][c + r] + S.red[1][c + r] + S.red[2][c + r] + S.red[3][c + r];
                S.inv_l[c + r] = lt > 0.0f ? 1.0f / lt : 0.0f;
              }
            }
            mass_sync();
          }
        } else {
          // ---- pass 2: this key's weight in every query, summed over the queries
          float w = 0.0f;
#pragma unroll
          for (int q = 0; q < NQ; ++q) w += exp2_approx(s[q] - S.m_use[q]) * S.inv_l[q];
          if (j < p.max_pos && ok) atomicAdd(mass + static_cast<size_t>(b) * p.max_pos + j, w);
        }
      }
      mass_sync();  // the next unit resets the running state and the tags
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.status, DLLM_DEV_TIMEOUT);
    }
  } else if (FP8 && warp >= 6) {
    // ------------------------------------------------------------ e4m3 -> f16 converters
    // Per unit: the Q chunk, bf16 -> f16 in place.  Per tile (both passes): thread r turns
    // key row r of the staged codes into both 64-column halves of the K operand tile,
    // keeping the 128-byte swizzle.
    const int r = (warp & 3) * 32 + lane;
    int ss = 0, ko = 0, uu = 0;
    uint32_t sph = 0, kph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uu) {
      {
        const int qb = uu & 1;
        if (!mbar_wait_warp(&S.q_full[qb], (uu >> 1) & 1u, abort_flag)) { ok = false; break; }
        uint4* qv = reinterpret_cast<uint4*>(S.q[qb]);
        for (int i = r; i < static_cast<int>(NQ * kHd * 2 / 16); i += 128) qv[i] = q_bf16x8_to_f16x8(qv[i]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.q_conv[qb]);
      }
      for (int i = 0; i < 2 * p.key_tiles; ++i) {
        if (!mbar_wait_warp(&S.sk_full[ss], sph, abort_flag)) { ok = false; break; }
        if (!mbar_wait_warp(&S.k_empty[ko], kph ^ 1u, abort_flag)) { ok = false; break; }
        const uint32_t sw = static_cast<uint32_t>(r & 7);
        const uint8_t* src = S.sk[ss] + r * 128;
        uint8_t* dst = S.k[ko] + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 in = *reinterpret_cast<const uint4*>(src + ((c ^ sw) << 4));
          uint4 lo, hi;
          codes16_to_f16(in, lo, hi);
          uint8_t* half = dst + (c >> 2) * (kKTileBytes / 2);
          const uint32_t c0 = (c & 3) * 2;
          *reinterpret_cast<uint4*>(half + ((c0 ^ sw) << 4)) = lo;
          *reinterpret_cast<uint4*>(half + (((c0 + 1) ^ sw) << 4)) = hi;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&S.k_full[ko]);
          mbar_arrive(&S.sk_empty[ss]);
        }
        if (++ko == KST) { ko = 0; kph ^= 1u; }
        if (++ss == SST) { ss = 0; sph ^= 1u; }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.status, DLLM_DEV_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NQ, bool FP8>
int launch_mass_one(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv, float* mass, int grid,
                    cudaStream_t s) {
  using Sm = MassSmem<NQ, FP8>;
  const size_t smem = sizeof(Sm) + 1024;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(attn_mass_tc<NQ, FP8>), (int)(smem));
  if (e != cudaSuccess) return (int)e;
  attn_mass_tc<NQ, FP8><<<grid, Sm::kThreads, smem, s>>>(tm_q, tm_kv, p, mass);
  return (int)cudaGetLastError();
}

}  // namespace

int launch_attn_mass(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv, float* mass, int grid,
                     cudaStream_t s) {
  if (p.kv_dtype == DLLM_E4M3)
    return p.nq_pad <= 32 ? launch_mass_one<32, true>(p, tm_q, tm_kv, mass, grid, s)
                          : launch_mass_one<64, true>(p, tm_q, tm_kv, mass, grid, s);
  return p.nq_pad <= 32 ? launch_mass_one<32, false>(p, tm_q, tm_kv, mass, grid, s)
                        : launch_mass_one<64, false>(p, tm_q, tm_kv, mass, grid, s);
}

}  // namespace dllm
