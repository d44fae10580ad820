// Bidirectional attention of a step's query rows over the flat K/V cache
// (tensor-core path, bf16 and FP8-e4m3 caches).
//
// "LaCache ...", technical summary, Problem Statement: inside a block every query
// attends to the full context (non-causal).  "Flash-Cache" article, section 3.1:
// softmax(q k^T / sqrt(d)) v fused in one kernel.  "Flash-dLLM ...", paragraph 3:
// Flash-Verify draft and mask views must not see each other.
//
// Design (sm_103a).  A work unit is (sequence b, head h, chunk of <= NQ query rows,
// key split).  Per 128-key tile the MMA warp computes S^T = K Q^T with tcgen05
// (M = 128 keys, N = NQ queries, K = hd = 128) into TMEM, so each softmax thread owns
// one key and holds that key's scores for every query.  Column (per-query) maxima and
// sums are warp reduce-scatters plus a 4-warp exchange in shared memory; the online
// softmax runs in fp32 with exp2.  Each thread writes its key's probabilities as bf16
// into P^T (K-major, 128-byte swizzle) and the MMA warp computes O^T = V^T P^T
// (M = hd, N = NQ, V read MN-major straight from the TMA-staged cache tile) into a
// second TMEM buffer; the same threads fold it into fp32 register accumulators with
// the running rescale.  K/V tiles stream through TMA rings (3 K + 2 V stages of 32 KB);
// S, P and O are double-buffered so the loads, both MMAs and the softmax overlap.
// With few units, keys are split across CTAs and a second kernel merges the partial
// (O, m, l) states.
//
// FP8-e4m3 cache ("LaCache ...", Methodology 2: per-group FP8; one group here = one
// head of one token, K or V, with an fp32 scale): TMA stages the e4m3 tiles (half the
// bytes of bf16) in a 3-deep ring and four converter warps widen them to bf16 in the
// MMA operand layout (exact: every e4m3 value is a bf16 value).  The K scale of a key
// multiplies that key's scores in fp32, and the V scale multiplies its probabilities
// before they are rounded for the PV MMA, so dequantisation adds no rounding step.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace dllm {
namespace {

constexpr uint32_t kTileBytes = kKeyTile * kHd * 2;  // 32 KB (bf16 K or V tile)
constexpr uint32_t kTile8Bytes = kKeyTile * kHd;     // 16 KB (e4m3 tile)
constexpr uint32_t kQBytes = kQChunk * kHd * 2;      // 16 KB
constexpr uint32_t kPBytes = kQChunk * kKeyTile * 2; // 16 KB
constexpr int kMaxBitmapWords = 512;                 // MASK-slot bitmap: max_pos <= 16384

// Per cache type: MMA-operand rings for K and V, e4m3 staging rings, thread count.
template <bool FP8>
struct Cfg {
  static constexpr int KST = FP8 ? 1 : 3;
  static constexpr int VST = FP8 ? 1 : 2;
  static constexpr int SST = FP8 ? 3 : 1;
  static constexpr uint32_t kStageBytes = FP8 ? kTile8Bytes : 1024;
  static constexpr int kThreads = FP8 ? 320 : 192;  // + 4 converter warps for FP8
};

template <bool FP8>
struct Smem {
  using C = Cfg<FP8>;
  // all operand tiles 1024-byte aligned
  uint8_t q[kQBytes];
  uint8_t k[C::KST][kTileBytes];
  uint8_t v[C::VST][kTileBytes];
  uint8_t p[2][kPBytes];
  uint8_t sk[C::SST][C::kStageBytes];  // e4m3 staging (FP8 only)
  uint8_t sv[C::SST][C::kStageBytes];
  float red_max[4][kQChunk];
  float red_sum[2][4][kQChunk];
  float m_run[kQChunk];
  float l_run[kQChunk];
  float m_use[kQChunk];
  float alpha[2][kQChunk];
  uint32_t mask_bits[kMaxBitmapWords];
  uint32_t draft_qmask[2];
  int n_draft;
  uint64_t q_full, q_empty;
  uint64_t k_full[C::KST], k_empty[C::KST];
  uint64_t v_full[C::VST], v_empty[C::VST];
  uint64_t sk_full[C::SST], sk_empty[C::SST];
  uint64_t sv_full[C::SST], sv_empty[C::SST];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t o_full[2], o_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Smem<false>) + 1024 <= 232448, "shared memory budget (bf16)");
static_assert(sizeof(Smem<true>) + 1024 <= 232448, "shared memory budget (e4m3)");

// Widen 16 e4m3 codes to 16 bf16 values (exact).
DEVI void widen16(const uint4 in, uint4& lo, uint4& hi) {
  const __nv_fp8x2_storage_t* pr = reinterpret_cast<const __nv_fp8x2_storage_t*>(&in);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 h(__nv_cvt_fp8x2_to_halfraw2(pr[i], __NV_E4M3));
    const float2 f = __half22float2(h);
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
}

struct Unit {
  int b, h, qc, split, t0, t1;
};

DEVI Unit decode_unit(const AttnParams& p, int u) {
  Unit x;
  x.split = u % p.n_splits;
  u /= p.n_splits;
  x.qc = u % p.n_qchunks;
  u /= p.n_qchunks;
  x.h = u % p.H;
  x.b = u / p.H;
  x.t0 = x.split * p.tiles_per_split;
  x.t1 = min(p.key_tiles, x.t0 + p.tiles_per_split);
  return x;
}

DEVI void named_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Reduce 32 per-lane values per column across the warp; afterwards lane i holds the
// reduction of column i.  MAX selects max, otherwise sum.
template <bool MAX>
DEVI float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

template <int NQ, bool FP8>
__global__ void __launch_bounds__(Cfg<FP8>::kThreads, 1)
    attn_cache_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                  const AttnParams p) {
  using C = Cfg<FP8>;
  constexpr int KST = C::KST, VST = C::VST, SST = C::SST;
  extern __shared__ uint8_t smem_raw[];
  Smem<FP8>& S = *reinterpret_cast<Smem<FP8>*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  volatile int* abort_flag = &S.abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr uint32_t kTmemCols = 4 * NQ;  // S[2] then O[2]
  constexpr uint32_t kQBox = NQ * 128;    // bytes of one 64-column Q box / one P region

  if (threadIdx.x == 0) {
    mbar_init(&S.q_full, 1);
    mbar_init(&S.q_empty, 1);
    // bf16: operand tiles are filled by TMA (one arrival + bytes); e4m3: by 4 converter warps
    for (int i = 0; i < KST; ++i) { mbar_init(&S.k_full[i], FP8 ? 4 : 1); mbar_init(&S.k_empty[i], 1); }
    for (int i = 0; i < VST; ++i) { mbar_init(&S.v_full[i], FP8 ? 4 : 1); mbar_init(&S.v_empty[i], 1); }
    for (int i = 0; i < SST; ++i) {
      mbar_init(&S.sk_full[i], 1);
      mbar_init(&S.sk_empty[i], 4);
      mbar_init(&S.sv_full[i], 1);
      mbar_init(&S.sv_empty[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.s_full[i], 1);
      mbar_init(&S.s_free[i], 4);
      mbar_init(&S.p_full[i], 4);
      mbar_init(&S.p_empty[i], 1);
      mbar_init(&S.o_full[i], 1);
      mbar_init(&S.o_free[i], 4);
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

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_q = policy_evict_last();
    int ks = 0, vs = 0;
    uint32_t kph = 0, vph = 0, qph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      const Unit x = decode_unit(p, u);
      if (!mbar_wait(&S.q_empty, qph ^ 1u, abort_flag)) { ok = false; break; }
      qph ^= 1u;
      mbar_arrive_expect_tx(&S.q_full, 2 * kQBox);
      const int qrow = x.b * p.n_tok + x.qc * kQChunk;
      tma_load_2d(S.q, &tm_q, &S.q_full, x.h * kHd, qrow, pol_q);
      tma_load_2d(S.q + kQBox, &tm_q, &S.q_full, x.h * kHd + 64, qrow, pol_q);
      const int slot0 = x.b * p.slots;
      for (int t = x.t0; t < x.t1; ++t) {
        const int key0 = slot0 + t * kKeyTile;
        if constexpr (FP8) {
          // e4m3 tiles into the staging rings (one 128-byte-wide box each)
          if (!mbar_wait(&S.sk_empty[ks], kph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.sk_full[ks], kTile8Bytes);
          tma_load_3d(S.sk[ks], &tm_kv, &S.sk_full[ks], 0, x.h, key0, pol_stream);
          if (!mbar_wait(&S.sv_empty[ks], kph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.sv_full[ks], kTile8Bytes);
          tma_load_3d(S.sv[ks], &tm_kv, &S.sv_full[ks], 0, p.H + x.h, key0, pol_stream);
          if (++ks == SST) { ks = 0; kph ^= 1u; }
        } else {
          if (!mbar_wait(&S.k_empty[ks], kph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.k_full[ks], kTileBytes);
          tma_load_3d(S.k[ks], &tm_kv, &S.k_full[ks], 0, x.h, key0, pol_stream);
          tma_load_3d(S.k[ks] + kTileBytes / 2, &tm_kv, &S.k_full[ks], 64, x.h, key0, pol_stream);
          if (++ks == KST) { ks = 0; kph ^= 1u; }
          if (!mbar_wait(&S.v_empty[vs], vph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.v_full[vs], kTileBytes);
          tma_load_3d(S.v[vs], &tm_kv, &S.v_full[vs], 0, p.H + x.h, key0, pol_stream);
          tma_load_3d(S.v[vs] + kTileBytes / 2, &tm_kv, &S.v_full[vs], 64, p.H + x.h, key0, pol_stream);
          if (++vs == VST) { vs = 0; vph ^= 1u; }
        }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.status, DLLM_DEV_TIMEOUT);
    }
    // let every copy issued here land before the CTA can exit
    volatile int never = 0;
    mbar_wait(&S.q_full, qph ^ 1u, &never);
    if constexpr (FP8) {
      for (int i = 0; i < SST; ++i) {
        mbar_wait(&S.sk_full[i], (i < ks) ? kph : (kph ^ 1u), &never);
        mbar_wait(&S.sv_full[i], (i < ks) ? kph : (kph ^ 1u), &never);
      }
    } else {
      for (int i = 0; i < KST; ++i) mbar_wait(&S.k_full[i], (i < ks) ? kph : (kph ^ 1u), &never);
      for (int i = 0; i < VST; ++i) mbar_wait(&S.v_full[i], (i < vs) ? vph : (vph ^ 1u), &never);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16(128, NQ, false, false);
    constexpr uint32_t idesc_o = idesc_bf16(128, NQ, true, false);
    int ks = 0, vs = 0;
    uint32_t kph = 0, vph = 0, qph = 0;
    uint32_t s_cnt = 0, pv_cnt = 0;
    bool ok = true;
    const uint32_t q0 = smem_u32(S.q);

    auto issue_pv = [&]() -> bool {
      const uint32_t pb = pv_cnt & 1u, pph = (pv_cnt >> 1) & 1u;
      if (!mbar_wait(&S.p_full[pb], pph, abort_flag)) return false;
      if (!mbar_wait(&S.o_free[pb], pph ^ 1u, abort_flag)) return false;
      if (!mbar_wait(&S.v_full[vs], vph, abort_flag)) return false;
      tc_fence_after();
      const uint32_t v0 = smem_u32(S.v[vs]);
      const uint32_t p0 = smem_u32(S.p[pb]);
      const uint32_t d = tmem + 2 * NQ + pb * NQ;
#pragma unroll
      for (int kk = 0; kk < kKeyTile / 16; ++kk) {
        const uint64_t a = sdesc_sw128(v0 + kk * 2048, 16384, 1024);
        const uint64_t b = sdesc_sw128(p0 + (kk >> 2) * kQBox + (kk & 3) * 32, 16, 1024);
        tc_mma_f16(d, a, b, idesc_o, kk != 0);
      }
      tc_commit(&S.v_empty[vs]);
      tc_commit(&S.p_empty[pb]);
      tc_commit(&S.o_full[pb]);
      if (++vs == VST) { vs = 0; vph ^= 1u; }
      ++pv_cnt;
      return true;
    };

    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      const Unit x = decode_unit(p, u);
      if (!mbar_wait(&S.q_full, qph, abort_flag)) { ok = false; break; }
      qph ^= 1u;
      tc_fence_after();
      for (int t = x.t0; t < x.t1 && ok; ++t) {
        const uint32_t sb = s_cnt & 1u, sph = (s_cnt >> 1) & 1u;
        if (!mbar_wait(&S.s_free[sb], sph ^ 1u, abort_flag)) { ok = false; break; }
        if (!mbar_wait(&S.k_full[ks], kph, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k0 = smem_u32(S.k[ks]);
        const uint32_t d = tmem + sb * NQ;
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * kQBox + (kk & 3) * 32;
          tc_mma_f16(d, sdesc_sw128(k0 + off, 16, 1024), sdesc_sw128(q0 + qoff, 16, 1024), idesc_s, kk != 0);
        }
        tc_commit(&S.k_empty[ks]);
        tc_commit(&S.s_full[sb]);
        if (++ks == KST) { ks = 0; kph ^= 1u; }
        ++s_cnt;
        if (t > x.t0 && !issue_pv()) { ok = false; break; }
      }
      if (!ok) break;
      tc_commit(&S.q_empty);
      if (x.t1 > x.t0 && !issue_pv()) { ok = false; break; }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.status, DLLM_DEV_TIMEOUT);
    }
    tc_commit(&S.drain);
    volatile int never = 0;
    mbar_wait(&S.drain, 0, &never);
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key within the tile (S^T) / hd index (O^T)
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const bool has_view = p.view != nullptr;
    constexpr bool fp8 = FP8;
    uint32_t s_cnt = 0, pv_cnt = 0;
    int vs = 0;  // V ring position, mirrors the producer
    uint32_t vph = 0;
    bool ok = true;
    const int mask_words = (p.max_pos + 31) >> 5;

    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      const Unit x = decode_unit(p, u);
      const int row0 = x.b * p.n_tok;  // first row of the sequence
      const int nrows = min(kQChunk, p.n_tok - x.qc * kQChunk);  // valid columns of this chunk
      // ---- per-unit set-up: running state and Flash-Verify tags
      if (r < NQ) {
        S.m_run[r] = -INFINITY;
        S.l_run[r] = 0.0f;
      }
      if (has_view) {
        for (int w = r; w < mask_words; w += 128) S.mask_bits[w] = 0u;
        if (r == 0) S.n_draft = 0;
        named_sync();
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
          const int q = r;  // quarters 0,1 cover columns 0..63
          const bool is_draft = q < nrows && p.view[row0 + x.qc * kQChunk + q] == DLLM_VIEW_DRAFT;
          const uint32_t bal = __ballot_sync(0xffffffffu, is_draft);
          if (lane == 0) S.draft_qmask[quarter] = bal;
        }
        named_sync();
      }
      const int n_draft = has_view ? min(S.n_draft, p.tail) : 0;
      const uint64_t dmask = has_view ? (static_cast<uint64_t>(S.draft_qmask[1]) << 32) | S.draft_qmask[0] : 0ull;
      float o_acc[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) o_acc[q] = 0.0f;

      for (int t = x.t0; t < x.t1; ++t) {
        const uint32_t sb = s_cnt & 1u, sph = (s_cnt >> 1) & 1u;
        const uint32_t tp = t & 1;  // parity slot for alpha / red_sum
        // ---- A: scores of this thread's key for every query
        if (!mbar_wait(&S.s_full[sb], sph, abort_flag)) { ok = false; break; }
        tc_fence_after();
        float s[NQ];
#pragma unroll
        for (int c = 0; c < NQ; c += 32) {
          float tmp[32];
          tmem_ld32(tmem + lane_base + sb * NQ + c, tmp);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c + i] = tmp[i];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.s_free[sb]);
        ++s_cnt;

        const int j = t * kKeyTile + r;  // slot index within the sequence
        uint64_t vis;
        if (!has_view) {
          vis = (j < p.max_pos) ? ~0ull : 0ull;
        } else if (j < p.max_pos) {
          vis = ((S.mask_bits[j >> 5] >> (j & 31)) & 1u) ? ~dmask : ~0ull;
        } else {
          vis = (j < p.max_pos + n_draft) ? dmask : 0ull;
        }
        float k_scale = 1.0f, v_scale = 1.0f;
        if (fp8 && vis) {
          const size_t srow = (static_cast<size_t>(x.b) * p.slots + j) * 2;
          k_scale = __ldg(p.kv_scale + srow * p.H + x.h);
          v_scale = __ldg(p.kv_scale + (srow + 1) * p.H + x.h);
        }
        const float sc = p.scale_log2 * k_scale;
#pragma unroll
        for (int q = 0; q < NQ; ++q) s[q] = ((vis >> q) & 1ull) ? s[q] * sc : -INFINITY;

        // column maxima: warp reduce-scatter, then 4-warp exchange
#pragma unroll
        for (int c = 0; c < NQ; c += 32) {
          float tmp[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) tmp[i] = s[c + i];
          S.red_max[quarter][c + lane] = reduce_scatter32<true>(tmp, lane);
        }
        named_sync();
        // ---- B: column owners update running max / sum
        if (r < NQ) {
          const float mt = fmaxf(fmaxf(S.red_max[0][r], S.red_max[1][r]), fmaxf(S.red_max[2][r], S.red_max[3][r]));
          const float m_old = S.m_run[r];
          const float m_new = fmaxf(m_old, mt);
          const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
          const float a = exp2f(m_old - m_use);
          if (t > x.t0) {
            const uint32_t pp = tp ^ 1u;
            const float ps = S.red_sum[pp][0][r] + S.red_sum[pp][1][r] + S.red_sum[pp][2][r] + S.red_sum[pp][3][r];
            S.l_run[r] = S.l_run[r] * S.alpha[pp][r] + ps;
          }
          S.m_run[r] = m_new;
          S.m_use[r] = m_use;
          S.alpha[tp][r] = a;
        }
        named_sync();
        // ---- C: probabilities -> P^T (bf16, swizzled) and their column sums
        {
          // Slots past the regular region that no query sees may hold anything (stale
          // draft views, the next sequence, never-written memory).  Their P is 0, but
          // 0 * NaN would still poison O, so their V rows are zeroed before the PV MMA.
          if (!FP8 && (t + 1) * kKeyTile > p.max_pos && vis == 0ull && j >= p.max_pos) {
            if (!mbar_wait(&S.v_full[vs], vph, abort_flag)) { ok = false; break; }
            uint4* row0 = reinterpret_cast<uint4*>(S.v[vs] + r * 128);
            uint4* row1 = reinterpret_cast<uint4*>(S.v[vs] + kTileBytes / 2 + r * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              row0[i] = make_uint4(0u, 0u, 0u, 0u);
              row1[i] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          if (++vs == VST) { vs = 0; vph ^= 1u; }
          const uint32_t pb = pv_cnt & 1u, pph = (pv_cnt >> 1) & 1u;
          // pv_cnt here counts tiles whose P has been produced; the PV that reads this
          // buffer two tiles ago must be done
          if (!mbar_wait(&S.p_empty[pb], pph ^ 1u, abort_flag)) { ok = false; break; }
          uint8_t* pbuf = S.p[pb] + (r >> 6) * kQBox;
          const uint32_t byte = (r & 63) * 2;
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            const float e = exp2f(s[q] - S.m_use[q]);
            s[q] = e;
            const __nv_bfloat16 hv = __float2bfloat16_rn(e * v_scale);
            *reinterpret_cast<__nv_bfloat16*>(pbuf + sw128_offset(q, byte)) = hv;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.p_full[pb]);
#pragma unroll
          for (int c = 0; c < NQ; c += 32) {
            float tmp[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) tmp[i] = s[c + i];
            S.red_sum[tp][quarter][c + lane] = reduce_scatter32<false>(tmp, lane);
          }
        }
        // ---- D: fold the previous tile's P V into the accumulators
        if (t > x.t0) {
          const uint32_t ob = (pv_cnt - 1) & 1u, oph = ((pv_cnt - 1) >> 1) & 1u;
          if (!mbar_wait(&S.o_full[ob], oph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const float* al = S.alpha[tp ^ 1u];
#pragma unroll
          for (int c = 0; c < NQ; c += 32) {
            float tmp[32];
            tmem_ld32(tmem + lane_base + 2 * NQ + ob * NQ + c, tmp);
#pragma unroll
            for (int i = 0; i < 32; ++i) o_acc[c + i] = o_acc[c + i] * al[c + i] + tmp[i];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.o_free[ob]);
        }
        ++pv_cnt;
      }
      if (!ok) break;
      // ---- unit end: last tile's PV, final sums, output
      if (x.t1 > x.t0) {
        const uint32_t ob = (pv_cnt - 1) & 1u, oph = ((pv_cnt - 1) >> 1) & 1u;
        if (!mbar_wait(&S.o_full[ob], oph, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const float* al = S.alpha[(x.t1 - 1) & 1];
#pragma unroll
        for (int c = 0; c < NQ; c += 32) {
          float tmp[32];
          tmem_ld32(tmem + lane_base + 2 * NQ + ob * NQ + c, tmp);
#pragma unroll
          for (int i = 0; i < 32; ++i) o_acc[c + i] = o_acc[c + i] * al[c + i] + tmp[i];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.o_free[ob]);
      }
      named_sync();
      if (r < NQ && x.t1 > x.t0) {
        const uint32_t pp = (x.t1 - 1) & 1;
        const float ps = S.red_sum[pp][0][r] + S.red_sum[pp][1][r] + S.red_sum[pp][2][r] + S.red_sum[pp][3][r];
        S.l_run[r] = S.l_run[r] * S.alpha[pp][r] + ps;
      }
      named_sync();
      if (p.n_splits == 1) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (q < nrows) {
            const float l = S.l_run[q];
            const float o = l > 0.0f ? o_acc[q] / l : 0.0f;
            out[static_cast<size_t>(row0 + x.qc * kQChunk + q) * p.D + x.h * kHd + r] = __float2bfloat16_rn(o);
          }
        }
      } else {
        float* wo = p.ws + static_cast<size_t>(u) * kQChunk * kHd;
#pragma unroll
        for (int q = 0; q < NQ; ++q) wo[q * kHd + r] = o_acc[q];
        if (r < NQ) {
          float* wml = p.ws + static_cast<size_t>(p.units) * kQChunk * kHd + (static_cast<size_t>(u) * kQChunk + r) * 2;
          wml[0] = S.m_run[r];
          wml[1] = S.l_run[r];
        }
      }
      named_sync();  // the next unit's set-up rewrites m_run / l_run / tags
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.status, DLLM_DEV_TIMEOUT);
    }
  } else if (FP8 && warp >= 6) {
    // ------------------------------------------------------------------ e4m3 -> bf16 converters
    // Thread r widens key row r of each staged tile into both 64-column halves of the
    // operand tile, keeping the 128-byte swizzle.  V rows of slots that no query can
    // see are written as zeros (their probability is 0, and 0 * NaN must not reach O).
    const int r = (warp & 3) * 32 + lane;
    int ss = 0, ko = 0, vo = 0;
    uint32_t sph = 0, kph = 0, vph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      const Unit x = decode_unit(p, u);
      int n_draft = 0;
      if (p.view) {
        for (int t = 0; t < p.n_tok; ++t) n_draft += (p.view[x.b * p.n_tok + t] == DLLM_VIEW_DRAFT);
        n_draft = min(n_draft, p.tail);
      }
      const int kend = p.max_pos + n_draft;
      for (int t = x.t0; t < x.t1; ++t) {
        const int j = t * kKeyTile + r;
        const uint32_t sw = static_cast<uint32_t>(r & 7);
        // K
        if (!mbar_wait(&S.sk_full[ss], sph, abort_flag)) { ok = false; break; }
        if (!mbar_wait(&S.k_empty[ko], kph ^ 1u, abort_flag)) { ok = false; break; }
        {
          const uint8_t* src = S.sk[ss] + r * 128;
          uint8_t* dst = S.k[ko] + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 in = *reinterpret_cast<const uint4*>(src + ((c ^ sw) << 4));
            uint4 lo, hi;
            widen16(in, lo, hi);
            uint8_t* half = dst + (c >> 2) * (kTileBytes / 2);
            const uint32_t c0 = (c & 3) * 2;
            *reinterpret_cast<uint4*>(half + ((c0 ^ sw) << 4)) = lo;
            *reinterpret_cast<uint4*>(half + (((c0 + 1) ^ sw) << 4)) = hi;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&S.k_full[ko]);
          mbar_arrive(&S.sk_empty[ss]);
        }
        if (++ko == KST) { ko = 0; kph ^= 1u; }
        // V
        if (!mbar_wait(&S.sv_full[ss], sph, abort_flag)) { ok = false; break; }
        if (!mbar_wait(&S.v_empty[vo], vph ^ 1u, abort_flag)) { ok = false; break; }
        {
          const uint8_t* src = S.sv[ss] + r * 128;
          uint8_t* dst = S.v[vo] + r * 128;
          const bool zero = j >= kend;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
            if (!zero) widen16(*reinterpret_cast<const uint4*>(src + ((c ^ sw) << 4)), lo, hi);
            uint8_t* half = dst + (c >> 2) * (kTileBytes / 2);
            const uint32_t c0 = (c & 3) * 2;
            *reinterpret_cast<uint4*>(half + ((c0 ^ sw) << 4)) = lo;
            *reinterpret_cast<uint4*>(half + (((c0 + 1) ^ sw) << 4)) = hi;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&S.v_full[vo]);
          mbar_arrive(&S.sv_empty[ss]);
        }
        if (++vo == VST) { vo = 0; vph ^= 1u; }
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

// Merge split-KV partial states: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
__global__ void __launch_bounds__(kHd) attn_combine(const AttnParams p) {
  const int row = blockIdx.x;  // global query row b * n_tok + t
  const int h = blockIdx.y;
  const int i = threadIdx.x;
  const int b = row / p.n_tok;
  const int t = row % p.n_tok;
  const int qc = t / kQChunk, q = t % kQChunk;
  const size_t base_unit = ((static_cast<size_t>(b) * p.H + h) * p.n_qchunks + qc) * p.n_splits;
  const float* ml = p.ws + static_cast<size_t>(p.units) * kQChunk * kHd;
  float M = -INFINITY;
  for (int s = 0; s < p.n_splits; ++s) M = fmaxf(M, ml[((base_unit + s) * kQChunk + q) * 2]);
  float L = 0.0f, O = 0.0f;
  if (M != -INFINITY) {
    for (int s = 0; s < p.n_splits; ++s) {
      const size_t uu = base_unit + s;
      const float m = ml[(uu * kQChunk + q) * 2];
      if (m == -INFINITY) continue;
      const float w = exp2f(m - M);
      L += w * ml[(uu * kQChunk + q) * 2 + 1];
      O += w * p.ws[(uu * kQChunk + q) * kHd + i];
    }
  }
  reinterpret_cast<__nv_bfloat16*>(p.out)[static_cast<size_t>(row) * p.D + h * kHd + i] =
      __float2bfloat16_rn(L > 0.0f ? O / L : 0.0f);
}

}  // namespace

size_t attn_tc_smem_bytes() { return sizeof(Smem<true>) + 1024; }

template <int NQ, bool FP8>
int launch_one(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv, int grid, cudaStream_t s) {
  const size_t smem = sizeof(Smem<FP8>) + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(attn_cache_tc<NQ, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  attn_cache_tc<NQ, FP8><<<grid, Cfg<FP8>::kThreads, smem, s>>>(tm_q, tm_kv, p);
  return (int)cudaGetLastError();
}

int launch_attn_tc(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv, int grid,
                   cudaStream_t s) {
  const bool fp8 = p.kv_dtype == DLLM_E4M3;
  if (p.nq_pad <= 32) return fp8 ? launch_one<32, true>(p, tm_q, tm_kv, grid, s) : launch_one<32, false>(p, tm_q, tm_kv, grid, s);
  return fp8 ? launch_one<64, true>(p, tm_q, tm_kv, grid, s) : launch_one<64, false>(p, tm_q, tm_kv, grid, s);
}

int launch_attn_combine(const AttnParams& p, cudaStream_t s) {
  dim3 grid(p.B * p.n_tok, p.H);
  attn_combine<<<grid, kHd, 0, s>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace dllm
