// Fused QKV projection + rotary embedding + cache scatter-write (tensor-core path).
//
// "Flash-dLLM: IO-aware KV caching and parallel decoding", paragraph 2: the projection,
// the rotary embedding and the cache write are one kernel whose intermediates never go
// back to HBM.  "LaCache ...", Methodology 1 (RoPECache): what the cache keeps per token
// is the projected, rotary-embedded K/V.  "LaCache ...", Methodology 2: groups of 128
// elements for FP8 (here one group = one head of one token, K or V).
//
// Design (sm_103a): persistent CTAs, one per SM, each walking a static list of
// 128 x BN output tiles.  Warp 0 streams x and W_qkv tiles with TMA into a
// STAGES-deep 128-byte-swizzled shared-memory ring; warp 1 issues tcgen05.mma
// (M=128, N=BN, K=16, bf16 -> fp32) into one of two TMEM accumulators; warps 2-5 (one
// per TMEM lane quarter) drain the other accumulator: each thread owns one token row,
// so both halves (i, i+64) of every rotary pair are in its own registers.  It rotates
// Q and K in fp32 with the per-position cos/sin table, rounds to bf16 (or quantises a
// head to e4m3 with scale amax/448) and writes 16-byte vectors straight to the token's
// cache slot, its probe row or the Q scratch.  The tiles left over after the last full
// round of CTAs are cut into two 128-column halves (one head each) when that keeps
// more SMs busy in the last round; a half uses N = 128 and loads half of the W tile.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace dllm {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;                  // bf16 elements per 128-byte swizzle row
constexpr int kThreads = 192;           // 6 warps
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KB

template <int BN>
struct Cfg {
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr uint32_t kBBytes = BN * BK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
  static constexpr size_t kSmem = 1024 + STAGES * kStageBytes + 256;
};

struct TileCoord {
  int grp;  // 0 = query rows (Q,K,V columns), 1 = K/V-only rows (K,V columns)
  int m0;   // first row
  int n0;   // first output feature in [0, 3D)
};

DEVI TileCoord decode_tile(const ProjParams& p, int tile, int BN) {
  TileCoord c;
  int mt, nt;
  if (tile < p.tiles_q) {
    c.grp = 0;
    if (p.m_fastest) { mt = tile % p.mt_q; nt = tile / p.mt_q; }
    else { nt = tile % p.nt_q; mt = tile / p.nt_q; }
    c.n0 = nt * BN;
  } else {
    c.grp = 1;
    const int t = tile - p.tiles_q;
    if (p.m_fastest) { mt = t % p.mt_kv; nt = t / p.mt_kv; }
    else { nt = t % p.nt_kv; mt = t / p.nt_kv; }
    c.n0 = p.D + nt * BN;
  }
  c.m0 = mt * BM;
  return c;
}

// A work item is a whole tile (items [0, whole_items)) or one 128-column half of one of
// the remaining tiles.
struct Item {
  int tile;
  int half;  // -1: whole tile; 0 or 1: which 128-column half
};

DEVI Item decode_item(const ProjParams& p, int item) {
  Item it;
  if (item < p.whole_items) {
    it.tile = item;
    it.half = -1;
  } else {
    const int i = item - p.whole_items;
    it.tile = p.whole_items + (i >> 1);
    it.half = i & 1;
  }
  return it;
}

DEVI void raise_status(int* status, int bits) { atomicOr(status, bits); }

// Pack 32 floats into bf16 and store 64 bytes.
DEVI void store_bf16x32(void* dst, const float (&v)[32]) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// Quantise 32 floats to e4m3 (x / scale, round to nearest even, saturating) and store 32 bytes.
DEVI void store_e4m3x32(void* dst, const float (&v)[32], float scale) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t b = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float2 f = make_float2(__fdiv_rn(v[4 * i + 2 * j], scale), __fdiv_rn(v[4 * i + 2 * j + 1], scale));
      __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      b |= static_cast<uint32_t>(q) << (16 * j);
    }
    w[i] = b;
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Rotate pairs (lo[i], hi[i]) by the angles of table entries cs[0..31].
DEVI void rotate32(float (&lo)[32], float (&hi)[32], const float2* __restrict__ cs) {
  const float4* cs4 = reinterpret_cast<const float4*>(cs);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 t = __ldg(cs4 + i);  // (cos, sin) of two consecutive pair indices
    {
      const float a = lo[2 * i], b = hi[2 * i];
      lo[2 * i] = a * t.x - b * t.y;
      hi[2 * i] = b * t.x + a * t.y;
    }
    {
      const float a = lo[2 * i + 1], b = hi[2 * i + 1];
      lo[2 * i + 1] = a * t.z - b * t.w;
      hi[2 * i + 1] = b * t.z + a * t.w;
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    proj_rope_store_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xkv,
                       const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_w_half,
                       const ProjParams p) {
  using C = Cfg<BN>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_xkv);
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_w_half);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_x = p.m_fastest ? policy_evict_last() : policy_evict_first();
    const uint64_t pol_w = p.m_fastest ? policy_evict_first() : policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < p.items_total && ok; item += gridDim.x) {
      const Item it = decode_item(p, item);
      const TileCoord c = decode_tile(p, it.tile, BN);
      const CUtensorMap* am = c.grp ? &tm_xkv : &tm_x;
      const bool half = it.half >= 0;
      const int n0 = half ? c.n0 + it.half * kHd : c.n0;
      const uint32_t bytes = half ? kABytes + kHd * BK * 2 : C::kStageBytes;
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&full[stage], bytes);
        tma_load_2d(sA + stage * kABytes, am, &full[stage], kb * BK, c.m0, pol_x);
        tma_load_2d(sB + stage * C::kBBytes, half ? &tm_w_half : &tm_w, &full[stage], kb * BK, n0, pol_w);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      raise_status(p.status, DLLM_DEV_TIMEOUT);
    }
    // Let every copy this thread issued land before the CTA can exit.
    for (int s = 0; s < STAGES; ++s) {
      // the most recent phase armed on stage s has parity (phase ^ 1) if s >= stage, else phase
      const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
      volatile int never = 0;
      mbar_wait(&full[s], par, &never);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_whole = idesc_bf16(BM, BN, false, false);
    constexpr uint32_t idesc_half = idesc_bf16(BM, kHd, false, false);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < p.items_total && ok; item += gridDim.x) {
      const uint32_t idesc = decode_item(p, item).half >= 0 ? idesc_half : idesc_whole;
      if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + stage * kABytes);
        const uint32_t b0 = smem_u32(sB + stage * C::kBBytes);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          tc_mma_f16(d_tmem, sdesc_sw128(a0 + k * 32, 16, 1024), sdesc_sw128(b0 + k * 32, 16, 1024), idesc,
                     (kb | k) != 0);
        }
        tc_commit(&empty[stage]);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      tc_commit(&tfull[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
      *abort_flag = 1;
      raise_status(p.status, DLLM_DEV_TIMEOUT);
    }
    // Drain: wait until every MMA issued here has finished before TMEM is released.
    tc_commit(drain);
    volatile int never = 0;
    mbar_wait(drain, 0, &never);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    const int hd = kHd;
    bool ok = true;  // a failed wait is recorded; the item sequence continues without stores
    for (int item = blockIdx.x; item < p.items_total; item += gridDim.x) {
      const Item it = decode_item(p, item);
      TileCoord c = decode_tile(p, it.tile, BN);
      if (it.half >= 0) c.n0 += it.half * kHd;
      const int heads = it.half >= 0 ? 1 : BN / kHd;
      if (!mbar_wait_warp(&tfull[acc], acc_phase, abort_flag)) {
        ok = false;
        *abort_flag = 1;
      }
      tc_fence_after();

      // ---- this thread's row
      const int m = c.m0 + r;
      bool valid;
      int b = 0, pos = 0, slot = 0;
      if (c.grp == 0) {
        valid = m < p.m_q;
        if (valid) {
          b = m / p.n_tok;
          pos = __ldg(p.positions + m);
          slot = pos;
          const int v = p.view ? static_cast<int>(__ldg(p.view + m)) : DLLM_VIEW_BASE;
          if (v > DLLM_VIEW_MASK) {
            if (c.n0 == 0) raise_status(p.status, DLLM_DEV_BAD_VIEW);
            valid = false;
          } else if (v == DLLM_VIEW_DRAFT) {
            int rank = 0;
            for (int t = b * p.n_tok; t < m; ++t) rank += (__ldg(p.view + t) == DLLM_VIEW_DRAFT);
            if (rank >= p.tail) {
              if (c.n0 == 0) raise_status(p.status, DLLM_DEV_TAIL_FULL);
              valid = false;
            }
            slot = p.max_pos + rank;
          }
        }
      } else {
        valid = m < p.m_kv;
        if (valid) {
          b = m / p.n_kv;
          pos = __ldg(p.kv_positions + m);
          slot = pos;
        }
      }
      if (valid && (pos < 0 || pos >= p.max_pos)) {
        if (c.n0 == (c.grp ? p.D : 0)) raise_status(p.status, DLLM_DEV_BAD_POSITION);
        valid = false;
      }
      valid = valid && ok;

      const int part = c.n0 / p.D;  // 0 Q, 1 K, 2 V
      const bool rope = part < 2;
      const float2* cs_row = p.rope + static_cast<size_t>(valid ? pos : 0) * (hd / 2);
#pragma unroll 1
      for (int hh = 0; hh < heads; ++hh) {
        const int h = (c.n0 - part * p.D) / kHd + hh;
        const uint32_t tcol = tmem_base + lane_base + acc * BN + hh * kHd;
        // destination of this row's 128 values
        uint8_t* dst = nullptr;
        float* sdst = nullptr;
        const bool to_probe = (c.grp == 1) && (p.probe != nullptr);
        if (part == 0) {
          dst = reinterpret_cast<uint8_t*>(p.q_out) + (static_cast<size_t>(m) * p.D + h * hd) * 2;
        } else if (to_probe) {
          dst = reinterpret_cast<uint8_t*>(p.probe) +
                ((static_cast<size_t>(m) * 2 + (part - 1)) * p.D + h * hd) * 2;
        } else {
          const size_t row = (static_cast<size_t>(b) * p.slots + slot) * 2 + (part - 1);
          if (p.kv_dtype == DLLM_E4M3) {
            dst = reinterpret_cast<uint8_t*>(p.cache_kv) + row * p.D + h * hd;
            sdst = p.cache_scale + row * p.H + h;
          } else {
            dst = reinterpret_cast<uint8_t*>(p.cache_kv) + (row * p.D + h * hd) * 2;
          }
        }
        const bool fp8 = (sdst != nullptr);
        float scale = 1.0f;
        if (fp8) {
          float amax = 0.0f;
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            float lo[32], hi[32];
            tmem_ld32(tcol + half * 32, lo);
            tmem_ld32(tcol + 64 + half * 32, hi);
            if (rope) rotate32(lo, hi, cs_row + half * 32);
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fmaxf(fabsf(lo[i]), fabsf(hi[i])));
          }
          scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        }
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          float lo[32], hi[32];
          tmem_ld32(tcol + half * 32, lo);
          tmem_ld32(tcol + 64 + half * 32, hi);
          if (rope) rotate32(lo, hi, cs_row + half * 32);
          if (valid) {
            if (fp8) {
              store_e4m3x32(dst + half * 32, lo, scale);
              store_e4m3x32(dst + 64 + half * 32, hi, scale);
            } else {
              store_bf16x32(dst + half * 64, lo);
              store_bf16x32(dst + 128 + half * 64, hi);
            }
          }
        }
        if (fp8 && valid) *sdst = scale;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) raise_status(p.status, DLLM_DEV_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace

size_t proj_tc_smem_bytes(int bn) { return bn == 256 ? Cfg<256>::kSmem : Cfg<128>::kSmem; }

int launch_proj_tc(const ProjParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_xkv,
                   const CUtensorMap& tm_w, const CUtensorMap& tm_w_half, int bn, int grid, cudaStream_t s) {
  cudaError_t e;
  if (bn == 256) {
    auto k = proj_rope_store_tc<256>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<256>::kSmem);
    if (e != cudaSuccess) return (int)e;
    k<<<grid, kThreads, Cfg<256>::kSmem, s>>>(tm_x, tm_xkv, tm_w, tm_w_half, p);
  } else {
    auto k = proj_rope_store_tc<128>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<128>::kSmem);
    if (e != cudaSuccess) return (int)e;
    k<<<grid, kThreads, Cfg<128>::kSmem, s>>>(tm_x, tm_xkv, tm_w, tm_w_half, p);
  }
  return (int)cudaGetLastError();
}

}  // namespace dllm
