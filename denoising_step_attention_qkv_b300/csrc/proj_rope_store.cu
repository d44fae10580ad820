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
  if (p.m_fastest) {
    // column-major over the output features; a K or V column tile is followed by both
    // row groups, so the CTAs in flight share each W tile in L2 (W is read from DRAM once)
    const int q_cols = p.D / BN;  // column tiles of the Q features (query rows only)
    const int q_tiles = q_cols * p.mt_q;
    if (tile < q_tiles) {
      c.grp = 0;
      c.n0 = (tile / p.mt_q) * BN;
      c.m0 = (tile % p.mt_q) * BM;
    } else {
      const int t = tile - q_tiles;
      const int per = p.mt_q + p.mt_kv;
      const int i = t % per;
      c.n0 = p.D + (t / per) * BN;
      c.grp = i < p.mt_q ? 0 : 1;
      c.m0 = (c.grp ? i - p.mt_q : i) * BM;
    }
    return c;
  }
  // row-major (large activations): query-row tiles, then K/V-only row tiles
  if (tile < p.tiles_q) {
    c.grp = 0;
    nt = tile % p.nt_q;
    mt = tile / p.nt_q;
    c.n0 = nt * BN;
  } else {
    c.grp = 1;
    const int t = tile - p.tiles_q;
    nt = t % p.nt_kv;
    mt = t / p.nt_kv;
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

// Selection of the K/V-only rows by sequence, one bit per sequence, built once per CTA
// (select_init) from the device flags; batches larger than the table read the flags.
constexpr int kSelWords = 64;  // up to 2048 sequences
__shared__ uint32_t s_kv_sel[kSelWords];
static_assert(Cfg<256>::kSmem + sizeof(s_kv_sel) <= 232448 && Cfg<128>::kSmem + sizeof(s_kv_sel) <= 232448,
              "shared memory budget of the single-CTA projection");

DEVI bool kv_seq_selected_flags(const ProjParams& p, int b) {
  for (int j = 0; j < p.n_flag_sets; ++j)
    if (__ldg(p.kv_seq_flags + j * p.batch + b) != 0) return true;
  return false;
}

// Whether sequence b's K/V-only rows are selected (always, without flags).
DEVI bool kv_seq_selected(const ProjParams& p, int b) {
  if (p.kv_seq_flags == nullptr) return true;
  if (p.batch <= kSelWords * 32) return (s_kv_sel[b >> 5] >> (b & 31)) & 1u;
  return kv_seq_selected_flags(p, b);
}

// Whether this launch has nothing to do: only K/V-only rows, selected by flags, and no
// sequence selected (the usual case of a refresh launch).  Read after the barrier that
// follows select_init; every thread gets the same answer.
DEVI bool nothing_selected(const ProjParams& p) {
  if (p.kv_seq_flags == nullptr || p.m_q > 0 || p.batch > kSelWords * 32) return false;
  uint32_t any = 0u;
  for (int w = 0; w < (p.batch + 31) / 32; ++w) any |= s_kv_sel[w];
  return any == 0u;
}

// Every thread of the CTA calls this after the dependency wait; a barrier follows
// before the first kv_seq_selected.
DEVI void select_init(const ProjParams& p) {
  if (p.kv_seq_flags == nullptr || p.batch > kSelWords * 32) return;
  const int words = (p.batch + 31) / 32;
  for (int w = threadIdx.x; w < words; w += blockDim.x) {
    uint32_t bits = 0u;
    for (int i = 0; i < 32 && w * 32 + i < p.batch; ++i)
      if (kv_seq_selected_flags(p, w * 32 + i)) bits |= 1u << i;
    s_kv_sel[w] = bits;
  }
}

// A tile of K/V-only rows [m0, m0 + rows) none of whose sequences is selected: every
// role of the kernel skips it (the flags do not change while the kernel runs, so all
// roles decide alike).
DEVI bool kv_tile_skipped(const ProjParams& p, int grp, int m0, int rows) {
  if (grp == 0 || p.kv_seq_flags == nullptr) return false;
  const int m_end = min(m0 + rows, p.m_kv);
  for (int b = m0 / p.n_kv; b <= (m_end - 1) / p.n_kv; ++b)
    if (kv_seq_selected(p, b)) return false;
  return true;
}

// ---- fused drift test ("Elastic-Cache ...", Core idea: cosine similarity between the
// cached and the recomputed K/V of the tracked tokens; the refresh flag is set when
// the smallest cosine of a sequence falls below gamma).

// Add <cache, probe>, |cache|^2 and |probe|^2 over 32 columns of one head: probe values
// v (fp32, after the rotation for K), cache values already loaded from the row's slot
// (bf16: 4 vectors, or e4m3 codes: 2 vectors, times the group scale).
template <bool FP8>
DEVI void drift_dot32(const float (&v)[32], const uint4* src, float scale, float& dot, float& nc, float& np) {
  if constexpr (FP8) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 w = src[i];
      const __nv_fp8x2_storage_t* pr = reinterpret_cast<const __nv_fp8x2_storage_t*>(&w);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pr[j], __NV_E4M3)));
        const float c0 = f.x * scale, c1 = f.y * scale;
        const float p0 = v[16 * i + 2 * j], p1 = v[16 * i + 2 * j + 1];
        dot = fmaf(c0, p0, fmaf(c1, p1, dot));
        nc = fmaf(c0, c0, fmaf(c1, c1, nc));
        np = fmaf(p0, p0, fmaf(p1, p1, np));
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 w = src[i];
      const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(pr[j]);
        const float p0 = v[8 * i + 2 * j], p1 = v[8 * i + 2 * j + 1];
        dot = fmaf(f.x, p0, fmaf(f.y, p1, dot));
        nc = fmaf(f.x, f.x, fmaf(f.y, f.y, nc));
        np = fmaf(p0, p0, fmaf(p1, p1, np));
      }
    }
  }
}

// Before an epilogue waits for a probe tile's accumulator: request into L2 the cached
// K (or V) rows that its drift sums will read, for the `heads` heads of the tile, so the
// epilogue's loads hit L2 (the tile's MMAs take tens of microseconds).
DEVI void drift_prefetch_l2(const ProjParams& p, int m0, int n0, int heads, int r) {
  const int m = m0 + r;
  if (m >= p.m_kv) return;
  const int b = m / p.n_kv;
  const int pos = p.kv_positions ? __ldg(p.kv_positions + m) : m - b * p.n_kv;
  if (pos < 0 || pos >= p.max_pos) return;
  const int part = n0 / p.D;  // 1 K, 2 V
  const bool fp8 = p.kv_dtype == DLLM_E4M3;
  const size_t crow_i = (static_cast<size_t>(b) * p.slots + pos) * 2 + (part - 1);
  const int h0 = (n0 - part * p.D) / kHd;
  const char* base = static_cast<const char*>(p.cache_kv) + (crow_i * p.D + h0 * kHd) * (fp8 ? 1 : 2);
  const int bytes = heads * kHd * (fp8 ? 1 : 2);
  for (int off = 0; off < bytes; off += 128)
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(base + off));
  if (fp8) asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p.cache_scale + crow_i * p.H + h0));
}

// One tile's share of probe row m (the `heads` heads of K, part 0, or V, part 1, that
// this tile covers).  The partial sums and the row's head count are device-wide
// atomics; the contribution that completes the row (2 H heads) turns its sums into the
// two cosines and resets them, and the row that completes its sequence (n_kv rows) sets
// the sequence's refresh flag.  Rows with a position outside the cache still count
// (with no sums) and get NaN cosines, which the minimum skips.
DEVI void drift_contribute(const ProjParams& p, int m, int part, float dot, float nc, float np, bool valid) {
  // fire-and-forget reductions: the sums are read only after this kernel has finished
  // (by drift_finalize_kernel), so no fence or arrival count is needed here
  float* acc = p.drift_acc + (static_cast<size_t>(m) * 2 + part) * 3;
  if (valid) {
    atomicAdd(acc + 0, dot);
    atomicAdd(acc + 1, nc);
    atomicAdd(acc + 2, np);
  }
}

// The epilogue of one accumulator tile for this thread's row c.m0 + r: `heads` heads
// starting at output feature c.n0, read from TMEM columns tacc ...  It rotates Q and K,
// rounds to bf16 (or quantises each head to e4m3 with scale amax/448) and stores the
// row's 128-value runs to the Q rows, the probe rows or the row's cache slot.  Nothing
// is stored for rows outside the matrix, rows with out-of-range positions or view tags
// (which raise a status bit), or when `ok` is false.
DEVI void store_rows(const ProjParams& p, const TileCoord& c, int heads, uint32_t tacc, int r, bool ok) {
  const int hd = kHd;
  if (p.raw_q != nullptr || p.raw_kv != nullptr) {
    // unfused pipeline: the plain projection output (fp32, or rounded to bf16), no rotation
    const int m = c.m0 + r;
    const bool exists = ok && (c.grp == 0 ? m < p.m_q : m < p.m_kv);
    const size_t off = c.grp == 0 ? static_cast<size_t>(m) * 3 * p.D + c.n0
                                  : static_cast<size_t>(m) * 2 * p.D + (c.n0 - p.D);
    void* base = c.grp == 0 ? p.raw_q : p.raw_kv;
#pragma unroll 1
    for (int col = 0; col < heads * kHd; col += 32) {
      float v[32];
      tmem_ld32(tacc + col, v);
      if (!exists) continue;
      if (p.raw_f32) {
        uint4* d = reinterpret_cast<uint4*>(static_cast<float*>(base) + off + col);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          d[i] = make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]), __float_as_uint(v[4 * i + 2]),
                            __float_as_uint(v[4 * i + 3]));
      } else {
        store_bf16x32(static_cast<__nv_bfloat16*>(base) + off + col, v);
      }
    }
    return;
  }
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
      pos = p.kv_positions ? __ldg(p.kv_positions + m) : m - b * p.n_kv;
      slot = pos;
      valid = kv_seq_selected(p, b);
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
  if (c.grp == 1 && p.drift_acc != nullptr) {
    // fused drift test: compare this probe row's K (or V) heads with the cached ones at
    // its position; nothing is stored.  Every lane runs the TMEM loads (warp-collective),
    // also for the rows past the last probe row, which only skip the sums.
    const bool fp8 = p.kv_dtype == DLLM_E4M3;
    const size_t crow_i = (static_cast<size_t>(b) * p.slots + (valid ? slot : 0)) * 2 + (part - 1);
    float dot = 0.0f, nc = 0.0f, np = 0.0f;
#pragma unroll 1
    for (int hh = 0; hh < heads; ++hh) {
      const int h = (c.n0 - part * p.D) / kHd + hh;
      const uint32_t tcol = tacc + hh * kHd;
      const uint4* crow =
          reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.cache_kv) + (crow_i * p.D + h * hd) * (fp8 ? 1 : 2));
      // the head's cached row (256 B bf16, 128 B e4m3), loaded before the TMEM reads so
      // that all its loads are in flight at once
      uint4 cv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) cv[i] = make_uint4(0u, 0u, 0u, 0u);
      if (valid) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (!fp8 || i < 8) cv[i] = __ldg(crow + i);
      }
      const float sc = (fp8 && valid) ? __ldg(p.cache_scale + crow_i * p.H + h) : 1.0f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float lo[32], hi[32];
        tmem_ld32(tcol + half * 32, lo);
        tmem_ld32(tcol + 64 + half * 32, hi);
        if (rope) rotate32(lo, hi, cs_row + half * 32);
        if (valid) {
          // columns [32 half, +32) and [64 + 32 half, +32): 16-byte vectors 4 half / 8 + 4 half
          // (bf16) or 2 half / 4 + 2 half (e4m3)
          if (fp8) {
            drift_dot32<true>(lo, cv + 2 * half, sc, dot, nc, np);
            drift_dot32<true>(hi, cv + 4 + 2 * half, sc, dot, nc, np);
          } else {
            drift_dot32<false>(lo, cv + 4 * half, sc, dot, nc, np);
            drift_dot32<false>(hi, cv + 8 + 4 * half, sc, dot, nc, np);
          }
        }
      }
    }
    if (m < p.m_kv) drift_contribute(p, m, part - 1, dot, nc, np, valid);
    return;
  }
#pragma unroll 1
  for (int hh = 0; hh < heads; ++hh) {
    const int h = (c.n0 - part * p.D) / kHd + hh;
    const uint32_t tcol = tacc + hh * kHd;
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
  grid_dep_launch();
  grid_dep_wait();  // x, positions, indices and flags may come from the previous kernel
  select_init(p);
  __syncthreads();
  const int items_end = nothing_selected(p) ? 0 : p.items_total;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_x = p.m_fastest ? policy_evict_last() : policy_evict_first();
    const uint64_t pol_w = p.m_fastest ? policy_evict_first() : policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < items_end && ok; item += gridDim.x) {
      const Item it = decode_item(p, item);
      const TileCoord c = decode_tile(p, it.tile, BN);
      if (kv_tile_skipped(p, c.grp, c.m0, BM)) continue;
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
    for (int item = blockIdx.x; item < items_end && ok; item += gridDim.x) {
      const Item itm = decode_item(p, item);
      const TileCoord ct = decode_tile(p, itm.tile, BN);
      if (kv_tile_skipped(p, ct.grp, ct.m0, BM)) continue;
      const uint32_t idesc = itm.half >= 0 ? idesc_half : idesc_whole;
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
    bool ok = true;  // a failed wait is recorded; the item sequence continues without stores
    for (int item = blockIdx.x; item < items_end; item += gridDim.x) {
      const Item it = decode_item(p, item);
      TileCoord c = decode_tile(p, it.tile, BN);
      if (kv_tile_skipped(p, c.grp, c.m0, BM)) continue;
      if (it.half >= 0) c.n0 += it.half * kHd;
      const int heads = it.half >= 0 ? 1 : BN / kHd;
      if (c.grp == 1 && p.drift_acc != nullptr) drift_prefetch_l2(p, c.m0, c.n0, heads, r);
      if (!mbar_wait_warp(&tfull[acc], acc_phase, abort_flag)) {
        ok = false;
        *abort_flag = 1;
      }
      tc_fence_after();

      store_rows(p, c, heads, tmem_base + lane_base + acc * BN, r, ok);
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

// ------------------------------------------------------------------------------------
// CTA-pair kernel.  Two CTAs of a cluster compute one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): each CTA stages its 128 rows of x
// and its 128 rows of W per k-block (32 KB a stage instead of 48 KB), so a 6-deep ring
// fits and the loads run further ahead of the tensor core.  Rank 0 issues the MMAs and
// commits to the barriers of both CTAs; each CTA's epilogue drains its own TMEM rows.
// Tiles left over after the last full round of pairs run as 128-column halves.
// ------------------------------------------------------------------------------------
constexpr int kPairStages = 6;
constexpr uint32_t kPairBBytes = 128 * BK * 2;  // 16 KB: this CTA's half of a W k-block
constexpr uint32_t kPairStageBytes = kABytes + kPairBBytes;
constexpr size_t kPairSmem = 1024 + kPairStages * kPairStageBytes + 256;

struct PairItem {
  int grp, pm0, n0;  // row group, first row of the 256-row pair tile, first output feature
  bool half;         // a 128-column half (n0 already offset)
};

DEVI PairItem decode_pair_item(const ProjParams& p, int item) {
  int tile = item, hf = -1;
  if (item >= p.whole_items) {
    const int i = item - p.whole_items;
    tile = p.whole_items + (i >> 1);
    hf = i & 1;
  }
  PairItem it;
  if (p.m_fastest) {
    // column-major: a K or V column tile is followed by both row groups (W read once)
    const int q_cols = p.D / 256;
    const int q_tiles = q_cols * p.pmt_q;
    if (tile < q_tiles) {
      it.grp = 0;
      it.n0 = (tile / p.pmt_q) * 256;
      it.pm0 = (tile % p.pmt_q) * 256;
    } else {
      const int t = tile - q_tiles;
      const int per = p.pmt_q + p.pmt_kv;
      const int i = t % per;
      it.n0 = p.D + (t / per) * 256;
      it.grp = i < p.pmt_q ? 0 : 1;
      it.pm0 = (it.grp ? i - p.pmt_q : i) * 256;
    }
  } else {
    const int nq = 3 * p.D / 256, nkv = 2 * p.D / 256;
    const int q_tiles = p.pmt_q * nq;
    if (tile < q_tiles) {
      it.grp = 0;
      it.n0 = (tile % nq) * 256;
      it.pm0 = (tile / nq) * 256;
    } else {
      const int t = tile - q_tiles;
      it.grp = 1;
      it.n0 = p.D + (t % nkv) * 256;
      it.pm0 = (t / nkv) * 256;
    }
  }
  it.half = hf >= 0;
  if (it.half) it.n0 += hf * kHd;
  return it;
}

__global__ void __launch_bounds__(kThreads, 1)
    proj_rope_store_pair(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xkv,
                         const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_w_half,
                         const ProjParams p) {
  constexpr int STAGES = kPairStages;
  constexpr uint32_t kTmemCols = 512;  // two 256-column accumulators
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * kPairStageBytes);
  uint64_t* full = bars;                  // rank 0's: both CTAs' copies complete here
  uint64_t* empty = bars + STAGES;        // each CTA's: rank 0's MMAs done with the stage
  uint64_t* tfull = bars + 2 * STAGES;    // each CTA's: accumulator ready
  uint64_t* tempty = bars + 2 * STAGES + 2;  // rank 0's: both CTAs' epilogues drained it
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);  // four epilogue warps in each CTA
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
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dep_launch();
  // Before the dependency wait the producer only prefetches into L2 the W half of the
  // first stages of its first item (not with selection flags, whose values decide which
  // items run), so W's DRAM latency overlaps the previous kernel.  Every copy into shared
  // memory comes after the wait: the work before this call on the stream may still be
  // writing W (a cast or a dequantisation), and only L2, the device's point of
  // coherence, can be read before its writes are visible.
  if (warp == 0 && lane == 0 && p.kv_seq_flags == nullptr && pair < p.items_total) {
    const PairItem it = decode_pair_item(p, pair);
    const int b_rows = it.half ? 64 : 128;
    const CUtensorMap* bm = it.half ? &tm_w_half : &tm_w;
    const int n0 = it.n0 + static_cast<int>(rank) * b_rows;
    const int npre = p.k_blocks < kPairStages ? p.k_blocks : kPairStages;
    for (int s = 0; s < npre; ++s)
      tma_prefetch_2d_l2(bm, s * BK, n0, p.m_fastest ? policy_evict_first() : policy_evict_last());
  }
  grid_dep_wait();  // x, W, positions, indices and flags may come from the previous kernel
  select_init(p);
  __syncthreads();
  const int items_end = nothing_selected(p) ? 0 : p.items_total;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    const uint64_t pol_x = p.m_fastest ? policy_evict_last() : policy_evict_first();
    const uint64_t pol_w = p.m_fastest ? policy_evict_first() : policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int item = pair; item < items_end && ok; item += n_pairs) {
      const PairItem it = decode_pair_item(p, item);
      if (kv_tile_skipped(p, it.grp, it.pm0, 256)) continue;
      const CUtensorMap* am = it.grp ? &tm_xkv : &tm_x;
      const int b_rows = it.half ? 64 : 128;
      const CUtensorMap* bm = it.half ? &tm_w_half : &tm_w;
      const int m0 = it.pm0 + static_cast<int>(rank) * 128;
      const int n0 = it.n0 + static_cast<int>(rank) * b_rows;
      const uint32_t bytes = 2 * (kABytes + b_rows * BK * 2);  // both CTAs' copies
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        const uint32_t fb = map_to_rank(smem_u32(&full[stage]), 0);
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        if (rank == 0) mbar_arrive_expect_tx(&full[stage], bytes);
        tma_load_2d_pair(sA + stage * kABytes, am, fb, kb * BK, m0, pol_x);
        tma_load_2d_pair(sB + stage * kPairBBytes, bm, fb, kb * BK, n0, pol_w);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      raise_status(p.status, DLLM_DEV_TIMEOUT);
    }
    if (rank == 0) {
      // every copy of both CTAs lands on these barriers: wait for the last phase of each
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
        volatile int never = 0;
        mbar_wait(&full[s], par, &never);
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    constexpr uint32_t idesc_whole = idesc_bf16(256, 256, false, false);
    constexpr uint32_t idesc_half = idesc_bf16(256, 128, false, false);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int item = pair; item < items_end && ok; item += n_pairs) {
      const PairItem itm = decode_pair_item(p, item);
      if (kv_tile_skipped(p, itm.grp, itm.pm0, 256)) continue;
      const uint32_t idesc = itm.half ? idesc_half : idesc_whole;
      if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * 256;
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + stage * kABytes);
        const uint32_t b0 = smem_u32(sB + stage * kPairBBytes);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          tc_mma_f16_pair(d_tmem, sdesc_sw128(a0 + k * 32, 16, 1024), sdesc_sw128(b0 + k * 32, 16, 1024), idesc,
                          (kb | k) != 0);
        }
        tc_commit_pair(&empty[stage]);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      tc_commit_pair(&tfull[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
      *abort_flag = 1;
      raise_status(p.status, DLLM_DEV_TIMEOUT);
    }
    // Drain: every MMA issued here (into both CTAs' TMEM) finishes before TMEM is freed.
    tc_commit_pair_local(drain);
    volatile int never = 0;
    mbar_wait(drain, 0, &never);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tempty0 = map_to_rank(smem_u32(&tempty[0]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;  // a failed wait is recorded; the item sequence continues without stores
    for (int item = pair; item < items_end; item += n_pairs) {
      const PairItem it = decode_pair_item(p, item);
      if (kv_tile_skipped(p, it.grp, it.pm0, 256)) continue;
      if (it.grp == 1 && p.drift_acc != nullptr)
        drift_prefetch_l2(p, it.pm0 + static_cast<int>(rank) * 128, it.n0, it.half ? 1 : 2, r);
      if (!mbar_wait_warp(&tfull[acc], acc_phase, abort_flag)) {
        ok = false;
        *abort_flag = 1;
      }
      tc_fence_after();
      TileCoord c;
      c.grp = it.grp;
      c.m0 = it.pm0 + static_cast<int>(rank) * 128;
      c.n0 = it.n0;
      store_rows(p, c, it.half ? 1 : 2, tmem_base + lane_base + acc * 256, r, ok);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + acc * 8);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) raise_status(p.status, DLLM_DEV_TIMEOUT);
  }

  tc_fence_before();
  cluster_sync();  // no CTA leaves while its pair may still touch its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

size_t proj_tc_smem_bytes(int bn) { return bn == 256 ? Cfg<256>::kSmem : Cfg<128>::kSmem; }

// The drift test's last stage, one block per sequence, launched right after the fused
// projection on its stream: each tracked token's K and V cosines from the projection's
// partial sums (NaN for a position outside [0, max_pos)), the sums zeroed for the next
// call, and the sequence's refresh flag (min cosine < gamma; NaN cosines are skipped).
__global__ void __launch_bounds__(256) drift_finalize_kernel(const ProjParams p) {
  grid_dep_launch();
  grid_dep_wait();  // the projection's sums are complete and visible
  const int b = blockIdx.x;
  float mn = INFINITY;
  for (int i = threadIdx.x; i < 2 * p.n_kv; i += blockDim.x) {
    const int m = b * p.n_kv + (i >> 1), q = i & 1;
    const int pos = p.kv_positions ? __ldg(p.kv_positions + m) : m - b * p.n_kv;
    float* a = p.drift_acc + (static_cast<size_t>(m) * 2 + q) * 3;
    const float d = a[0], c = a[1], r = a[2];
    a[0] = 0.0f;
    a[1] = 0.0f;
    a[2] = 0.0f;
    const float den = sqrtf(c) * sqrtf(r);
    const float cs = (pos < 0 || pos >= p.max_pos) ? __int_as_float(0x7fc00000) : (den > 0.0f ? d / den : 0.0f);
    p.drift_cos[static_cast<size_t>(m) * 2 + q] = cs;
    mn = fminf(mn, cs);
  }
  if (p.drift_refresh == nullptr) return;
  __shared__ float red[8];
  for (int o = 16; o >= 1; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mn;
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = red[0];
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) v = fminf(v, red[w]);
    p.drift_refresh[b] = (v < p.drift_gamma) ? 1 : 0;
  }
}

int launch_proj_tc(const ProjParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_xkv,
                   const CUtensorMap& tm_w, const CUtensorMap& tm_w_half, int bn, int grid, cudaStream_t s) {
  cudaError_t e;
  if (bn == 256) {
    auto k = proj_rope_store_tc<256>;
    e = ensure_smem_limit(reinterpret_cast<const void*>(k), (int)(Cfg<256>::kSmem));
    if (e != cudaSuccess) return (int)e;
    e = launch_pdl(k, dim3(grid), dim3(kThreads), Cfg<256>::kSmem, s, tm_x, tm_xkv, tm_w, tm_w_half, p);
    if (e != cudaSuccess) return (int)e;
  } else {
    auto k = proj_rope_store_tc<128>;
    e = ensure_smem_limit(reinterpret_cast<const void*>(k), (int)(Cfg<128>::kSmem));
    if (e != cudaSuccess) return (int)e;
    e = launch_pdl(k, dim3(grid), dim3(kThreads), Cfg<128>::kSmem, s, tm_x, tm_xkv, tm_w, tm_w_half, p);
    if (e != cudaSuccess) return (int)e;
  }
  return (int)cudaGetLastError();
}

int launch_drift_finalize(const ProjParams& p, cudaStream_t s) {
  return (int)launch_pdl(drift_finalize_kernel, dim3(p.batch), dim3(256), 0, s, p);
}

int launch_proj_pair(const ProjParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_xkv,
                     const CUtensorMap& tm_w, const CUtensorMap& tm_w_half, int grid, cudaStream_t s) {
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(proj_rope_store_pair), (int)(kPairSmem));
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, proj_rope_store_pair, tm_x, tm_xkv, tm_w, tm_w_half, p);
  if (e != cudaSuccess) return (int)e;
  return (int)cudaGetLastError();
}

// Clusters of two CTAs of the pair kernel that the device can hold at once.
int proj_pair_max_clusters(int* clusters) {
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(proj_rope_store_pair), (int)(kPairSmem));
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kPairSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaOccupancyMaxActiveClusters(clusters, proj_rope_store_pair, &cfg);
}

}  // namespace dllm
