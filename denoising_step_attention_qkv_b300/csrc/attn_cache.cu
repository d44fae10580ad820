// Bidirectional attention of a step's query rows over the flat K/V cache
// (tensor-core path, bf16 and FP8-e4m3 caches).
//
// "LaCache ...", technical summary, Problem Statement: inside a block every query
// attends to the full context (non-causal).  "Flash-Cache" article, section 3.1:
// softmax(q k^T / sqrt(d)) v fused in one kernel.  "Flash-dLLM ...", paragraph 3:
// Flash-Verify draft and mask views must not see each other.
//
// Design (sm_103a).  A work unit is (sequence b, head h, chunk of <= NQ query rows,
// key split) and is processed by one persistent CTA.  Per 128-key tile the MMA warp
// computes S^T = K Q^T with tcgen05 (M = 128 keys, N = NQ queries, K = hd = 128) into
// TMEM, so a softmax thread owns one key and holds that key's scores for the queries
// of its warpgroup (with e4m3 caches and with 48 query columns two softmax warpgroups
// split the columns in halves and run independently); per-query maxima and sums are
// warp reductions plus a 4-warp exchange in shared memory, and the online softmax runs
// in fp32 with exp2.  The thread writes its key's
// probabilities as bf16 into the P tile (MN-major: each key's query columns contiguous,
// eight of them per 16-byte store) and the MMA warp computes O^T = V^T P^T (M = hd,
// N = NQ, V read MN-major straight from the TMA-staged cache tile) into TMEM, which the
// same threads fold into fp32 register accumulators.
//
// The softmax of one tile is a chain of dependent steps, kept short: per-query maxima
// come from redux.sync (one instruction per query and warp) and a 4-warp exchange;
// the row sums are kept per thread (each thread rescales its own partial sums) and
// reduced once per unit; exponentials use ex2.approx and two probabilities share one
// packed bf16 conversion.  S, P and O are double-buffered so the loads, both MMAs and
// the softmax overlap; K/V tiles stream through TMA rings and Q is double-buffered, so
// the next unit's loads start while this one finishes.  With few units, keys are
// split across CTAs and a second kernel merges the partial (O, m, l) states.
//
// FP8-e4m3 cache ("LaCache ...", Methodology 2: per-group FP8; one group here = one
// head of one token, K or V, with an fp32 scale): TMA stages the e4m3 tiles (half the
// bytes of bf16) in a 3-deep ring (2 with 64 queries).  The staged K codes are the A
// operand of an 8-bit S MMA (kind::f8f6f4) as they are: a key's K scale is constant
// along its row of the score tile, so the softmax folds it into that row's logit scale
// (in fp32).  The B operand is the unit's Q chunk as two e4m3 parts, Q_hi = e4m3(s q)
// and Q_lo = e4m3(s q - Q_hi), with one scale s per chunk that takes its largest |q| to
// 448: two MMAs give K (Q_hi + Q_lo)^T, within about 2^-9 of K (s Q)^T per term, as
// close as bf16's rounding of Q; 1/s joins the logit scale.  Four converter warps split
// Q once per unit and turn each V tile into an f16 operand, code times the group's
// scale (one f16 multiply per pair, a single f16 rounding of relative size 2^-11, far
// below the e4m3 step of 2^-4); the softmax writes P as f16 for the f16 P V MMA.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace dllm {
namespace {

constexpr uint32_t kTileBytes = kKeyTile * kHd * 2;  // 32 KB (bf16 K or V tile)
constexpr uint32_t kTile8Bytes = kKeyTile * kHd;     // 16 KB (e4m3 tile)
constexpr int kMaxBitmapWords = 512;                 // MASK-slot bitmap: max_pos <= 16384
constexpr int kMaxOrder = 256;                       // ragged batches: sequences ranked by length

// Per (query columns, cache type): MMA-operand rings for K and V, e4m3 staging rings,
// thread count.
template <int NQ, bool FP8>
struct Cfg {
  // e4m3: the staging ring (TMA -> converters) and the V operand ring are 2 deep and the
  // K operand ring 1 deep with 32 queries (measured best of the splits that fit); with
  // 64 queries only the staging ring is doubled
  static constexpr int KST = FP8 ? 1 : (NQ <= 48 ? 3 : 2);
  static constexpr uint32_t kKBytes = FP8 ? 1024 : kTileBytes;  // e4m3: the K codes feed the MMA from staging
  static constexpr int VST = FP8 ? (NQ == 32 ? 2 : 1) : 2;
  static constexpr int SST = FP8 ? (NQ == 64 ? 2 : 3) : 1;
  static constexpr uint32_t kStageBytes = FP8 ? kTile8Bytes : 1024;
  static constexpr uint32_t kQBytes = NQ * kHd * 2;       // one Q chunk (two 64-column boxes)
  static constexpr uint32_t kPBytes = NQ * kKeyTile * 2;  // one P^T tile (two 64-key halves)
  // softmax warpgroups, each owning NQ / kSmWG query columns: two where the softmax's
  // per-tile chain bounds the kernel (e4m3 caches, 48 columns), one where HBM does
  static constexpr int kSmWG = (FP8 || NQ == 48) ? 2 : 1;
  static constexpr int kThreads = 64 + 128 * kSmWG + (FP8 ? 128 : 0);  // TMA + MMA, softmax, converters
};

template <int NQ, bool FP8>
struct Smem {
  using C = Cfg<NQ, FP8>;
  // all operand tiles 1024-byte aligned
  uint8_t q[2][C::kQBytes];
  uint8_t k[C::KST][C::kKBytes];
  uint8_t v[C::VST][kTileBytes];
  uint8_t p[2][C::kPBytes];
  uint8_t q8[2][2][FP8 ? NQ * 128 : 1024];  // e4m3: per Q buffer, the high and low e4m3 parts of Q
  uint8_t sk[C::SST][C::kStageBytes];  // e4m3 staging (FP8 only)
  uint8_t sv[C::SST][C::kStageBytes];
  float red[4][NQ];  // per-warp column maxima (per tile) / partial sums (per unit)
  float m_run[NQ];
  float m_use[NQ];
  float alpha[2][NQ];
  float l_fin[NQ];
  float inv_l[NQ];
  float fin_alpha[2][NQ];  // per unit parity: the last tile's rescale factor and running max
  float fin_m[2][NQ];
  float mrg_a[NQ], mrg_c[NQ];  // merge with a cached state: weights of this range's and the cached O
  uint32_t mask_bits[kMaxBitmapWords];
  int seq_order[kMaxOrder];  // ragged batches: sequences by key length, longest first
  uint32_t draft_qmask[2];
  int n_draft;
  float q8inv[2];       // e4m3: per Q buffer, 1 / the scale that took the chunk's max |q| to 448
  float cv_red[2][4];   // e4m3: per Q buffer, the converter warps' max |q|
  int merge_last[2];    // per softmax warpgroup: this piece completed its tail unit
  float mrg_w[kMaxPieces][NQ];  // merge of a tail unit's pieces: weight of piece j, column q
  uint64_t q_full[2], q_empty[2];
  uint64_t q_conv[2];  // e4m3 caches: the Q chunk has been converted to f16 in place
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
static_assert(sizeof(Smem<32, false>) + 1024 <= 232448, "shared memory budget (bf16, 32 queries)");
static_assert(sizeof(Smem<64, false>) + 1024 <= 232448, "shared memory budget (bf16, 64 queries)");
static_assert(sizeof(Smem<48, false>) + 1024 <= 232448, "shared memory budget (bf16, 48 queries)");
static_assert(sizeof(Smem<48, true>) + 1024 <= 232448, "shared memory budget (e4m3, 48 queries)");
static_assert(sizeof(Smem<32, true>) + 1024 <= 232448, "shared memory budget (e4m3, 32 queries)");
static_assert(sizeof(Smem<64, true>) + 1024 <= 232448, "shared memory budget (e4m3, 64 queries)");

// Dequantise 16 e4m3 codes of one group to f16: code (exact in f16) times the group's
// scale, one f16 rounding.
DEVI void dequant16_f16(const uint4 in, __half2 scale, uint4& lo, uint4& hi) {
  const __nv_fp8x2_storage_t* pr = reinterpret_cast<const __nv_fp8x2_storage_t*>(&in);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 h = __hmul2(__half2(__nv_cvt_fp8x2_to_halfraw2(pr[i], __NV_E4M3)), scale);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
}

struct Unit {
  int b, h, qc, split, t0, t1;
  int u;      // the unit's number (before the ragged reordering)
  int part;   // 1: a piece of a tail unit (its state is merged with the other pieces')
  int piece;  // which piece, and which tail unit (part == 1)
  int tu;
};

// Unit u -> (sequence, head, query chunk, key split).  With `order` (ragged batches) the
// sequence part of u is a rank in order of decreasing key length.
DEVI Unit decode_unit(const AttnParams& p, int u, const int* order) {
  Unit x;
  x.u = u;
  x.part = 0;
  x.piece = 0;
  x.tu = 0;
  x.split = u % p.n_splits;
  u /= p.n_splits;
  x.qc = u % p.n_qchunks;
  u /= p.n_qchunks;
  x.h = u % p.H;
  x.b = u / p.H;
  if (order) x.b = order[x.b];
  x.t0 = p.tile_lo + x.split * p.tiles_per_split;
  x.t1 = min(p.tile_lo + p.key_tiles, x.t0 + p.tiles_per_split);
  if (p.key_len) {  // ragged batch: nothing past this sequence's length
    const int len = min(max(p.key_len[x.b], 0), p.max_pos);
    x.t1 = min(x.t1, (len + kKeyTile - 1) / kKeyTile);
  }
  if (x.t0 > x.t1) x.t0 = x.t1;  // a unit may be empty
  return x;
}

// The r-th unit this CTA processes.  Round-robin over the CTAs; for ragged batches, whose
// units are numbered longest first, a snake (CTA c takes the c-th unit of even rounds and
// the (P-1-c)-th of odd ones), so that long units pair with short ones across rounds.
// Increasing in r for every CTA.
DEVI int cta_unit(const AttnParams& p, int r) {
  const int c = (p.key_len && (r & 1)) ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  return r * static_cast<int>(gridDim.x) + c;
}

// The rnd-th work item of this CTA; false past its last.  Without tail pieces: the
// round-robin over the units (cta_unit).  With them (tail_pieces > 0): dp_waves rounds
// of whole units, round-robin, then the last tail_units units, each cut into
// tail_pieces pieces of piece_tiles key tiles, dealt round-robin piece-major (item i of
// the tail is piece i / tail_units of tail unit i % tail_units), so that neighbouring
// CTAs read the same slots of neighbouring heads in both phases.  Every warp role walks
// the same items.
template <bool PIECES>
DEVI bool cta_item(const AttnParams& p, int rnd, const int* order, Unit& x) {
  if (!PIECES || p.tail_pieces == 0) {
    const int u = cta_unit(p, rnd);
    if (u >= p.units) return false;
    x = decode_unit(p, u, order);
    return true;
  }
  const int g = static_cast<int>(gridDim.x);
  const int i0 = rnd * g + static_cast<int>(blockIdx.x);
  const int whole = p.dp_waves * g;
  if (i0 < whole) {
    x = decode_unit(p, i0, nullptr);
    return true;
  }
  const int i = i0 - whole;
  if (i >= p.tail_units * p.tail_pieces) return false;
  const int piece = i / p.tail_units, tu = i - piece * p.tail_units;
  x = decode_unit(p, whole + tu, nullptr);
  x.t0 = p.tile_lo + piece * p.piece_tiles;
  x.t1 = min(p.tile_lo + p.key_tiles, x.t0 + p.piece_tiles);
  x.part = p.tail_pieces > 1 ? 1 : 0;
  x.piece = piece;
  x.tu = tu;
  return true;
}

// End (exclusive) of the regular slots sequence b attends to.
DEVI int key_end(const AttnParams& p, int b) {
  const int len = p.key_len ? min(max(p.key_len[b], 0), p.max_pos) : p.max_pos;
  return min(p.key_hi, len);
}


// Maximum of v over the 32 lanes of the warp, in every lane.
DEVI float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// 2^x (PTX ex2.approx.ftz.f32: relative error about 2^-22, far below the bf16 rounding
// that every probability goes through; 2^-inf = +0).
DEVI float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (a, b) rounded to bf16 (F16: to f16), a in the low half.
template <bool F16 = false>
DEVI uint32_t pack_pair(float a, float b) {
  uint32_t packed;
  if constexpr (F16)
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(packed) : "f"(b), "f"(a));  // hi = b, lo = a
  else
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed) : "f"(b), "f"(a));
  return packed;
}

// The P tile of the P V product, the MMA's B operand (K = keys, N = query columns),
// stored MN-major: key r's row holds its NQ columns contiguously, so the softmax thread
// that owns key r writes eight columns with one 16-byte store.  Rows of 64 bytes with
// the 64-byte swizzle (32 columns), of 128 bytes with the 128-byte swizzle (64), or,
// with 48 columns, three strips of 16 columns (32-byte swizzle), each strip 128 rows
// of 32 bytes, 4 KB apart.  Byte offset of columns [q, q + 8) of row r (q a multiple
// of 8), and the descriptor of the 16 rows from row 16 kk on.
template <int NQ>
DEVI uint32_t p_chunk_offset(uint32_t r, uint32_t q) {
  if constexpr (NQ == 32) {
    return r * 64u + ((((q >> 3) ^ (r >> 1)) & 3u) << 4);
  } else if constexpr (NQ == 64) {
    return r * 128u + ((((q >> 3) ^ r) & 7u) << 4);
  } else {
    static_assert(NQ == 48, "query columns of a P tile");
    return (q >> 4) * 4096u + r * 32u + ((((q >> 3) ^ (r >> 2)) & 1u) << 4);
  }
}
template <int NQ>
DEVI uint64_t p_desc(uint32_t p0, int kk) {
  if constexpr (NQ == 32) return sdesc_swz(p0 + kk * 1024u, 1024, 512, 4);
  else if constexpr (NQ == 64) return sdesc_swz(p0 + kk * 2048u, 1024, 1024, 2);
  else return sdesc_swz(p0 + kk * 512u, 4096, 256, 6);
}

// Reduce 32 per-lane values per column, for C columns (C = 8, 16 or 32), across the
// warp; afterwards lane i holds the reduction of column i % C.  Each step halves the
// columns a lane keeps and exchanges the other half with the lane whose id differs in
// that bit; the lanes that then hold the same column add theirs.
template <bool MAX, int C>
DEVI float reduce_scatter(float* v, int lane) {
#pragma unroll
  for (int w = C / 2; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  float r = v[0];
#pragma unroll
  for (int w = C; w < 32; w <<= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, r, w);
    r = MAX ? fmaxf(r, o) : r + o;
  }
  return r;
}

// Column sums of QH per-lane values over the warp, written to dst[0 .. QH) (QH = 16, 24,
// 32 or 64); clobbers l.
template <int QH>
DEVI void reduce_cols(float (&l)[QH], float* dst, int lane) {
  if constexpr (QH % 32 == 0) {
#pragma unroll
    for (int c = 0; c < QH; c += 32) dst[c + lane] = reduce_scatter<false, 32>(l + c, lane);
  } else if constexpr (QH == 16) {
    const float v = reduce_scatter<false, 16>(l, lane);
    if (lane < 16) dst[lane] = v;
  } else {
    static_assert(QH == 24, "query columns per warpgroup");
    const float v = reduce_scatter<false, 16>(l, lane);
    if (lane < 16) dst[lane] = v;
    const float v8 = reduce_scatter<false, 8>(l + 16, lane);
    if (lane < 8) dst[16 + lane] = v8;
  }
}

// Load N TMEM columns of this warp's lanes in chunks of 32 (of 16, or of 8 when N is not
// a multiple of 16), each chunk starting at a multiple of its width.
template <int N>
DEVI void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
  if constexpr (N % 32 == 0) {
#pragma unroll
    for (int c = 0; c < N; c += 32) tmem_ld32(taddr + c, *reinterpret_cast<float(*)[32]>(v + c));
  } else if constexpr (N % 16 == 0) {
#pragma unroll
    for (int c = 0; c < N; c += 16) tmem_ld16(taddr + c, *reinterpret_cast<float(*)[16]>(v + c));
  } else {
    static_assert(N % 8 == 0, "TMEM column chunks");
#pragma unroll
    for (int c = 0; c < N; c += 8) tmem_ld8(taddr + c, *reinterpret_cast<float(*)[8]>(v + c));
  }
}

// PIECES: the instantiation that runs the balanced schedule's tail pieces and their
// merge (bf16 caches only); the others contain neither, so that code does not weigh on
// their tile loop.
template <int NQ, bool FP8, bool PIECES>
__global__ void __launch_bounds__(Cfg<NQ, FP8>::kThreads, 1)
    attn_cache_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                  const __grid_constant__ CUtensorMap tm_kv_tail, const AttnParams p) {
  static_assert(!(PIECES && FP8), "tail pieces are scheduled for bf16 caches only");
  using C = Cfg<NQ, FP8>;
  constexpr int KST = C::KST, VST = C::VST, SST = C::SST;
  constexpr int kSmWarps = 4 * C::kSmWG;  // softmax warps
  constexpr int QH = NQ / C::kSmWG;      // query columns of each softmax warpgroup
  // With 32 bf16 queries a unit's finish runs inside the next unit's first tile (see the
  // softmax warps); the other variants finish at the unit's end.
  constexpr bool kDefer = (NQ == 32) && !FP8;
  extern __shared__ uint8_t smem_raw[];
  Smem<NQ, FP8>& S =
      *reinterpret_cast<Smem<NQ, FP8>*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  volatile int* abort_flag = &S.abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr uint32_t kTmemCols = 4 * NQ <= 128 ? 128 : (4 * NQ <= 256 ? 256 : 512);  // S[2] then O[2]
  constexpr uint32_t kQBox = NQ * 128;    // bytes of one 64-column Q box

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.q_full[i], 1);
      mbar_init(&S.q_empty[i], 1);
      mbar_init(&S.q_conv[i], 4);  // the four converter warps (e4m3 caches)
    }
    // bf16: operand tiles are filled by TMA (one arrival + bytes); e4m3: by 4 converter warps
    for (int i = 0; i < KST; ++i) { mbar_init(&S.k_full[i], FP8 ? 4 : 1); mbar_init(&S.k_empty[i], 1); }
    for (int i = 0; i < VST; ++i) { mbar_init(&S.v_full[i], FP8 ? 4 : 1); mbar_init(&S.v_empty[i], 1); }
    for (int i = 0; i < SST; ++i) {
      mbar_init(&S.sk_full[i], 1);
      mbar_init(&S.sk_empty[i], 1);  // e4m3: the S MMA that read the staged K codes
      mbar_init(&S.sv_full[i], 1);
      mbar_init(&S.sv_empty[i], 4);  // the four converter warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.s_full[i], 1);
      mbar_init(&S.s_free[i], kSmWarps);  // one arrival per softmax warp
      mbar_init(&S.p_full[i], kSmWarps);
      mbar_init(&S.p_empty[i], 1);
      mbar_init(&S.o_full[i], 1);
      mbar_init(&S.o_free[i], kSmWarps);
    }
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_kv);
    if (p.tail_rows) prefetch_tmap(&tm_kv_tail);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // Keys split over CTAs (fewer units than SMs, as with batch 1: each CTA runs a few
  // tiles, so the first loads' latency is most of its time): the K and V tiles of the
  // CTA's first unit (as many as the rings hold) are requested into L2 before the wait
  // for the previous kernel, so that the loads after it hit L2.  A prefetch returns no
  // data, and L2 is the point of coherence, so rows that kernel writes (the block's own
  // slots) are still read as written.  Ragged batches, whose unit order needs their
  // lengths, and tiles past the slots are left out.  (With every SM running whole units
  // the same prefetch measured slower: its traffic competes with the first loads.)
  if (warp == 0 && lane == 0 && p.n_splits > 1 && p.key_len == nullptr) {
    Unit y;
    if (cta_item<PIECES>(p, 0, nullptr, y)) {
      const uint64_t pol = policy_evict_last();  // kept until the loads after the wait
      const int t_end = min(y.t1, y.t0 + (FP8 ? SST : KST));
      for (int t = y.t0; t < t_end && (t + 1) * kKeyTile <= p.slots; ++t) {
        const int key0 = y.b * p.slots + t * kKeyTile;
        if constexpr (FP8) {
          tma_prefetch_3d_l2(&tm_kv, 0, y.h, key0, pol);
          tma_prefetch_3d_l2(&tm_kv, 0, p.H + y.h, key0, pol);
        } else {
          for (int c = 0; c < kHd; c += 64) {
            tma_prefetch_3d_l2(&tm_kv, c, y.h, key0, pol);
            tma_prefetch_3d_l2(&tm_kv, c, p.H + y.h, key0, pol);
          }
        }
      }
    }
  }
  // Everything below may read what the previous kernel on the stream wrote.
  grid_dep_launch();
  grid_dep_wait();
  // Ragged batch: rank the sequences by key length (longest first, ties by index).
  const int* order = nullptr;
  if (p.key_len && p.B <= kMaxOrder) {
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
      const int lb = min(max(__ldg(p.key_len + b), 0), p.max_pos);
      int rank = 0;
      for (int o = 0; o < p.B; ++o) {
        const int lo = min(max(__ldg(p.key_len + o), 0), p.max_pos);
        rank += (lo > lb) || (lo == lb && o < b);
      }
      S.seq_order[rank] = b;
    }
    order = S.seq_order;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_q = policy_evict_last();
    int ks = 0, vs = 0, uu = 0;
    uint32_t kph = 0, vph = 0;
    bool ok = true;
    Unit x;
    for (int rnd = 0; ok && cta_item<PIECES>(p, rnd, order, x); ++rnd, ++uu) {
      const int qb = uu & 1;
      if (!mbar_wait(&S.q_empty[qb], ((uu >> 1) & 1) ^ 1u, abort_flag)) { ok = false; break; }
      mbar_arrive_expect_tx(&S.q_full[qb], 2 * kQBox);
      const int qrow = x.b * p.n_tok + x.qc * kQChunk;
      tma_load_2d(S.q[qb], &tm_q, &S.q_full[qb], x.h * kHd, qrow, pol_q);
      tma_load_2d(S.q[qb] + kQBox, &tm_q, &S.q_full[qb], x.h * kHd + 64, qrow, pol_q);
      const int slot0 = x.b * p.slots;
      for (int t = x.t0; t < x.t1; ++t) {
        const int key0 = slot0 + t * kKeyTile;
        // A tile that runs past the sequence's slots (the Flash-Verify draft tail, or a
        // slot count that is not a multiple of 128) loads only its first tail_rows rows;
        // the rows after them are keys no query sees (their scores are masked, their V
        // rows zeroed before the P V MMA).
        const bool trim = p.tail_rows != 0 && (t + 1) * kKeyTile > p.slots;
        const CUtensorMap* mkv = trim ? &tm_kv_tail : &tm_kv;
        const uint32_t rows = trim ? static_cast<uint32_t>(p.tail_rows) : static_cast<uint32_t>(kKeyTile);
        if constexpr (FP8) {
          // e4m3 tiles into the staging rings (one 128-byte-wide box each)
          if (!mbar_wait(&S.sk_empty[ks], kph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.sk_full[ks], rows * 128u);
          tma_load_3d(S.sk[ks], mkv, &S.sk_full[ks], 0, x.h, key0, pol_stream);
          if (!mbar_wait(&S.sv_empty[ks], kph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.sv_full[ks], rows * 128u);
          tma_load_3d(S.sv[ks], mkv, &S.sv_full[ks], 0, p.H + x.h, key0, pol_stream);
          if (++ks == SST) { ks = 0; kph ^= 1u; }
        } else {
          if (!mbar_wait(&S.k_empty[ks], kph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.k_full[ks], rows * 256u);
          tma_load_3d(S.k[ks], mkv, &S.k_full[ks], 0, x.h, key0, pol_stream);
          tma_load_3d(S.k[ks] + kTileBytes / 2, mkv, &S.k_full[ks], 64, x.h, key0, pol_stream);
          if (++ks == KST) { ks = 0; kph ^= 1u; }
          if (!mbar_wait(&S.v_empty[vs], vph ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.v_full[vs], rows * 256u);
          tma_load_3d(S.v[vs], mkv, &S.v_full[vs], 0, p.H + x.h, key0, pol_stream);
          tma_load_3d(S.v[vs] + kTileBytes / 2, mkv, &S.v_full[vs], 64, p.H + x.h, key0, pol_stream);
          if (++vs == VST) { vs = 0; vph ^= 1u; }
        }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.status, DLLM_DEV_TIMEOUT);
    }
    // let every copy issued here land before the CTA can exit: on each ring slot, wait
    // for the most recent phase armed on it (a slot never armed passes at once)
    volatile int never = 0;
    const int qn = uu & 1;
    const uint32_t qph = (uu >> 1) & 1u;
    for (int i = 0; i < 2; ++i) mbar_wait(&S.q_full[i], (i < qn) ? qph : (qph ^ 1u), &never);
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
    // Per tile: S(t) = K(t) Q^T into S[t & 1], then P V of the previous tile into
    // O[(t - 1) & 1], so the softmax of tile t - 1 overlaps the S MMA of tile t.  With
    // e4m3 caches P V of tile t - 2 follows S(t) instead (kLag): a P V waits for the
    // converters' f16 V tile, and the next tiles' scores should not queue behind it.
    // e4m3 caches: S on the 8-bit path (K codes x the two e4m3 parts of Q), P V in f16
    constexpr uint32_t idesc_s = FP8 ? idesc_e4m3(128, NQ) : idesc_bf16(128, NQ, false, false);
    constexpr uint32_t idesc_o = FP8 ? idesc_f16(128, NQ, true, true) : idesc_bf16(128, NQ, true, true);
    int ks = 0, vs = 0, uu = 0;
    uint32_t kph = 0, vph = 0;
    uint32_t s_cnt = 0, pv_cnt = 0;
    bool ok = true;

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
        const uint64_t b = p_desc<NQ>(p0, kk);
        tc_mma_f16(d, a, b, idesc_o, kk != 0);
      }
      tc_commit(&S.v_empty[vs]);
      tc_commit(&S.p_empty[pb]);
      tc_commit(&S.o_full[pb]);
      if (++vs == VST) { vs = 0; vph ^= 1u; }
      ++pv_cnt;
      return true;
    };

    // With a deferred finish, the P V of a unit's last tile stays pending until the next
    // unit's first S MMA has been issued (or an empty unit, or the end), so at unit
    // boundaries too the softmax finds its next S ready.  Without one, the softmax's
    // finish waits for that P V, so it is issued at once.
    constexpr uint32_t kLag = FP8 ? 2 : 1;  // P V products pending after an S MMA
    Unit x;
    for (int rnd = 0; ok && cta_item<PIECES>(p, rnd, order, x); ++rnd, ++uu) {
      const int qb = uu & 1;
      if (x.t1 == x.t0) {
        while (ok && pv_cnt != s_cnt) ok = issue_pv();
        if (!ok) break;
      }
      if (!mbar_wait(FP8 ? &S.q_conv[qb] : &S.q_full[qb], (uu >> 1) & 1u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t q0 = smem_u32(S.q[qb]);
      for (int t = x.t0; t < x.t1 && ok; ++t) {
        const uint32_t sb = s_cnt & 1u, sph = (s_cnt >> 1) & 1u;
        if (!mbar_wait(&S.s_free[sb], sph ^ 1u, abort_flag)) { ok = false; break; }
        if (!mbar_wait(FP8 ? &S.sk_full[ks] : &S.k_full[ks], kph, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + sb * NQ;
        if constexpr (FP8) {
          // S^T = K codes (Q_hi + Q_lo)^T straight from the staged tile: one 128-byte row
          // of codes per key, four K = 32 steps for each part of Q
          const uint32_t k0 = smem_u32(S.sk[ks]);
          const uint32_t qh = smem_u32(S.q8[qb][0]), ql = smem_u32(S.q8[qb][1]);
#pragma unroll
          for (int kk = 0; kk < kHd / 32; ++kk)
            tc_mma_f8(d, sdesc_sw128(k0 + kk * 32, 16, 1024), sdesc_sw128(qh + kk * 32, 16, 1024), idesc_s, kk != 0);
#pragma unroll
          for (int kk = 0; kk < kHd / 32; ++kk)
            tc_mma_f8(d, sdesc_sw128(k0 + kk * 32, 16, 1024), sdesc_sw128(ql + kk * 32, 16, 1024), idesc_s, 1u);
          tc_commit(&S.sk_empty[ks]);
        } else {
          const uint32_t k0 = smem_u32(S.k[ks]);
#pragma unroll
          for (int kk = 0; kk < kHd / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
            const uint32_t qoff = (kk >> 2) * kQBox + (kk & 3) * 32;
            tc_mma_f16(d, sdesc_sw128(k0 + off, 16, 1024), sdesc_sw128(q0 + qoff, 16, 1024), idesc_s, kk != 0);
          }
          tc_commit(&S.k_empty[ks]);
        }
        tc_commit(&S.s_full[sb]);
        if (++ks == (FP8 ? SST : KST)) { ks = 0; kph ^= 1u; }
        ++s_cnt;
        while (ok && s_cnt - pv_cnt > kLag) ok = issue_pv();
      }
      if (!ok) break;
      if (!kDefer) {
        while (ok && pv_cnt != s_cnt) ok = issue_pv();
        if (!ok) break;
      }
      tc_commit(&S.q_empty[qb]);
    }
    while (ok && pv_cnt != s_cnt) ok = issue_pv();
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.status, DLLM_DEV_TIMEOUT);
    }
    tc_commit(&S.drain);
    volatile int never = 0;
    mbar_wait(&S.drain, 0, &never);
  } else if (warp >= 2 && warp < 2 + kSmWarps) {
    // ------------------------------------------------------------------ softmax warps
    // One or two warpgroups (kSmWG), g = 0 (warps 2-5) and g = 1 (warps 6-9), each owning
    // QH = NQ / kSmWG of the query columns, [q0, q0 + QH).  Warp w reads TMEM lanes 32 * (w % 4) .., so thread r
    // of either warpgroup owns key r of the S^T tile and hd index r of the O^T tile, for
    // its warpgroup's columns.  The warpgroups run independently (their own named
    // barriers; the per-query shared arrays are indexed by column), and meet only in the
    // per-unit Flash-Verify set-up.  Every warp runs the same sequence of barriers; a
    // failed wait is recorded and the sequence continues, so no warp is left waiting at
    // a barrier.
    const int g = C::kSmWG == 1 ? 0 : (warp - 2) >> 2;  // compile-time 0 with one warpgroup
    const int q0 = g * QH;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int tid = g * 128 + r;  // over every softmax warpgroup
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const bool has_view = p.view != nullptr;
    uint32_t s_cnt = 0, pv_cnt = 0;
    int vs = 0;  // V ring position, mirrors the producer
    uint32_t vph = 0;
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t par) {
      if (!mbar_wait(bar, par, abort_flag)) {
        ok = false;
        *abort_flag = 1;
      }
    };
    auto wg_sync = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory"); };
    auto both_sync = [&]() { asm volatile("bar.sync 3, %0;" ::"r"(kSmWarps * 32) : "memory"); };
    const int mask_words = (p.max_pos + 31) >> 5;

    // Finishing a unit (fold its last P V, reduce the row sums, write the output or the
    // split partials) waits for that P V MMA.  With 32 bf16 queries the finish is
    // deferred into the next unit's first tile, whose P V fold slot is empty, so the
    // wait hides behind that tile's softmax.
    constexpr int kSt = kHd + 2;
    // can_merge (a constant at every call site): whether this call may finish a
    // tail unit's piece (deferred finishes never do: pieces finish at once, which keeps the
    // merge's registers out of the tile loop).
    auto finish = [&](bool can_merge, float (&o)[QH], float (&l)[QH], const Unit& fx, int fuu, uint32_t fpv) {
      const bool has_pv = fx.t1 > fx.t0;  // an empty unit (ragged batch, key range) has none
      const int frow0 = fx.b * p.n_tok + fx.qc * kQChunk;
      const int fnrows = min(kQChunk, p.n_tok - fx.qc * kQChunk);
      // a cached state to merge: this thread's O values of it are requested into L1 before
      // the wait for the last P V, so that their latency overlaps it
      const float* stc = p.state_in + static_cast<size_t>(frow0) * p.H * kSt + fx.h * kSt + r;
      if (p.state_in != nullptr) {
#pragma unroll
        for (int i = 0; i < QH; ++i)
          if (q0 + i < fnrows) asm volatile("prefetch.global.L1 [%0];" ::"l"(stc + static_cast<size_t>(q0 + i) * p.H * kSt));
      }
      if (has_pv) {
        const uint32_t ob = fpv & 1u, oph = (fpv >> 1) & 1u;  // the unit's last P V
        wait(&S.o_full[ob], oph);
        tc_fence_after();
        const float4* al4 = reinterpret_cast<const float4*>(S.fin_alpha[fuu & 1] + q0);
        {
          float tmp[QH];
          tmem_ld_cols<QH>(tmem + lane_base + 2 * NQ + ob * NQ + q0, tmp);
#pragma unroll
          for (int i = 0; i < QH; i += 4) {
            const float4 al = al4[i / 4];
            o[i] = o[i] * al.x + tmp[i];
            o[i + 1] = o[i + 1] * al.y + tmp[i + 1];
            o[i + 2] = o[i + 2] * al.z + tmp[i + 2];
            o[i + 3] = o[i + 3] * al.w + tmp[i + 3];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.o_free[ob]);
      }
      // row sums: reduce the per-key partial sums over the warpgroup's 128 threads
      reduce_cols<QH>(l, S.red[quarter] + q0, lane);
      wg_sync();
      if (r < QH) {
        const int q = q0 + r;
        const float lt = S.red[0][q] + S.red[1][q] + S.red[2][q] + S.red[3][q];
        S.l_fin[q] = lt;
        if (p.state_in != nullptr) {
          // merge with the cached state of the other keys (LaCache, FACache): M = max of
          // both maxima, each side weighted by 2^(m - M)
          const float ma = has_pv ? S.fin_m[fuu & 1][q] : -INFINITY;
          float mc = -INFINITY, lc = 0.0f;
          if (q < fnrows) {
            const float2 ml = __ldg(reinterpret_cast<const float2*>(
                p.state_in + (static_cast<size_t>(frow0 + q) * p.H + fx.h) * kSt + kHd));
            mc = ml.x;
            lc = ml.y;
          }
          const float M = fmaxf(ma, mc);
          const float wa = (ma == -INFINITY) ? 0.0f : exp2f(ma - M);
          const float wc = (mc == -INFINITY) ? 0.0f : exp2f(mc - M);
          const float L = lt * wa + lc * wc;
          S.mrg_a[q] = wa;
          S.mrg_c[q] = wc;
          S.inv_l[q] = L > 0.0f ? 1.0f / L : 0.0f;
        } else {
          S.inv_l[q] = lt > 0.0f ? 1.0f / lt : 0.0f;
        }
      }
      wg_sync();
      if (p.state_in != nullptr) {  // this range merged with the cached state: normalised output
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(frow0) * p.D + fx.h * kHd + r;
#pragma unroll
        for (int i0 = 0; i0 < QH; i0 += 8) {
          float oc[8];  // eight loads (L1 hits after the prefetch) before their stores
#pragma unroll
          for (int j = 0; j < 8; ++j)
            oc[j] = (q0 + i0 + j < fnrows) ? __ldg(stc + static_cast<size_t>(q0 + i0 + j) * p.H * kSt) : 0.0f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int q = q0 + i0 + j;
            if (ok && q < fnrows)
              out[static_cast<size_t>(q) * p.D] =
                  __float2bfloat16_rn((o[i0 + j] * S.mrg_a[q] + oc[j] * S.mrg_c[q]) * S.inv_l[q]);
          }
        }
      } else if (p.state != nullptr) {  // partial softmax state of the key range
        float* st = p.state + (static_cast<size_t>(frow0) * p.H + fx.h) * kSt;
#pragma unroll
        for (int i = 0; i < QH; ++i)
          if (ok && q0 + i < fnrows) st[static_cast<size_t>(q0 + i) * p.H * kSt + r] = o[i];
        if (ok && r < QH && q0 + r < fnrows) {
          const int q = q0 + r;
          st[static_cast<size_t>(q) * p.H * kSt + kHd] = has_pv ? S.fin_m[fuu & 1][q] : -INFINITY;
          st[static_cast<size_t>(q) * p.H * kSt + kHd + 1] = S.l_fin[q];
        }
      } else if (PIECES && can_merge && fx.part != 0) {
        // a piece of a tail unit: store its partial state in the piece's slot (O as
        // [column / 4][hd row][4]: a thread's four columns are one 16-byte vector, and a
        // warp's 32 rows are 512 contiguous bytes) and count it in
        // (one release per warpgroup, after the barrier that orders every thread's
        // stores before it); the piece that completes the unit merges all pieces'
        // states, in piece order whichever came last (so the rounding does not depend on
        // timing), per query M = max m, weights 2^(m - M), and writes the output.  The
        // count returns to zero for the next launch.
        const int np = p.tail_pieces;
        const size_t n_slots = static_cast<size_t>(p.tail_units) * np;
        const size_t slot = static_cast<size_t>(fx.piece) * p.tail_units + fx.tu;
        float4* wo = reinterpret_cast<float4*>(p.ws + slot * kQChunk * kHd) + (q0 / 4) * kHd + r;
        float* wml = p.ws + n_slots * kQChunk * kHd + slot * kQChunk * 2;
        if (ok) {
#pragma unroll
          for (int i = 0; i < QH; i += 4) wo[(i / 4) * kHd] = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
          if (r < QH) {
            *reinterpret_cast<float2*>(wml + (q0 + r) * 2) =
                make_float2(has_pv ? S.fin_m[fuu & 1][q0 + r] : -INFINITY, S.l_fin[q0 + r]);
          }
        }
        wg_sync();
        if (r == 0) {
          int last = 0;
          if (ok) {
            int* cnt = p.merge_cnt + 2 * fx.tu + g;
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            last = atomicAdd(cnt, 1) == np - 1;
            if (last) {
              *reinterpret_cast<volatile int*>(cnt) = 0;  // every piece has counted in
              asm volatile("fence.acq_rel.gpu;" ::: "memory");
            }
          }
          S.merge_last[g] = last;
        }
        wg_sync();
        if (S.merge_last[g]) {
          const float* wml0 = p.ws + n_slots * kQChunk * kHd + static_cast<size_t>(fx.tu) * kQChunk * 2;
          const size_t ml_stride = static_cast<size_t>(p.tail_units) * kQChunk * 2;
          if (r < QH) {
            // this column's (m, l) of every piece (loads in flight together), then the
            // maximum and each piece's weight
            const float* mlc = wml0 + (q0 + r) * 2;
            float2 ml[kMaxPieces];
#pragma unroll
            for (int j = 0; j < kMaxPieces; ++j)
              ml[j] = j < np ? __ldcg(reinterpret_cast<const float2*>(mlc + j * ml_stride)) : make_float2(-INFINITY, 0.0f);
            float M = -INFINITY;
#pragma unroll
            for (int j = 0; j < kMaxPieces; ++j) M = fmaxf(M, ml[j].x);
            float L = 0.0f;
#pragma unroll
            for (int j = 0; j < kMaxPieces; ++j) {
              const float w = (ml[j].x == -INFINITY) ? 0.0f : exp2f(ml[j].x - M);
              L = fmaf(w, ml[j].y, L);
              S.mrg_w[j][q0 + r] = w;
            }
            S.inv_l[q0 + r] = L > 0.0f ? 1.0f / L : 0.0f;
          }
          wg_sync();
          // per chunk of 4 columns of this thread's hd row: every piece's 16-byte vector,
          // all loads in flight together, folded in piece order
          const float4* wo0 = reinterpret_cast<const float4*>(p.ws + static_cast<size_t>(fx.tu) * kQChunk * kHd) +
                              (q0 / 4) * kHd + r;
          const size_t o_stride = static_cast<size_t>(p.tail_units) * kQChunk * kHd / 4;
#pragma unroll
          for (int c = 0; c < QH / 4; ++c) {
            float4 v[kMaxPieces];
#pragma unroll
            for (int j = 0; j < kMaxPieces; ++j)
              v[j] = j < np ? __ldcg(wo0 + j * o_stride + c * kHd) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
            for (int j = 0; j < kMaxPieces; ++j) {
              const float* wj = S.mrg_w[j] + q0 + 4 * c;
              a0 = fmaf(wj[0], v[j].x, a0);
              a1 = fmaf(wj[1], v[j].y, a1);
              a2 = fmaf(wj[2], v[j].z, a2);
              a3 = fmaf(wj[3], v[j].w, a3);
            }
            o[4 * c] = a0;
            o[4 * c + 1] = a1;
            o[4 * c + 2] = a2;
            o[4 * c + 3] = a3;
          }
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(frow0) * p.D + fx.h * kHd + r;
#pragma unroll
          for (int i = 0; i < QH; ++i) {
            const int q = q0 + i;
            if (ok && q < fnrows) out[static_cast<size_t>(q) * p.D] = __float2bfloat16_rn(o[i] * S.inv_l[q]);
          }
        }
      } else if (p.n_splits == 1) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(frow0) * p.D + fx.h * kHd + r;
        const float4* il4 = reinterpret_cast<const float4*>(S.inv_l + q0);
#pragma unroll
        for (int i = 0; i < QH; i += 4) {
          const float4 il = il4[i / 4];
          const int q = q0 + i;
          if (ok && q < fnrows) out[static_cast<size_t>(q) * p.D] = __float2bfloat16_rn(o[i] * il.x);
          if (ok && q + 1 < fnrows) out[static_cast<size_t>(q + 1) * p.D] = __float2bfloat16_rn(o[i + 1] * il.y);
          if (ok && q + 2 < fnrows) out[static_cast<size_t>(q + 2) * p.D] = __float2bfloat16_rn(o[i + 2] * il.z);
          if (ok && q + 3 < fnrows) out[static_cast<size_t>(q + 3) * p.D] = __float2bfloat16_rn(o[i + 3] * il.w);
        }
      } else {
        // split partials are stored by the unit's canonical number (sequence-major, the
        // combine's indexing), whatever order the units ran in
        const size_t cu = ((static_cast<size_t>(fx.b) * p.H + fx.h) * p.n_qchunks + fx.qc) * p.n_splits + fx.split;
        float* wo = p.ws + cu * kQChunk * kHd;
#pragma unroll
        for (int i = 0; i < QH; ++i) wo[(q0 + i) * kHd + r] = o[i];
        if (r < QH) {
          const int q = q0 + r;
          float* wml = p.ws + static_cast<size_t>(p.units) * kQChunk * kHd + (cu * kQChunk + q) * 2;
          wml[0] = has_pv ? S.fin_m[fuu & 1][q] : -INFINITY;
          wml[1] = S.l_fin[q];
        }
      }
    };

    // e4m3: the K group scale of this thread's key, fetched one tile ahead (it comes
    // from HBM); it multiplies the key's logits, the K operand holding the bare code
    auto fetch_ks = [&](const Unit& y, int t) -> float {
      const int jj = t * kKeyTile + r;
      return jj < p.slots ? __ldg(p.kv_scale + (static_cast<size_t>(y.b) * p.slots + jj) * 2 * p.H + y.h) : 0.0f;
    };
    auto first_tile = [&](int from, Unit& y) -> bool {
      for (int r2 = from; cta_item<PIECES>(p, r2, order, y); ++r2)
        if (y.t1 > y.t0) return true;
      return false;
    };
    float ks_next = 0.0f;
    if constexpr (FP8) {
      Unit y;
      if (first_tile(0, y)) ks_next = fetch_ks(y, y.t0);
    }

    float o_prev[QH], l_prev[QH];  // the unit waiting to be finished (deferred finish only)
    Unit px{};
    int puu = 0;
    uint32_t ppv = 0;
    bool pending = false;
    int uu = 0;  // units started by this CTA (parity selects the finish buffers)

    Unit x;
    for (int rnd = 0; cta_item<PIECES>(p, rnd, order, x); ++rnd, ++uu) {
      const int row0 = x.b * p.n_tok;  // first row of the sequence
      const int nrows = min(kQChunk, p.n_tok - x.qc * kQChunk);  // valid columns of this chunk
      const int kend = key_end(p, x.b);  // regular slots past this are not attended
      // e4m3: the S MMA multiplies the K codes by Q scaled by s (the converters' split of
      // the chunk into e4m3 parts); 1/s joins each key's logit factor
      float q8i = 1.0f;
      if constexpr (FP8) {
        wait(&S.q_conv[uu & 1], (uu >> 1) & 1u);
        q8i = S.q8inv[uu & 1];
      }
      // ---- per-unit set-up: running max and Flash-Verify tags (the tags over every
      // softmax warpgroup)
      if (r < QH) S.m_run[q0 + r] = -INFINITY;
      if (has_view) {
        for (int w = tid; w < mask_words; w += kSmWarps * 32) S.mask_bits[w] = 0u;
        if (tid == 0) S.n_draft = 0;
        both_sync();
        int my_draft = 0;
        for (int t = tid; t < p.n_tok; t += kSmWarps * 32) {
          const int v = p.view[row0 + t];
          if (v == DLLM_VIEW_MASK) {
            const int pos = p.positions[row0 + t];
            if (pos >= 0 && pos < p.max_pos) atomicOr(&S.mask_bits[pos >> 5], 1u << (pos & 31));
          } else if (v == DLLM_VIEW_DRAFT) {
            ++my_draft;
          }
        }
        if (my_draft) atomicAdd(&S.n_draft, my_draft);
        if (g == 0 && quarter < 2) {  // quarters 0 and 1 of warpgroup 0 tag columns 0..63
          const bool is_draft = r < nrows && p.view[row0 + x.qc * kQChunk + r] == DLLM_VIEW_DRAFT;
          const uint32_t bal = __ballot_sync(0xffffffffu, is_draft);
          if (lane == 0) S.draft_qmask[quarter] = bal;
        }
        both_sync();
      }
      const int n_draft = has_view ? min(S.n_draft, p.tail) : 0;
      const uint64_t dmask = has_view ? (static_cast<uint64_t>(S.draft_qmask[1]) << 32) | S.draft_qmask[0] : 0ull;
      float o_acc[QH];  // O^T row r (hd index r) for this warpgroup's queries, relative to the running max
      float l_part[QH];  // this thread's key's share of each of those queries' row sums
#pragma unroll
      for (int i = 0; i < QH; ++i) {
        o_acc[i] = 0.0f;
        l_part[i] = 0.0f;
      }

      for (int t = x.t0; t < x.t1; ++t) {
        const uint32_t sb = s_cnt & 1u, sph = (s_cnt >> 1) & 1u;
        const uint32_t tp = t & 1;  // parity slot for alpha
        float ks_cur = 1.0f;
        if constexpr (FP8) {
          ks_cur = ks_next;
          if (t + 1 < x.t1) {
            ks_next = fetch_ks(x, t + 1);
          } else {
            Unit y;
            if (first_tile(rnd + 1, y)) ks_next = fetch_ks(y, y.t0);
          }
        }
        // ---- A: scores of this thread's key for the warpgroup's queries
        wait(&S.s_full[sb], sph);
        tc_fence_after();
        float s[QH];
        tmem_ld_cols<QH>(tmem + lane_base + sb * NQ + q0, s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.s_free[sb]);
        ++s_cnt;

        const int j = t * kKeyTile + r;  // slot index within the sequence
        uint64_t vis;  // over all NQ columns
        if (!has_view) {
          vis = (j < p.max_pos) ? ~0ull : 0ull;
        } else if (j < p.max_pos) {
          vis = ((S.mask_bits[j >> 5] >> (j & 31)) & 1u) ? ~dmask : ~0ull;
        } else {
          vis = (j < p.max_pos + n_draft) ? dmask : 0ull;
        }
        if (p.ranged && (j < p.key_lo || j >= kend)) vis = 0ull;
        const uint64_t visg = vis >> q0;  // this warpgroup's columns from bit 0
        const float sc = p.scale_log2 * ks_cur * q8i;  // e4m3: times the key's K group scale and 1/s
        if (vis == ~0ull) {
#pragma unroll
          for (int i = 0; i < QH; ++i) s[i] *= sc;
        } else {
#pragma unroll
          for (int i = 0; i < QH; ++i) s[i] = ((visg >> i) & 1ull) ? s[i] * sc : -INFINITY;
        }

        // column maxima: one redux per query over the warp, then over the 4 warps
        {
          float mx[QH];
#pragma unroll
          for (int i = 0; i < QH; ++i) mx[i] = warp_max(s[i]);
          if (lane == 0) {
            float4* dst = reinterpret_cast<float4*>(S.red[quarter] + q0);
#pragma unroll
            for (int i = 0; i < QH; i += 4) dst[i / 4] = make_float4(mx[i], mx[i + 1], mx[i + 2], mx[i + 3]);
          }
        }
        wg_sync();
        // ---- B: column owners update the running max and the rescale factor
        if (r < QH) {
          const int q = q0 + r;
          const float mt = fmaxf(fmaxf(S.red[0][q], S.red[1][q]), fmaxf(S.red[2][q], S.red[3][q]));
          const float m_old = S.m_run[q];
          const float m_new = fmaxf(m_old, mt);
          const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
          const float a = fast_exp2(m_old - m_use);
          S.m_run[q] = m_new;
          S.m_use[q] = m_use;
          S.alpha[tp][q] = a;
          if (t == x.t1 - 1) {  // the unit's last tile: what its finish needs
            S.fin_alpha[uu & 1][q] = a;
            S.fin_m[uu & 1][q] = m_new;
          }
        }
        wg_sync();
        // ---- C: probabilities -> P^T (bf16, swizzled); this thread's partial row sums
        {
          // Slots past the regular region that no query sees may hold anything (stale
          // draft views, the next sequence, never-written memory).  Their P is 0, but
          // 0 * NaN would still poison O, so their V rows are zeroed before the PV MMA
          // (by warpgroup 0, before its P arrival, which the PV MMA waits for).
          if (!FP8 && g == 0 && (p.ranged || (t + 1) * kKeyTile > p.max_pos) && vis == 0ull &&
              (p.ranged || j >= p.max_pos)) {
            wait(&S.v_full[vs], vph);
            uint4* row0v = reinterpret_cast<uint4*>(S.v[vs] + r * 128);
            uint4* row1v = reinterpret_cast<uint4*>(S.v[vs] + kTileBytes / 2 + r * 128);
            // chunk order rotated per row (the 128-byte swizzle), so that neighbouring
            // rows write different banks
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              row0v[k ^ (r & 7)] = make_uint4(0u, 0u, 0u, 0u);
              row1v[k ^ (r & 7)] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          if (++vs == VST) { vs = 0; vph ^= 1u; }
          const uint32_t pb = pv_cnt & 1u, pph = (pv_cnt >> 1) & 1u;
          // the P V MMA that read this buffer two tiles ago must be done
          wait(&S.p_empty[pb], pph ^ 1u);
          const uint32_t pbase = smem_u32(S.p[pb]);
          const float4* mu4 = reinterpret_cast<const float4*>(S.m_use + q0);
          const float4* al4 = reinterpret_cast<const float4*>(S.alpha[tp] + q0);
#pragma unroll
          for (int i = 0; i < QH; i += 8) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int c = i + 4 * h;
              const float4 mu = mu4[c / 4];
              const float4 al = al4[c / 4];
              const float e0 = fast_exp2(s[c] - mu.x), e1 = fast_exp2(s[c + 1] - mu.y);
              const float e2 = fast_exp2(s[c + 2] - mu.z), e3 = fast_exp2(s[c + 3] - mu.w);
              l_part[c] = l_part[c] * al.x + e0;
              l_part[c + 1] = l_part[c + 1] * al.y + e1;
              l_part[c + 2] = l_part[c + 2] * al.z + e2;
              l_part[c + 3] = l_part[c + 3] * al.w + e3;
              w[2 * h] = pack_pair<FP8>(e0, e1);
              w[2 * h + 1] = pack_pair<FP8>(e2, e3);
            }
            st_shared_v4(pbase + p_chunk_offset<NQ>(r, q0 + i), w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.p_full[pb]);
        }
        // ---- D: fold the previous tile's P V into the accumulators (in a unit's first
        // tile: finish the previous unit instead, when that was deferred)
        if (kDefer && t == x.t0 && pending) {
          finish(false, o_prev, l_prev, px, puu, ppv);
          pending = false;
        }
        if (t > x.t0) {
          const uint32_t ob = (pv_cnt - 1) & 1u, oph = ((pv_cnt - 1) >> 1) & 1u;
          wait(&S.o_full[ob], oph);
          tc_fence_after();
          const float4* al4 = reinterpret_cast<const float4*>(S.alpha[tp ^ 1u] + q0);
          {
            float tmp[QH];
            tmem_ld_cols<QH>(tmem + lane_base + 2 * NQ + ob * NQ + q0, tmp);
#pragma unroll
            for (int i = 0; i < QH; i += 4) {
              const float4 al = al4[i / 4];
              o_acc[i] = o_acc[i] * al.x + tmp[i];
              o_acc[i + 1] = o_acc[i + 1] * al.y + tmp[i + 1];
              o_acc[i + 2] = o_acc[i + 2] * al.z + tmp[i + 2];
              o_acc[i + 3] = o_acc[i + 3] * al.w + tmp[i + 3];
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.o_free[ob]);
        }
        ++pv_cnt;
      }
      // ---- unit end: finish now, or hand the state to the next unit's first tile
      if constexpr (kDefer) {
        if (pending) {  // this unit had no tile to finish the previous one in
          finish(false, o_prev, l_prev, px, puu, ppv);
          pending = false;
        }
        if (PIECES && x.part != 0) {
          finish(true, o_acc, l_part, x, uu, pv_cnt - 1);
        } else {
#pragma unroll
          for (int i = 0; i < QH; ++i) {
            o_prev[i] = o_acc[i];
            l_prev[i] = l_part[i];
          }
          px = x;
          puu = uu;
          ppv = pv_cnt - 1;
          pending = true;
        }
      } else {
        finish(true, o_acc, l_part, x, uu, pv_cnt - 1);
      }
      // the next unit's set-up rewrites the running max (per warpgroup) and the shared tags
      if (has_view)
        both_sync();
      else
        wg_sync();
    }
    if constexpr (kDefer) {
      if (pending) finish(false, o_prev, l_prev, px, puu, ppv);
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(p.status, DLLM_DEV_TIMEOUT);
    }
  } else if (FP8 && warp >= 2 + kSmWarps) {
    // ------------------------------------------------------------------ e4m3 converters
    // Per unit: the Q chunk, split into two e4m3 parts for the 8-bit S MMA.  One scale
    // s for the chunk takes its largest |q| to 448; Q_hi = e4m3(s q) and Q_lo = e4m3(s q
    // - Q_hi), so Q_hi + Q_lo = s q to within about 2^-9 of each value (two 4-bit
    // significands, as close as bf16's rounding of Q), and 1/s goes to the softmax with
    // the key's K scale.  Per tile: thread r turns key row r of the staged V codes into
    // both 64-column halves of the f16 V operand, keeping the 128-byte swizzle: code
    // times the key's V scale, one f16 rounding.  V rows of slots that no query can see
    // are written as zeros (their probability is 0, and 0 * NaN must not reach O).  The
    // staged K codes feed the S MMA directly.
    const int r = (warp & 3) * 32 + lane;
    const int cw = (warp - 2 - kSmWarps);  // converter warp 0..3: column quarter of Q
    int ss = 0, vo = 0, uu = 0;
    uint32_t sph = 0, vph = 0;
    bool ok = true;
    // The V group scale of key r of a tile (fetched one tile ahead: it comes from HBM;
    // the K scale multiplies the key's logits in the softmax instead).
    auto fetch_vscale = [&](const Unit& y, int t) -> float {
      const int j = t * kKeyTile + r;
      return j < p.slots ? __ldg(p.kv_scale + ((static_cast<size_t>(y.b) * p.slots + j) * 2 + 1) * p.H + y.h) : 0.0f;
    };
    // the first tile of the first non-empty unit from round `from` on
    auto next_tile = [&](int from, Unit& y) -> bool {
      for (int r2 = from; cta_item<PIECES>(p, r2, order, y); ++r2)
        if (y.t1 > y.t0) return true;
      return false;
    };
    float nvs = 0.0f;
    {
      Unit y;
      if (next_tile(0, y)) nvs = fetch_vscale(y, y.t0);
    }
    // The four converter warps share a named barrier once per unit, so after a failed
    // wait a warp keeps walking the units (doing no work) instead of leaving the loop:
    // every warp passes that barrier the same number of times.
    Unit x;
    for (int rnd = 0; cta_item<PIECES>(p, rnd, order, x); ++rnd, ++uu) {
      {
        // Q chunk -> (Q_hi, Q_lo, 1/s).  Warp cw takes columns [32 cw, 32 cw + 32) of rows
        // lane and lane + 32: 64 bytes of bf16 from box cw / 2 of the Q tile, 32 bytes of
        // each e4m3 part.
        const int qb = uu & 1;
        if (ok && !mbar_wait_warp(&S.q_full[qb], (uu >> 1) & 1u, abort_flag)) ok = false;
        constexpr int kRows = NQ > 32 ? 2 : 1;
        float qv[kRows][32];
        float amax = 0.0f;
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const int row = lane + 32 * rr;
          const uint8_t* src = S.q[qb] + (cw >> 1) * kQBox + row * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (ok && row < NQ) w = *reinterpret_cast<const uint4*>(src + ((((cw & 1) * 4 + c) ^ (row & 7)) << 4));
            const uint32_t* wi = reinterpret_cast<const uint32_t*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              qv[rr][c * 8 + 2 * e] = __uint_as_float(wi[e] << 16);
              qv[rr][c * 8 + 2 * e + 1] = __uint_as_float(wi[e] & 0xffff0000u);
            }
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(qv[rr][i]));
        }
        amax = warp_max(amax);
        if (lane == 0) S.cv_red[qb][cw] = amax;
        asm volatile("bar.sync 4, 128;" ::: "memory");  // the four converter warps
        amax = fmaxf(fmaxf(S.cv_red[qb][0], S.cv_red[qb][1]), fmaxf(S.cv_red[qb][2], S.cv_red[qb][3]));
        const float sq = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 1.0f;
        if (cw == 0 && lane == 0) S.q8inv[qb] = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const int row = lane + 32 * rr;
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t hw = 0u, lw = 0u;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const float y0 = qv[rr][4 * i + 2 * j] * sq, y1 = qv[rr][4 * i + 2 * j + 1] * sq;
              const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
              const float2 hv = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3)));
              const __nv_fp8x2_storage_t l =
                  __nv_cvt_float2_to_fp8x2(make_float2(y0 - hv.x, y1 - hv.y), __NV_SATFINITE, __NV_E4M3);
              hw |= static_cast<uint32_t>(h) << (16 * j);
              lw |= static_cast<uint32_t>(l) << (16 * j);
            }
            hi[i] = hw;
            lo[i] = lw;
          }
          if (ok && row < NQ) {
            uint8_t* dh = S.q8[qb][0] + row * 128;
            uint8_t* dl = S.q8[qb][1] + row * 128;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint32_t off = (((2 * cw + c) ^ (row & 7)) << 4);
              *reinterpret_cast<uint4*>(dh + off) = make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
              *reinterpret_cast<uint4*>(dl + off) = make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.q_conv[qb]);
      }
      if (!ok) continue;
      int n_draft = 0;
      if (p.view) {
        for (int t = 0; t < p.n_tok; ++t) n_draft += (p.view[x.b * p.n_tok + t] == DLLM_VIEW_DRAFT);
        n_draft = min(n_draft, p.tail);
      }
      const int tail_end = p.max_pos + n_draft;
      const int kend = key_end(p, x.b);
      for (int t = x.t0; t < x.t1; ++t) {
        const int j = t * kKeyTile + r;
        const uint32_t sw = static_cast<uint32_t>(r & 7);
        // this key's V scale (prefetched), and the next tile's
        const float vsc = nvs;
        if (t + 1 < x.t1) {
          nvs = fetch_vscale(x, t + 1);
        } else {
          Unit y;
          if (next_tile(rnd + 1, y)) nvs = fetch_vscale(y, y.t0);
        }
        // V
        if (!mbar_wait_warp(&S.sv_full[ss], sph, abort_flag)) { ok = false; break; }
        if (!mbar_wait_warp(&S.v_empty[vo], vph ^ 1u, abort_flag)) { ok = false; break; }
        {
          const __half2 sc2 = __float2half2_rn(vsc);
          const uint8_t* src = S.sv[ss] + r * 128;
          uint8_t* dst = S.v[vo] + r * 128;
          const bool zero = j < p.max_pos ? (p.ranged && (j < p.key_lo || j >= kend)) : j >= tail_end;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
            if (!zero) dequant16_f16(*reinterpret_cast<const uint4*>(src + ((c ^ sw) << 4)), sc2, lo, hi);
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
  grid_dep_launch();
  grid_dep_wait();
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

// Merge two partial states of the same rows (FACache-style: a cached state of keys that
// did not change and a fresh state of keys that did).  m in base-2 units:
//   M = max(m_a, m_b), O = 2^(m_a - M) O_a + 2^(m_b - M) O_b, l likewise.
// One warp per (row, head).  A state is 130 floats (8-byte aligned), so each lane moves
// float2 pairs: elements 2*lane, 2*lane+1 and 64+2*lane, 64+2*lane+1 of O; (m, l) is the
// 65th pair.
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(kMergeWarps * 32) state_merge(const float* __restrict__ a,
                                                                const float* __restrict__ b, long long n_rh,
                                                                __nv_bfloat16* out, float* state_out) {
  constexpr int kSt = kHd + 2;
  const long long rh = static_cast<long long>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (rh >= n_rh) return;
  const float2* pa = reinterpret_cast<const float2*>(a + rh * kSt);
  const float2* pb = reinterpret_cast<const float2*>(b + rh * kSt);
  const float2 mla = __ldg(pa + kHd / 2), mlb = __ldg(pb + kHd / 2);
  const float2 a0 = __ldg(pa + lane), a1 = __ldg(pa + 32 + lane);
  const float2 b0 = __ldg(pb + lane), b1 = __ldg(pb + 32 + lane);
  const float M = fmaxf(mla.x, mlb.x);
  float wa = 0.0f, wb = 0.0f;
  if (M != -INFINITY) {
    wa = mla.x == -INFINITY ? 0.0f : exp2f(mla.x - M);
    wb = mlb.x == -INFINITY ? 0.0f : exp2f(mlb.x - M);
  }
  const float2 o0 = make_float2(a0.x * wa + b0.x * wb, a0.y * wa + b0.y * wb);
  const float2 o1 = make_float2(a1.x * wa + b1.x * wb, a1.y * wa + b1.y * wb);
  const float L = mla.y * wa + mlb.y * wb;
  if (out) {
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    __nv_bfloat162* po = reinterpret_cast<__nv_bfloat162*>(out + rh * kHd);
    po[lane] = __floats2bfloat162_rn(o0.x * inv, o0.y * inv);
    po[32 + lane] = __floats2bfloat162_rn(o1.x * inv, o1.y * inv);
  }
  if (state_out) {
    float2* so = reinterpret_cast<float2*>(state_out + rh * kSt);
    so[lane] = o0;
    so[32 + lane] = o1;
    if (lane == 0) so[kHd / 2] = make_float2(M, L);
  }
}

}  // namespace

int launch_state_merge(const float* a, const float* b, int rows, int H, void* out, float* state_out, cudaStream_t s) {
  const long long n_rh = static_cast<long long>(rows) * H;
  if (n_rh == 0) return 0;
  const long long blocks = (n_rh + kMergeWarps - 1) / kMergeWarps;
  state_merge<<<static_cast<unsigned>(blocks), kMergeWarps * 32, 0, s>>>(
      a, b, n_rh, reinterpret_cast<__nv_bfloat16*>(out), state_out);
  return (int)cudaGetLastError();
}

template <int NQ, bool FP8, bool PIECES = false>
int launch_one(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const CUtensorMap& tm_kv_tail,
               int grid, cudaStream_t s) {
  if constexpr (!FP8 && !PIECES) {
    if (p.tail_pieces > 0) return launch_one<NQ, false, true>(p, tm_q, tm_kv, tm_kv_tail, grid, s);
  }
  const size_t smem = sizeof(Smem<NQ, FP8>) + 1024;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(attn_cache_tc<NQ, FP8, PIECES>), (int)smem);
  if (e != cudaSuccess) return (int)e;
  return (int)launch_pdl(attn_cache_tc<NQ, FP8, PIECES>, dim3(grid), dim3(Cfg<NQ, FP8>::kThreads), smem, s, tm_q,
                         tm_kv, tm_kv_tail, p);
}

int launch_attn_tc(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                   const CUtensorMap& tm_kv_tail, int grid, cudaStream_t s) {
  const bool fp8 = p.kv_dtype == DLLM_E4M3;
  if (p.nq_pad <= 32)
    return fp8 ? launch_one<32, true>(p, tm_q, tm_kv, tm_kv_tail, grid, s)
               : launch_one<32, false>(p, tm_q, tm_kv, tm_kv_tail, grid, s);
  if (p.nq_pad <= 48)
    return fp8 ? launch_one<48, true>(p, tm_q, tm_kv, tm_kv_tail, grid, s)
               : launch_one<48, false>(p, tm_q, tm_kv, tm_kv_tail, grid, s);
  return fp8 ? launch_one<64, true>(p, tm_q, tm_kv, tm_kv_tail, grid, s)
             : launch_one<64, false>(p, tm_q, tm_kv, tm_kv_tail, grid, s);
}

int launch_attn_combine(const AttnParams& p, cudaStream_t s) {
  dim3 grid(p.B * p.n_tok, p.H);
  return (int)launch_pdl(attn_combine, grid, dim3(kHd), 0, s, p);
}

}  // namespace dllm
