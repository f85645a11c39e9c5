// spec_verify, rows with top-p and no top-k: the threshold search as
// grid-wide passes (sm_103a).
//
// Such a row keeps the shortest prefix of the total order whose mass reaches
// P, the crossing entry included (inclusionAI/AReno PR #550, "What does this
// PR do?" Phase 2: the sampler-equivalent target distribution).  Where that
// prefix ends depends on the mass of the whole row above every candidate
// threshold, so these units run after the stream and settle roles, in passes
// over tiles of 2048 to 8192 logits.  Every warp of the grid takes a
// contiguous share of all tiles of all top-p units (one tile where the units
// allow it), streaming a tile's rows through its shared memory with
// cp.async, two chunks in flight, and a grid barrier separates the passes:
//   1. max: each tile's maximum (or that it holds a NaN or +inf) goes into
//      the tile's record; the tile's draft probabilities are prefetched into
//      L2 for pass 5.  Later passes take the unit's max from its tiles';
//   2. mass: every entry's fixed-point weight e * 2^40, e = exp2((l - m) c),
//      goes into one of 256 bins of 1/8 in log2 of the weight, summed in the
//      warp's shared memory and then added to the unit's histogram in global
//      memory (fixed point makes every sum exact and independent of order);
//   3. refinement: each warp reads the unit's histograms, finds the bin where
//      the mass from the top reaches ceil(P Z) and the bin's range of order
//      keys, and histograms the mass of the entries in that range by key, 8
//      key bits a level, until one key, the crossing key, is left (one level
//      for most bf16 rows; at most two for bf16 and four for fp32).  The
//      level whose bins are single keys also lists each tile's keys with
//      their counts (bf16);
//   4. ties (fp32 rows, or a tile whose list overflowed): the entries at the
//      crossing key in each tile.  The first n of them by index are kept,
//      where n comes from the mass still missing;
//   5. tiles: with the kept set known, alpha = sum min(p, q) and the level-1
//      races over the tile's 256-entry blocks, of the residual max(p - q, 0)
//      and of p;
//   6. settle: one warp per unit merges the tiles' alphas and races, runs the
//      accept test and the level-2 race in the winning block, and writes the
//      unit's record (the row's last unit finalizes the row).
// After each barrier every warp derives its unit's threshold state from the
// state the previous pass stored and the newest histogram (one round trip and
// a warp scan), so no pass waits for a settle step.  Each barrier wait is
// bounded (a second): one that gives up sets ERR_BARRIER, and the units come
// back with SPEC_F_TIMEOUT.
#pragma once

#include "spec_common.cuh"
#include "spec_general.cuh"

namespace specv {

constexpr unsigned kAll = 0xffffffffu;
// A tile is 8 to 32 blocks of 256 entries (chosen per call so that the
// tiles of all top-p units spread evenly over the grid's warps); with at
// least 2048 entries a tile, a unit's tiles fit its A-record slots.
constexpr int kTpMinBlocks = 8;
constexpr int kTpMaxBlocks = 32;
static_assert(kTpMinBlocks * kRaceBlock == Geo<false>::EA, "a top-p tile takes one A-record slot of its unit");

// The top-p rows of the call: their place in the row order and the levels run.
struct TpPlan {
  const uint32_t* order;
  const RowPack* cfg;     // per-row configs in shared memory (null: classify from the parameters)
  int base;               // index of the first top-p row in the order
  int nU;                 // top-p units
  int nlev;               // refinement levels run
  int NR, ET, NT;         // tiles: 256-entry blocks a tile (8..32), entries a tile, tiles a unit
  bool ties;              // pass 4 ran (tie counts in the tile records)
};

struct TpUnit {
  int row, pos, uid;
  bool has_q;
  RowCfg cfg;
  size_t lrow, qrow;
};
__device__ __noinline__ TpUnit tp_unit(const Args& A, const TpPlan& T, int j) {
  TpUnit U;
  const int k1 = A.k + 1;
  U.row = (int)T.order[T.base + j / k1];
  U.pos = j % k1;
  U.uid = U.row * k1 + U.pos;
  U.has_q = U.pos < A.k;
  U.cfg = T.cfg ? unpack_cfg(T.cfg[U.row]) : classify(A.params[U.row], A.V);
  U.lrow = (size_t)U.uid * A.V;
  U.qrow = ((size_t)U.row * A.k + U.pos) * (size_t)A.V;
  return U;
}

__device__ __forceinline__ u64* tp_hist(const Args& A, int j, int lvl) {
  return A.tp + (size_t)j * kTpStride + kTpUnitWords + lvl * kTpBins;
}
// A unit's summary, tagged words at the start of its scratch: [0] the
// crossing key, [1] n_need, [2] Z_S, [3] its SPEC_F_MARGIN_TOPP flag
// (written in pass 4), [4] the index of the last kept entry at the crossing
// key (pass 5), [5] the unit's max key (pass 2).  Then, plain words, the
// threshold state after each level (5 words a level).
constexpr int kTpStateWords = 5;
constexpr int kTpStateBase = 8;
static_assert(kTpStateBase + kTpLevels * kTpStateWords <= kTpUnitWords, "unit words");
__device__ __forceinline__ u64* tp_summary(const Args& A, int j) { return A.tp + (size_t)j * kTpStride; }
__device__ __forceinline__ u64* tp_state_at(const Args& A, int j, int L) {
  return A.tp + (size_t)j * kTpStride + kTpStateBase + L * kTpStateWords;
}
// A tile's record: tagged words in the unit's A-record slot of that tile
// (top-p units have no stream tiles).  [0] ties at the crossing key,
// [1] alpha, [2..6] residual race (s1, t1, s2, t2, v1), [7..11] race of p,
// [12] the tile max's order key (0: no finite entry, kTpBadKey: a NaN or
// +inf), [13..15] the first three entries of the tile's key list.
//   The key list (bf16 rows): the keys of the unit's last refinement level
// present in the tile with their counts (key | count << 16; 0: none), up to
// kTpListLen of them, or kTpTieOverflow in entry 0 when the tile holds more.
// Entries 3.. sit in the unit's B-record slot of the same index (top-p units
// have no B tiles; a unit has at least as many B slots as top-p tiles).
constexpr uint32_t kTpBadKey = 0xffffffffu;
constexpr uint32_t kTpTieOverflow = 0xffffffffu;
constexpr int kTpTieWord = 13;
constexpr int kTpListLen = 3 + kBRecWords;
__device__ __forceinline__ u64* tp_list(const Args& A, int uid, int t, int i) {
  return i < 3 ? A.rec + ((size_t)uid * A.NTA + t) * kRecWords + kTpTieWord + i
               : A.brec + ((size_t)uid * A.NTB + t) * kBRecWords + (i - 3);
}
constexpr uint32_t kTpNeedTies = 1u << 8;   // tp_more: a tile's key list overflowed, run the ties pass
constexpr uint32_t kTpMissKey = 0xfffffffeu;   // summary only: a tile's max did not arrive (no finite key is this large)
constexpr int kTpMaxWord = 12;
__device__ __forceinline__ u64* tp_rec(const Args& A, int uid, int t) {
  return A.rec + ((size_t)uid * A.NTA + t) * kRecWords;
}

// Group of 8 logits starting at entry e0 of a row, as raw words (entries
// past V read as -inf).
template <bool kBF16>
__device__ __forceinline__ void tp_group(const Args& A, size_t lrow, int e0, uint32_t (&w)[kBF16 ? 4 : 8]) {
  if constexpr (kBF16) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(A.logits) + lrow;
    if (A.vec_logits && e0 + 8 <= A.V) {
      const uint4 x = __ldcg(reinterpret_cast<const uint4*>(p + e0));
      w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = e0 + 2 * i < A.V ? (uint32_t)p[e0 + 2 * i] : 0xff80u;
        const uint32_t hi = e0 + 2 * i + 1 < A.V ? (uint32_t)p[e0 + 2 * i + 1] : 0xff80u;
        w[i] = lo | (hi << 16);
      }
    }
  } else {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(A.logits) + lrow;
    if (A.vec_logits && e0 + 8 <= A.V) {
      const uint4 a = __ldcg(reinterpret_cast<const uint4*>(p + e0));
      const uint4 b = __ldcg(reinterpret_cast<const uint4*>(p + e0 + 4));
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = e0 + i < A.V ? p[e0 + i] : 0xff800000u;
    }
  }
}
template <bool kBF16>
__device__ __forceinline__ float tp_v(const uint32_t* w, int j) {
  if constexpr (kBF16) return __uint_as_float((j & 1) ? (w[j >> 1] & 0xffff0000u) : (w[j >> 1] << 16));
  else return __uint_as_float(w[j]);
}
// The mass bin of x = (l - m) c <= 0: 1/8 in log2 of the weight a bin, the
// tail (weights below 2^-31.875) in bin 255.  floor(t) for t in [0, 255] by
// rounding on the float adder (t + 2^23 is t rounded to an integer, exactly)
// and stepping down when that rounded up: no conversion instruction.
__device__ __forceinline__ int tp_bin(float x) {
  const float t = fminf(-x * 8.0f, 255.0f);
  const float r = t + 8388608.0f;
  const int k = (int)(__float_as_uint(r) - 0x4b000000u);
  return k - ((r - 8388608.0f > t) ? 1 : 0);
}
template <bool kBF16>
__device__ __forceinline__ float tp_key_val(uint32_t key) { return from_okey(full_key<kBF16>(key)); }

__device__ __forceinline__ u64 shfl_u64(u64 v, int src) {
  const uint32_t lo = __shfl_sync(kAll, (uint32_t)v, src), hi = __shfl_sync(kAll, (uint32_t)(v >> 32), src);
  return ((u64)hi << 32) | lo;
}
__device__ __forceinline__ u64 warp_incl_scan_u64(u64 v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t lo = __shfl_up_sync(kAll, (uint32_t)v, o), hi = __shfl_up_sync(kAll, (uint32_t)(v >> 32), o);
    if (lane >= o) v += ((u64)hi << 32) | lo;
  }
  return v;
}
__device__ __forceinline__ uint32_t warp_excl_scan_u32(uint32_t v, uint32_t* total) {
  const int lane = threadIdx.x & 31;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kAll, inc, o);
    if (lane >= o) inc += y;
  }
  *total = __shfl_sync(kAll, inc, 31);
  return inc - v;
}

// In a 256-bin histogram held 8 bins a lane (lane l: bins 8l .. 8l + 7), the
// first bin at which the sum from bin 0 reaches `need`, and the sum of the
// bins before it (bin 255 if the histogram holds less).
__device__ __noinline__ void tp_select(const u64 (&h)[8], u64 need, int* bin, u64* before) {
  const int lane = threadIdx.x & 31;
  u64 tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += h[i];
  const u64 inc = warp_incl_scan_u64(tot);
  const unsigned b = __ballot_sync(kAll, inc >= need);
  const int f = b ? __ffs(b) - 1 : 31;
  int bi = -1;
  u64 cum = inc - tot, bef = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (bi < 0 && cum + h[i] >= need) {
      bi = i;
      bef = cum;
    }
    cum += h[i];
  }
  if (bi < 0) {
    bi = 7;
    bef = cum - h[7];
  }
  *bin = __shfl_sync(kAll, lane * 8 + bi, f);
  *before = shfl_u64(bef, f);
}

// The smallest key in [lo, hi] at which pred holds (pred is false, then
// true, along the keys), or hi + 1 when it holds nowhere; 32 keys probed a
// round, one per lane.
template <typename Pred>
__device__ __forceinline__ uint32_t tp_first_true(uint32_t lo, uint32_t hi, Pred pred) {
  const int lane = threadIdx.x & 31;
  u64 L = lo, H = (u64)hi + 1u;   // the answer lies in [L, H]
  while (L < H) {
    const u64 step = (H - L + 31u) / 32u;
    const u64 key = L + step * (u64)lane;
    const bool p = key >= H || pred((uint32_t)key);
    const unsigned b = __ballot_sync(kAll, p);
    if (b == 0u) {
      L += 31u * step + 1u;
      continue;
    }
    const int f = __ffs(b) - 1;
    if (f == 0) break;
    const u64 nL = L + (u64)(f - 1) * step + 1u;
    H = min(L + (u64)f * step, H);
    L = nL;
  }
  return (uint32_t)L;
}

// Threshold state of a unit: the mass bin b0 where the sum from the top
// reaches target = ceil(P zk), the key range [lo, hi] still holding the
// crossing key, the shift of the next level's bins ((hi - key) >> s), the
// mass above the range and the mass still missing within it (rem).
// lo == hi: the crossing key is found.
struct TpState {
  u64 zk, above, rem;
  uint32_t lo, hi;
  int s, b0;
  int s_prev;   // the shift of the level this state came out of (0: its bins were single keys)
};
__device__ __forceinline__ int tp_shift(uint32_t lo, uint32_t hi) {
  const int nb = 32 - __clz((int)(hi - lo));
  return nb > 8 ? nb - 8 : 0;
}
// The state before any refinement, from the mass histogram.
template <bool kBF16>
__device__ __noinline__ TpState tp_state0(const Args& A, int j, float m, float c, float P) {
  const int lane = threadIdx.x & 31;
  TpState st;
  u64 h[8];
  const u64* H0 = tp_hist(A, j, 0) + lane * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = __ldcg(H0 + i);
  u64 tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += h[i];
  st.zk = warp_sum_u64(tot);
  const u64 target = (u64)ceil((double)P * (double)st.zk);
  u64 bef;
  tp_select(h, target, &st.b0, &bef);
  st.above = bef;
  st.rem = target - bef;
  // the keys of bin b0: the bin falls as the key rises
  const int b0 = st.b0;
  const uint32_t kmin = kf<kBF16>(-INFINITY), kmax = kf<kBF16>(m);
  st.lo = tp_first_true(kmin, kmax, [&](uint32_t key) { return tp_bin((tp_key_val<kBF16>(key) - m) * c) <= b0; });
  st.hi = b0 == 0 ? kmax
                  : tp_first_true(kmin, kmax,
                                  [&](uint32_t key) { return tp_bin((tp_key_val<kBF16>(key) - m) * c) <= b0 - 1; }) -
                        1u;
  st.s = tp_shift(st.lo, st.hi);
  st.s_prev = 0;
  return st;
}
// The state after one more level: the level's histogram h (8 bins a lane).
__device__ __noinline__ TpState tp_state_step(TpState st, const u64 (&h)[8]) {
  st.s_prev = st.s;
  if (st.lo >= st.hi) {
    st.s_prev = 0;   // found before this level: nothing more to list
    return st;
  }
  int sb;
  u64 ab;
  tp_select(h, st.rem, &sb, &ab);
  st.rem -= ab;
  st.above += ab;
  const uint32_t nhi = st.hi - ((uint32_t)sb << st.s);
  const uint32_t wdt = (1u << st.s) - 1u;
  st.lo = (nhi - st.lo >= wdt) ? nhi - wdt : st.lo;
  st.hi = nhi;
  st.s = tp_shift(st.lo, st.hi);
  return st;
}
// The state a level pass starts from is kept in the unit's words (by the
// warp holding the unit's first tile), so that later passes read it back
// instead of walking every level again.
__device__ __forceinline__ void tp_state_store(const Args& A, int j, int L, const TpState& st) {
  const int lane = threadIdx.x & 31;
  const u64 v = lane == 0 ? ((u64)st.hi << 32 | st.lo)
              : lane == 1 ? ((u64)(uint32_t)st.b0 << 32 | (uint32_t)st.s)
              : lane == 2 ? st.above
              : lane == 3 ? st.rem
                          : st.zk;
  if (lane < kTpStateWords) __stcg(tp_state_at(A, j, L) + lane, v);
}
// The state after level L (L >= 0): the stored state of level L and that
// level's histogram, read in one round trip.
__device__ __noinline__ TpState tp_state_after(const Args& A, int j, int L) {
  const int lane = threadIdx.x & 31;
  const u64 sw = lane < kTpStateWords ? __ldcg(tp_state_at(A, j, L) + lane) : 0ull;
  u64 h[8];
  const u64* HL = tp_hist(A, j, 1 + L) + lane * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = __ldcg(HL + i);
  TpState st;
  const u64 w0 = shfl_u64(sw, 0), w1 = shfl_u64(sw, 1);
  st.lo = (uint32_t)w0;
  st.hi = (uint32_t)(w0 >> 32);
  st.s = (int)(uint32_t)w1;
  st.b0 = (int)(uint32_t)(w1 >> 32);
  st.above = shfl_u64(sw, 2);
  st.rem = shfl_u64(sw, 3);
  st.zk = shfl_u64(sw, 4);
  return tp_state_step(st, h);
}

// The unit's max and validity from its tiles' records (a NaN or +inf, or no
// finite entry: invalid; a record of another call: a pass gave up).
struct TpMax {
  float m;
  uint32_t key;   // the max's order key, kTpBadKey, 0 (no finite entry) or kTpMissKey
  bool live;      // valid, and every tile's max arrived
  bool invalid;   // a NaN or +inf, or no finite entry
  bool missing;   // a tile's record is not this call's
};
__device__ __forceinline__ TpMax tp_max_decode(uint32_t mk) {
  TpMax r;
  r.key = mk;
  r.missing = mk == kTpMissKey;
  r.invalid = !r.missing && (mk == kTpBadKey || mk == 0u);
  r.live = !r.missing && !r.invalid;
  r.m = r.live ? from_okey(mk) : 0.f;
  return r;
}
__device__ __noinline__ TpMax tp_max_of(const Args& A, const TpPlan& T, int uid, uint32_t tag) {
  uint32_t mk = 0u;
  bool ok = true;
  for (int t = (int)(threadIdx.x & 31); t < T.NT; t += 32) {
    const u64 w = __ldcg(tp_rec(A, uid, t) + kTpMaxWord);
    ok = ok && tag_ok(w, tag);
    mk = max(mk, wu(w));
  }
  mk = __reduce_max_sync(kAll, mk);
  return tp_max_decode(__all_sync(kAll, ok) ? mk : kTpMissKey);
}
// The same from the unit's summary word (after pass 2).
__device__ __forceinline__ TpMax tp_max_from(u64 w, uint32_t tag) {
  return tp_max_decode(tag_ok(w, tag) ? wu(w) : kTpMissKey);
}

// The warp's share of the call's top-p tiles: a contiguous range, so that
// consecutive tiles of a warp mostly belong to one unit.
__device__ __forceinline__ void tp_share(const TpPlan& T, uint32_t gw, uint32_t nwg, u64* t0, u64* t1) {
  const u64 tiles = (u64)T.nU * (u64)T.NT;
  *t0 = tiles * gw / nwg;
  *t1 = tiles * (gw + 1u) / nwg;
}

// Rows of a tile pass through the warp's shared memory in chunks of CH
// rows, two chunk buffers (b0, b1) in turn: the copies of chunk c + 1 are in
// flight while chunk c is reduced.  Row r of a tile is the 32 groups of 8
// entries from e_base + 256 r; the lane's group of a chunk row sits at
// cb + (32 r + lane) * G (G = 16 bytes bf16, 32 fp32) and, with q, its draft
// probabilities at cb + CH * 32 * G + (32 r + lane) * 32.  Copies are
// cp.async (16 bytes each) where the rows are 16-byte aligned, else plain
// loads and stores; entries past V read as -inf (q as 0).  A lane reads back
// only its own groups.  fn(r, logits group, q group) runs for every row in
// order, done() after every chunk.
template <bool kBF16>
__device__ __forceinline__ void tp_issue(const Args& A, size_t lrow, size_t qrow, bool with_q, int e_base, int r0,
                                         int n, unsigned char* cb, int CH) {
  constexpr int G = kBF16 ? 16 : 32;
  constexpr int es = kBF16 ? 2 : 4;
  const int lane = threadIdx.x & 31;
  const unsigned char* row = reinterpret_cast<const unsigned char*>(A.logits) + lrow * es;
#pragma unroll 1
  for (int r = 0; r < n; ++r) {
    const int e0 = e_base + ((r0 + r) * 32 + lane) * 8;
    unsigned char* d = cb + (r * 32 + lane) * G;
    if (A.vec_logits && e0 + 8 <= A.V) {
      cp_async16(d, row + (size_t)e0 * es);
      if constexpr (!kBF16) cp_async16(d + 16, row + (size_t)e0 * es + 16);
    } else {
      uint32_t w[kBF16 ? 4 : 8];
      tp_group<kBF16>(A, lrow, e0, w);
      uint4* d4 = reinterpret_cast<uint4*>(d);
      d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
      if constexpr (!kBF16) d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    if (with_q) {
      unsigned char* dq = cb + CH * 32 * G + (r * 32 + lane) * 32;
      if (A.vec_q && e0 + 8 <= A.V) {
        cp_async16(dq, A.q + qrow + e0);
        cp_async16(dq + 16, A.q + qrow + e0 + 4);
      } else {
        float qv[8];
        load_q8(A, qrow, e0, qv);
        float4* d4 = reinterpret_cast<float4*>(dq);
        d4[0] = make_float4(qv[0], qv[1], qv[2], qv[3]);
        d4[1] = make_float4(qv[4], qv[5], qv[6], qv[7]);
      }
    }
  }
}
template <bool kBF16, typename F, typename D>
__device__ __forceinline__ void tp_rows(const Args& A, size_t lrow, size_t qrow, bool with_q, int e_base, int nrows,
                                        unsigned char* b0, unsigned char* b1, int CH, F fn, D done) {
  constexpr int G = kBF16 ? 16 : 32;
  const int lane = threadIdx.x & 31;
  const int nch = (nrows + CH - 1) / CH;
  tp_issue<kBF16>(A, lrow, qrow, with_q, e_base, 0, min(CH, nrows), b0, CH);
  cp_async_commit();
#pragma unroll 1
  for (int c = 0; c < nch; ++c) {
    unsigned char* cur = (c & 1) ? b1 : b0;
    if (c + 1 < nch) {
      const int r0 = (c + 1) * CH;
      tp_issue<kBF16>(A, lrow, qrow, with_q, e_base, r0, min(CH, nrows - r0), (c & 1) ? b0 : b1, CH);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    const int n = min(CH, nrows - c * CH);
#pragma unroll 1
    for (int r = 0; r < n; ++r)
      fn(c * CH + r, cur + (r * 32 + lane) * G, cur + CH * 32 * G + (r * 32 + lane) * 32);
    done();
    __syncwarp();
  }
}
template <bool kBF16>
__device__ __forceinline__ void tp_load_group(const unsigned char* g, uint32_t (&w)[kBF16 ? 4 : 8]) {
  const uint4* s = reinterpret_cast<const uint4*>(g);
  const uint4 a = s[0];
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  if constexpr (!kBF16) {
    const uint4 b = s[1];
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
}
// Chunk rows of the logits-only passes: 4 KB a chunk (2048 bf16 / 1024 fp32
// entries), so that a shared histogram flushed once a chunk cannot overflow.
template <bool kBF16>
__device__ __forceinline__ constexpr int tp_chunk() { return kBF16 ? 8 : 4; }

// Pass 1: tile maxima.
template <bool kBF16>
__device__ __noinline__ void tp_max_pass(const Args& A, const TpPlan& T, uint32_t tag, uint32_t gw, uint32_t nwg,
                                         unsigned char* b0, unsigned char* b1) {
  const int lane = threadIdx.x & 31;
  u64 t0, t1;
  tp_share(T, gw, nwg, &t0, &t1);
  int cj = -1;
  TpUnit U;
  for (u64 tt = t0; tt < t1; ++tt) {
    const int j = (int)(tt / (u64)T.NT), t = (int)(tt % (u64)T.NT);
    if (j != cj) {
      cj = j;
      U = tp_unit(A, T, j);
    }
    const int e_base = t * T.ET;
    if (lane == 0 && U.has_q && A.vec_q) {
      // the tile's draft probabilities, read by pass 5
      const uint32_t bytes = (uint32_t)(min(T.ET, A.V - e_base) * 4) & ~15u;
      if (bytes) bulk_prefetch_l2(A.q + U.qrow + e_base, bytes);
    }
    float mx = -INFINITY;
    tp_rows<kBF16>(A, U.lrow, 0, false, e_base, T.NR, b0, b1, tp_chunk<kBF16>(),
                   [&](int, const unsigned char* g, const unsigned char*) {
                     uint32_t w[kBF16 ? 4 : 8];
                     tp_load_group<kBF16>(g, w);
                     if constexpr (kBF16) {
                       const uint32_t a = max_nan_bf16x2(max_nan_bf16x2(w[0], w[1]), max_nan_bf16x2(w[2], w[3]));
                       mx = max_nan(mx, max_nan(bf16_lo(a), bf16_hi(a)));
                     } else {
#pragma unroll
                       for (int i = 0; i < 8; ++i) mx = max_nan(mx, __uint_as_float(w[i]));
                     }
                   },
                   [] {});
    mx = warp_max_nan(mx);
    if (lane == 0) {
      const uint32_t key = (mx != mx || mx == INFINITY) ? kTpBadKey : (mx > -INFINITY ? okey(mx) : 0u);
      __stcg(tp_rec(A, U.uid, t) + kTpMaxWord, tagw(tag, key));
    }
  }
}

// floor(e * 2^40) for e = 0 or a normal e in (0, 1], as hi = bits 20 and up
// and lo = bits 0..19, from the float's fields in integer arithmetic:
// e = m24 * 2^(E - 23), so floor(e * 2^40) = m24 * 2^(E + 17), the 24-bit
// significand shifted (right by -E from m24 * 2^17, truncating).
__device__ __forceinline__ void tp_fixed(float e, uint32_t& hi, uint32_t& lo) {
  const uint32_t b = __float_as_uint(e);
  const uint32_t m24 = (b & 0x7fffffu) | 0x800000u;
  const int r = 127 - (int)(b >> 23);   // -E, in [0, 127]; e = 0 gives 127
  const u64 f = r < 64 ? (((u64)m24 << 17) >> r) : 0ull;
  hi = (uint32_t)(f >> 20);
  lo = (uint32_t)f & 0xfffffu;
}
// A weight (hi, lo) into bin b of the warp's shared histogram (lo words at
// hl[0..255], hi words at hl[256..511]).  Between two flushes (at most 2048
// entries, each word < 2^20 + 1) no word overflows, so the additions need
// no carry and no returned value.
__device__ __forceinline__ void tp_add(uint32_t* hl, int b, uint32_t hi, uint32_t lo) {
  atomicAdd(&hl[b], lo);
  if (hi) atomicAdd(&hl[256 + b], hi);
}
// The warp's shared histogram added into a global one and cleared; `tail`
// goes into bin 255.
__device__ __forceinline__ void tp_flush(uint32_t* hl, u64* H, u64 tail) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int bin = lane * 8 + i;
    u64 v = ((u64)hl[256 + bin] << 20) + hl[bin];
    if (bin == 255) v += tail;
    if (v) atomicAdd(H + bin, v);   // a reduction: the result is not used
    hl[bin] = 0u;
    hl[256 + bin] = 0u;
  }
  __syncwarp();
}

// Pass 2: the mass histogram.
template <bool kBF16>
__device__ __noinline__ void tp_mass_pass(const Args& A, const TpPlan& T, uint32_t tag, uint32_t gw, uint32_t nwg,
                                          uint32_t* hl, unsigned char* b0, unsigned char* b1) {
  u64 t0, t1;
  tp_share(T, gw, nwg, &t0, &t1);
  int cj = -1;
  TpUnit U;
  TpMax M;
  M.live = false;
  M.m = 0.f;
  for (u64 tt = t0; tt < t1; ++tt) {
    const int j = (int)(tt / (u64)T.NT), t = (int)(tt % (u64)T.NT);
    if (j != cj) {
      cj = j;
      U = tp_unit(A, T, j);
      M = tp_max_of(A, T, U.uid, tag);
      if (t == 0 && (threadIdx.x & 31) == 0) __stcg(tp_summary(A, j) + 5, tagw(tag, M.key));
    }
    if (!M.live) continue;
    const float m = M.m, c = U.cfg.c;
    u64 tail = 0;
    u64* H = tp_hist(A, j, 0);
    tp_rows<kBF16>(A, U.lrow, 0, false, t * T.ET, T.NR, b0, b1, tp_chunk<kBF16>(),
                   [&](int, const unsigned char* g, const unsigned char*) {
                     uint32_t w[kBF16 ? 4 : 8];
                     tp_load_group<kBF16>(g, w);
#pragma unroll
                     for (int i = 0; i < 8; ++i) {
                       // e = 0 (-inf, or below 2^-126) weighs 0 and changes nothing
                       const float x = (tp_v<kBF16>(w, i) - m) * c;
                       uint32_t hi, lo;
                       tp_fixed(ex2(x), hi, lo);
                       const int b = tp_bin(x);
                       if (b < 255) tp_add(hl, b, hi, lo);
                       else tail += ((u64)hi << 20) | lo;
                     }
                   },
                   [&] { tp_flush(hl, H, 0ull); });
    tail = warp_sum_u64(tail);
    if ((threadIdx.x & 31) == 31 && tail) atomicAdd(H + 255, tail);
  }
}

// Pass 3, level L: the mass of the entries in the unit's key range, by key.
template <bool kBF16>
__device__ __noinline__ void tp_level_pass(const Args& A, const TpPlan& T, uint32_t tag, uint32_t gw, uint32_t nwg,
                                           uint32_t* hl, unsigned char* b0, unsigned char* b1, int L) {
  const int lane = threadIdx.x & 31;
  u64 t0, t1;
  tp_share(T, gw, nwg, &t0, &t1);
  int cj = -1;
  TpUnit U;
  TpMax M;
  TpState st;
  bool run = false;
  for (u64 tt = t0; tt < t1; ++tt) {
    const int j = (int)(tt / (u64)T.NT), t = (int)(tt % (u64)T.NT);
    if (j != cj) {
      cj = j;
      U = tp_unit(A, T, j);
      const u64 mw = __ldcg(tp_summary(A, j) + 5);
      if (L > 0) st = tp_state_after(A, j, L - 1);
      M = tp_max_from(mw, tag);
      run = false;
      if (M.live) {
        if (L == 0) st = tp_state0<kBF16>(A, j, M.m, U.cfg.c, U.cfg.P);
        if (t == 0) tp_state_store(A, j, L, st);
        // a unit found without a level of single-key bins (its crossing bin
        // holds one key, or the last level's sub-bin did) runs once more,
        // to list that key's entries per tile
        run = L == 0 || st.lo < st.hi || st.s_prev > 0;
        // the sub-bins hold several keys: the next level is needed (said
        // once, by the warp holding the unit's first tile)
        if (run && st.s > 0 && t == 0 && lane == 0) atomicOr(&cur(A).tp_more, 1u << (L + 1));
      }
    }
    if (!run) continue;
    const float m = M.m, c = U.cfg.c;
    // keys in [lo, hi] are the values in [vlo, vhi] (-0 and +0 share a key)
    const float vlo = tp_key_val<kBF16>(st.lo), vhi = tp_key_val<kBF16>(st.hi);
    // the unit's last level (its bins are single keys): count the entries
    // of each key too, for the tile's key list (bf16)
    const bool last = kBF16 && st.s == 0;
    uint32_t* cnt = hl + 512;
    u64* H = tp_hist(A, j, 1 + L);
    tp_rows<kBF16>(A, U.lrow, 0, false, t * T.ET, T.NR, b0, b1, tp_chunk<kBF16>(),
                   [&](int, const unsigned char* g, const unsigned char*) {
                     uint32_t w[kBF16 ? 4 : 8];
                     tp_load_group<kBF16>(g, w);
#pragma unroll
                     for (int i = 0; i < 8; ++i) {
                       const float v = tp_v<kBF16>(w, i);
                       if (v >= vlo && v <= vhi) {
                         const uint32_t key = kf<kBF16>(v);
                         const float x = (v - m) * c;
                         const float e = ex2(x);
                         if (e > 0.f && tp_bin(x) == st.b0) {
                           uint32_t hi, lo;
                           tp_fixed(e, hi, lo);
                           const int b = (int)((st.hi - key) >> st.s);
                           tp_add(hl, b, hi, lo);
                           if (last) atomicAdd(&cnt[b], 1u);
                         }
                       }
                     }
                   },
                   [&] { tp_flush(hl, H, 0ull); });
    if (last) {
      // the tile's key list: up to three keys with their counts
      uint32_t c8[8];
      uint32_t nz = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c8[i] = cnt[lane * 8 + i];
        cnt[lane * 8 + i] = 0u;
        nz += c8[i] ? 1u : 0u;
      }
      uint32_t total;
      uint32_t pos = warp_excl_scan_u32(nz, &total);
      if (total <= (uint32_t)kTpListLen) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (c8[i]) __stcg(tp_list(A, U.uid, t, (int)pos++), tagw(tag, (st.hi - (uint32_t)(lane * 8 + i)) | (c8[i] << 16)));
        if ((uint32_t)lane >= total && lane < kTpListLen) __stcg(tp_list(A, U.uid, t, lane), tagw(tag, 0u));
      } else if (lane == 0) {
        __stcg(tp_list(A, U.uid, t, 0), tagw(tag, kTpTieOverflow));
        atomicOr(&cur(A).tp_more, kTpNeedTies);
      }
      __syncwarp();
    }
  }
}

// The unit's summary from its final threshold state: the crossing key,
// how many entries at it are kept (n_need: enough of them to cover the mass
// still missing), Z_S over the kept set and whether P lies within the
// margin of the mass before or at the crossing entry.
struct TpSum {
  uint32_t tkey, n_need, mf;
  float Zs;
};
template <bool kBF16>
__device__ __forceinline__ TpSum tp_sum_of(const TpState& st, float m, const RowCfg& cfg, bool with_margin) {
  TpSum r;
  r.tkey = st.hi;
  const u64 efx = mass_fixed(ex2((tp_key_val<kBF16>(st.hi) - m) * cfg.c));
  u64 n = efx ? (st.rem + efx - 1u) / efx : 1u;
  if (n == 0) n = 1;
  r.n_need = (uint32_t)n;
  const u64 zs_fx = st.above + n * efx;
  r.Zs = (float)((double)zs_fx * (1.0 / 1099511627776.0));
  r.mf = 0u;
  if (with_margin) {
    const double P = (double)cfg.P;
    const double at = (double)zs_fx / (double)st.zk, bef = (double)(zs_fx - efx) / (double)st.zk;
    if (fabs(at - P) < 1e-6 || fabs(P - bef) < 1e-6) r.mf = SPEC_F_MARGIN_TOPP;
  }
  return r;
}
__device__ __forceinline__ void tp_sum_store(const Args& A, int j, uint32_t tag, const TpSum& r) {
  const int lane = threadIdx.x & 31;
  const uint32_t v = lane == 0 ? r.tkey : lane == 1 ? r.n_need : lane == 2 ? __float_as_uint(r.Zs) : r.mf;
  if (lane < 4) __stcg(tp_summary(A, j) + lane, tagw(tag, v));
}

// Pass 4 (fp32 rows, or a bf16 tile whose key list overflowed): entries at
// the crossing key, per tile.  The warp holding a unit's first tile also
// writes the unit's summary.
template <bool kBF16>
__device__ __noinline__ void tp_ties_pass(const Args& A, const TpPlan& T, uint32_t tag, uint32_t gw, uint32_t nwg,
                                          unsigned char* b0, unsigned char* b1) {
  const int lane = threadIdx.x & 31;
  u64 t0, t1;
  tp_share(T, gw, nwg, &t0, &t1);
  int cj = -1;
  TpUnit U;
  TpMax M;
  uint32_t tkey = 0u;
  for (u64 tt = t0; tt < t1; ++tt) {
    const int j = (int)(tt / (u64)T.NT), t = (int)(tt % (u64)T.NT);
    if (j != cj) {
      cj = j;
      U = tp_unit(A, T, j);
      const u64 mw = __ldcg(tp_summary(A, j) + 5);
      const TpState st = tp_state_after(A, j, T.nlev - 1);
      M = tp_max_from(mw, tag);
      tkey = st.hi;
      if (M.live && t == 0) tp_sum_store(A, j, tag, tp_sum_of<kBF16>(st, M.m, U.cfg, true));
    }
    if (!M.live) continue;
    const float tval = tp_key_val<kBF16>(tkey);   // the entries at the crossing key hold this value
    uint32_t n = 0;
    tp_rows<kBF16>(A, U.lrow, 0, false, t * T.ET, T.NR, b0, b1, tp_chunk<kBF16>(),
                   [&](int, const unsigned char* g, const unsigned char*) {
                     uint32_t w[kBF16 ? 4 : 8];
                     tp_load_group<kBF16>(g, w);
#pragma unroll
                     for (int i = 0; i < 8; ++i) n += tp_v<kBF16>(w, i) == tval ? 1u : 0u;
                   },
                   [] {});
    n = __reduce_add_sync(kAll, n);
    if (lane == 0) __stcg(tp_rec(A, U.uid, t), tagw(tag, n));
  }
}

// Entries at the crossing key in tile t: from pass 4's count, or from the
// tile's key list of the last refinement level.
__device__ __forceinline__ uint32_t tp_tile_ties(const Args& A, int uid, int t, uint32_t tag, bool counted,
                                                 uint32_t tkey, bool* ok) {
  const u64* R = tp_rec(A, uid, t);
  if (counted) {
    const u64 wd = __ldcg(R);
    *ok = *ok && tag_ok(wd, tag);
    return wu(wd);
  }
  u64 e[kTpListLen];
#pragma unroll
  for (int i = 0; i < kTpListLen; ++i) e[i] = __ldcg(tp_list(A, uid, t, i));
  bool good = wu(e[0]) != kTpTieOverflow;
  uint32_t n = 0;
#pragma unroll
  for (int i = 0; i < kTpListLen; ++i) {
    good = good && tag_ok(e[i], tag);
    if ((wu(e[i]) & 0xffffu) == tkey) n = wu(e[i]) >> 16;
  }
  *ok = *ok && good;
  return n;
}
// Entries at the crossing key in tiles [0, t) of a unit.
__device__ __forceinline__ u64 tp_ties_before(const Args& A, int uid, int t, uint32_t tag, bool counted,
                                              uint32_t tkey, bool* ok) {
  const int lane = threadIdx.x & 31;
  u64 s = 0;
  bool good = true;
  for (int i = lane; i < t; i += 32) s += tp_tile_ties(A, uid, i, tag, counted, tkey, &good);
  *ok = __all_sync(kAll, good);
  return warp_sum_u64(s);
}

// Pass 5: alpha and the level-1 races of each tile over the kept set (a tile
// has at most 32 blocks: lane r keeps the sums of block r).
template <bool kBF16>
__device__ __noinline__ void tp_tiles_pass(const Args& A, const TpPlan& T, uint32_t tag, uint32_t gw, uint32_t nwg,
                                           unsigned char* b0, unsigned char* b1) {
  const int lane = threadIdx.x & 31;
  u64 t0, t1;
  tp_share(T, gw, nwg, &t0, &t1);
  int cj = -1;
  TpUnit U;
  TpMax M;
  uint32_t tkey = 0u;
  u64 n_need = 0;
  float invZ = 0.f;
  for (u64 tt = t0; tt < t1; ++tt) {
    const int j = (int)(tt / (u64)T.NT), t = (int)(tt % (u64)T.NT);
    if (j != cj) {
      cj = j;
      U = tp_unit(A, T, j);
      if (T.ties) {
        // the unit's summary: crossing key, n_need, Z_S (pass 4) and max (pass 2)
        const u64 sw = lane < 6 ? __ldcg(tp_summary(A, j) + lane) : 0ull;
        const bool sok = __all_sync(kAll, lane > 3 || tag_ok(sw, tag));
        M = tp_max_from(shfl_u64(sw, 5), tag);
        if (!sok) M.live = false;   // the settle finds the summary missing too
        tkey = __shfl_sync(kAll, wu(sw), 0);
        n_need = __shfl_sync(kAll, wu(sw), 1);
        invZ = 1.0f / __uint_as_float(__shfl_sync(kAll, wu(sw), 2));
      } else {
        // no pass 4: the summary from the final state (the first tile's warp keeps it)
        const u64 mw = __ldcg(tp_summary(A, j) + 5);
        const TpState st = tp_state_after(A, j, T.nlev - 1);
        M = tp_max_from(mw, tag);
        if (M.live) {
          const TpSum sm = tp_sum_of<kBF16>(st, M.m, U.cfg, t == 0);
          if (t == 0) tp_sum_store(A, j, tag, sm);
          tkey = sm.tkey;
          n_need = sm.n_need;
          invZ = 1.0f / sm.Zs;
        }
      }
    }
    if (!M.live) continue;
    const float m = M.m, c = U.cfg.c;
    const float tval = tp_key_val<kBF16>(tkey);   // keys above tkey: values above tval
    bool ok;
    const u64 pre = tp_ties_before(A, U.uid, t, tag, T.ties, tkey, &ok);
    bool own_ok = true;
    const u64 cnt = tp_tile_ties(A, U.uid, t, tag, T.ties, tkey, &own_ok);
    // the tile's ties are all kept, none, or its first n_need - pre; the
    // tile holding the n_need-th tie ranks its ties and names that one
    const bool all_ties = pre + cnt <= n_need;
    const bool boundary = pre < n_need && n_need <= pre + cnt;
    const bool has_q = U.has_q;
    uint32_t run = (uint32_t)pre;   // ties before the current row
    uint32_t last_kept = 0xffffffffu;
    float a0 = 0.f, a1 = 0.f;
    float myW = 0.f, myU = 0.f, myP = 0.f;   // lane r: the sums of block r of the tile
    const int e_base = t * T.ET;
    tp_rows<kBF16>(
        A, U.lrow, U.qrow, has_q, e_base, T.NR, b0, b1, 4,
        [&](int r, const unsigned char* g, const unsigned char* gq) {
          uint32_t w[kBF16 ? 4 : 8];
          tp_load_group<kBF16>(g, w);
          float q[8];
          if (has_q) {
            const float4* s4 = reinterpret_cast<const float4*>(gq);
            const float4 qa = s4[0], qb = s4[1];
            q[0] = qa.x; q[1] = qa.y; q[2] = qa.z; q[3] = qa.w;
            q[4] = qb.x; q[5] = qb.y; q[6] = qb.z; q[7] = qb.w;
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) q[i] = 0.f;
          }
          uint32_t rank = 0u;
          if (boundary) {
            uint32_t cr = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) cr += tp_v<kBF16>(w, i) == tval ? 1u : 0u;
            uint32_t tot;
            rank = run + warp_excl_scan_u32(cr, &tot);
            run += tot;
          }
          float ws = 0.f, us = 0.f, ps = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float v = tp_v<kBF16>(w, i);
            bool in = v > tval;
            if (v == tval) {
              if (boundary) {
                in = (u64)rank < n_need;
                if ((u64)rank + 1u == n_need) last_kept = (uint32_t)(e_base + (r * 32 + lane) * 8 + i);
                ++rank;
              } else {
                in = all_ties;
              }
            }
            const float e = in ? ex2((v - m) * c) : 0.f;
            if (has_q) {
              const float p = e * invZ;
              if (i & 1) a1 += fminf(p, q[i]);
              else a0 += fminf(p, q[i]);
              const float wv = fmaxf(p - q[i], 0.f);   // >= 0: adding a zero changes nothing
              ws += wv;
              us += wv > 0.f ? wv + 2.0f * q[i] : 0.f;
            }
            ps += e;
          }
          const float W = has_q ? warp_sum(ws) : 0.f;
          const float Uq = has_q ? warp_sum(us) : 0.f;
          const float WP = warp_sum(ps);
          if (lane == r) {
            myW = W;
            myU = Uq;
            myP = WP;
          }
        },
        [] {});
    // one step of each level-1 race per block: lane r for block r of the tile
    Race rr, rp;
    race_init(rr);
    race_init(rp);
    if (lane < T.NR && (myW > 0.f || myP > 0.f)) {
      const uint32_t blk = (uint32_t)(t * T.NR + lane);
      const uint32_t word = block_word(A, U.row, U.pos, blk);
      if (myW > 0.f) race_consider(rr, myW, myU - myW, blk, word);
      if (myP > 0.f) race_consider(rp, myP, 0.f, blk, word);
    }
    if (has_q) warp_race_merge(rr);
    warp_race_merge(rp);
    if (boundary) {
      last_kept = __reduce_min_sync(kAll, last_kept);
      if (lane == 0) __stcg(tp_summary(A, j) + 4, tagw(tag, last_kept));
    }
    const float alpha = has_q ? warp_sum(a0 + a1) : 0.f;
    // a tile whose tie counts were not all there writes no record: the
    // settle then finds an old tag and gives the unit up
    const uint32_t v = lane == 1 ? __float_as_uint(alpha)
                     : lane == 2 ? __float_as_uint(rr.s1)
                     : lane == 3 ? __float_as_uint(rr.t1)
                     : lane == 4 ? __float_as_uint(rr.s2)
                     : lane == 5 ? __float_as_uint(rr.t2)
                     : lane == 6 ? rr.v1
                     : lane == 7 ? __float_as_uint(rp.s1)
                     : lane == 8 ? __float_as_uint(rp.t1)
                     : lane == 9 ? __float_as_uint(rp.s2)
                     : lane == 10 ? __float_as_uint(rp.t2)
                                  : rp.v1;
    if (ok && own_ok && lane >= 1 && lane <= 11) __stcg(tp_rec(A, U.uid, t) + lane, tagw(tag, v));
  }
}

__device__ __forceinline__ Race tp_race_of(const u64* R, bool* ok, uint32_t tag) {
  Race r;
  const u64 w0 = __ldcg(R), w1 = __ldcg(R + 1), w2 = __ldcg(R + 2), w3 = __ldcg(R + 3), w4 = __ldcg(R + 4);
  *ok = *ok && tag_ok(w0, tag) && tag_ok(w1, tag) && tag_ok(w2, tag) && tag_ok(w3, tag) && tag_ok(w4, tag);
  r.s1 = wf(w0);
  r.t1 = wf(w1);
  r.s2 = wf(w2);
  r.t2 = wf(w3);
  r.v1 = wu(w4);
  r.s1lo = r.s1 * 0.99999905f;
  return r;
}

// Pass 6: one warp settles a unit.
template <bool kBF16>
__device__ __noinline__ void tp_settle_pass(const Args& A, const TpPlan& T, uint32_t tag, uint32_t gw, uint32_t nwg,
                                            bool failed) {
  const int lane = threadIdx.x & 31;
  // unit j on CTA j mod n_ctas, warp j / n_ctas: consecutive units on
  // different SMs, so that the settles (one warp's latency-bound code each)
  // do not share an SM's schedulers while others sit idle
  const uint32_t wpc = blockDim.x >> 5;
  const uint32_t jfirst = (gw % wpc) * (uint32_t)A.n_ctas + gw / wpc;
  for (int j = (int)jfirst; j < T.nU; j += (int)nwg) {
    const TpUnit U = tp_unit(A, T, j);
    if (failed) {
      commit_record(A, tag, U.uid, U.row, empty_record(SPEC_F_TIMEOUT));
      continue;
    }
    // the summary, the draft and the tiles' alphas and races, in one round trip
    const int xd = U.has_q ? A.drafts[(size_t)U.row * A.k + U.pos] : -1;
    const u64 sw = lane < 6 ? __ldcg(tp_summary(A, j) + lane) : 0ull;
    bool ok = lane > 4 || tag_ok(sw, tag);
    float asum = 0.f;
    Race rr, rp;
    race_init(rr);
    race_init(rp);
    for (int t = lane; t < T.NT; t += 32) {
      const u64* R = tp_rec(A, U.uid, t);
      const u64 wa = __ldcg(R + 1);
      ok = ok && tag_ok(wa, tag);
      asum += wf(wa);
      if (U.has_q) race_merge(rr, tp_race_of(R + 2, &ok, tag));
      race_merge(rp, tp_race_of(R + 7, &ok, tag));
    }
    const TpMax M = tp_max_from(shfl_u64(sw, 5), tag);
    if (!M.live) {
      commit_record(A, tag, U.uid, U.row, empty_record(M.missing ? SPEC_F_TIMEOUT : SPEC_F_NAN));
      continue;
    }
    if (!__all_sync(kAll, ok)) {
      // a record of this unit is missing (a pass gave up)
      commit_record(A, tag, U.uid, U.row, empty_record(SPEC_F_TIMEOUT));
      continue;
    }
    const RowCfg& cfg = U.cfg;
    const float m = M.m, c = cfg.c;
    AcceptInfo ai = accept_load(A, U.row, U.pos, kBF16, xd);   // in flight during the merges
    const uint32_t tkey = __shfl_sync(kAll, wu(sw), 0);
    const float Zs = __uint_as_float(__shfl_sync(kAll, wu(sw), 2));
    const uint32_t flags = __shfl_sync(kAll, wu(sw), 3);
    Thresh th;
    th.tkey = full_key<kBF16>(tkey);
    th.tidx = __shfl_sync(kAll, wu(sw), 4);
    const float alpha_v = U.has_q ? warp_sum(asum) : 0.f;
    if (U.has_q) warp_race_merge(rr);
    warp_race_merge(rp);
    const float invZ = 1.0f / Zs, lnZ = logf(Zs);
    bool need_race = !U.has_q;
    if (U.has_q) {
      ai = accept_decide(A, U.row, U.pos, ai, false, 0, m, c, Zs, &th);
      need_race = !ai.accept;
    }
    uint32_t draw_flags = 0u;
    uint32_t y = 0xffffffffu;
    float ly = 0.f;
    if (need_race) {
      Race l1 = rp;
      int mode = U.has_q ? RW_P : RW_BONUS;
      if (U.has_q) {
        if (rr.s1 >= 0.f) {
          l1 = rr;
          mode = RW_RESIDUAL;
        } else {
          draw_flags |= SPEC_F_RESIDUAL_EMPTY;
        }
      }
      if (l1.s1 >= 0.f) {
        const Race l2 = race_in_block<kBF16, true>(A, U.row, U.pos, l1.v1, m, c, invZ, mode, &th, &ly);
        if (l2.s1 >= 0.f) y = l2.v1;
        if (draw_margin(l1) || draw_margin(l2)) draw_flags |= SPEC_F_MARGIN_DRAW;
      }
    }
    UnitRecord rec = empty_record(flags);
    if (lane == 0) {
      if (U.has_q) {
        if (!ai.valid) rec.flags |= SPEC_F_BAD_TOKEN;
        if (ai.margin) rec.flags |= SPEC_F_MARGIN_ACCEPT;
        rec.accept = ai.accept ? 1 : 0;
        rec.lp_x = ai.valid ? (ai.lx - m) * cfg.invT - lnZ : 0.f;
        rec.alpha = alpha_v;
      }
      if (need_race) {
        if (y < (uint32_t)A.V) {
          rec.y = (int32_t)y;
          rec.lp_y = (ly - m) * cfg.invT - lnZ;
        } else {
          // no entry won (not reachable: the kept set holds the max)
          rec.flags |= SPEC_F_TIMEOUT;
        }
        rec.draw_flags = draw_flags;
      }
    }
    publish_desc(A, tag, U.uid, DESC_THRESH, m, invZ, th.tkey, th.tidx);
    commit_record(A, tag, U.uid, U.row, rec);
  }
}

// Every CTA arrives before any leaves (the launch is cooperative, so all are
// resident).  The count only grows within a call: barrier i waits for
// i x n_ctas arrivals.  Bounded by the global timer: a wait that lasts a
// second gives up and sets ERR_BARRIER.
constexpr unsigned long long kBarrierNs = 1000000000ull;
__device__ __noinline__ void grid_barrier(const Args& A, uint32_t target) {
  __syncthreads();
  if (threadIdx.x == 0) {
    // a release add (ordering the CTA's writes, which the block barrier
    // made this thread's to release, before the arrival) and acquire loads
    // (ordering everything after the wait, which the block barrier below
    // passes on to the CTA's other threads)
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&cur(A).bar) : "memory");
    const unsigned long long t0 = global_ns();
    long long spins = 0;
    while (load_acquire(&cur(A).bar) < target) {
      if ((++spins & 63) == 0 && global_ns() - t0 > kBarrierNs) {
        atomicOr(&cur(A).error, (uint32_t)ERR_BARRIER);
        break;
      }
      __nanosleep(spins > 16 ? 128 : 16);
    }
  }
  __syncthreads();
}

// The passes, run by every thread of every CTA.  `buf` is the warp's 16 KB
// of shared memory: the mass passes' histogram and key counts (3 KB) and two
// 4 KB chunk buffers; pass 5 uses all of it for two chunks of logits and q.  `usable`
// is false for a warp whose buffers may still receive a copy that gave up
// (it then takes no tiles, and the units come back with SPEC_F_TIMEOUT).
template <bool kBF16>
__device__ __noinline__ void topp_passes(const Args& A, TpPlan T, uint32_t tag, unsigned char* buf, bool usable) {
  const uint32_t w = threadIdx.x >> 5;
  const uint32_t nwg = (uint32_t)A.n_ctas * (uint32_t)(blockDim.x >> 5);
  const uint32_t gw = blockIdx.x * (blockDim.x >> 5) + w;
  // tile size: one tile per warp where the units allow it
  const int NB = ceil_div(A.V, kRaceBlock);
  const int per = max(1, (int)(nwg / (uint32_t)max(1, T.nU)));
  T.NR = min(kTpMaxBlocks, max(kTpMinBlocks, ceil_div(NB, per)));
  T.ET = T.NR * kRaceBlock;
  T.NT = ceil_div(NB, T.NR);
  uint32_t* hist = reinterpret_cast<uint32_t*>(buf);   // 3 KB: mass low and high words, key counts
  unsigned char* c0 = buf + 3072;                      // chunk buffers of the logits-only passes
  unsigned char* c1 = buf + 7168;
  unsigned char* d0 = buf;                             // pass 5: chunks of logits and q
  unsigned char* d1 = buf + 8192;
  uint32_t nb = 0;
  const uint32_t n = (uint32_t)A.n_ctas;
  // timeline stamps (instrumented builds): barrier exits of CTA 0, pass ends per warp
  auto stamp_bar = [&]() { if (threadIdx.x == 0 && blockIdx.x == 0) TL(TL_TP, (int)nb, 16); };
  auto stamp_pass = [&](int p) { if ((threadIdx.x & 31) == 0) TL(TL_TP_WARP + p * 2048, (int)gw, 2048); };
  for (int i = (int)(threadIdx.x & 31); i < 3 * kTpBins / 4; i += 32)
    reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncwarp();
  // test hook: CTA 0 reaches the first barrier 1.5 s late, after the
  // others' wait has given up (a bounded sleep)
  if (threadIdx.x == 0 && blockIdx.x == 0 && (__ldcg(&A.ws->inject) & 2u) != 0u) {
    const unsigned long long t0 = global_ns();
    for (int i = 0; i < 4000 && global_ns() - t0 < kBarrierNs + kBarrierNs / 2; ++i) __nanosleep(1000000);
  }
  stamp_bar();
  grid_barrier(A, ++nb * n);   // the roles are done and the scratch is zero everywhere
  stamp_bar();
  if (usable) tp_max_pass<kBF16>(A, T, tag, gw, nwg, c0, c1);
  stamp_pass(0);
  grid_barrier(A, ++nb * n);
  stamp_bar();
  if (usable) tp_mass_pass<kBF16>(A, T, tag, gw, nwg, hist, c0, c1);
  stamp_pass(1);
  grid_barrier(A, ++nb * n);
  stamp_bar();
  int L = 0;
  for (; L < kTpLevels; ++L) {
    if (L > 0 && (__ldcg(&cur(A).tp_more) & (1u << L)) == 0u) break;
    if (usable) tp_level_pass<kBF16>(A, T, tag, gw, nwg, hist, c0, c1, L);
    stamp_pass(2 + L);
    grid_barrier(A, ++nb * n);
    stamp_bar();
  }
  T.nlev = L;
  T.ties = !kBF16 || (__ldcg(&cur(A).tp_more) & kTpNeedTies) != 0u;
  if (T.ties) {
    if (usable) tp_ties_pass<kBF16>(A, T, tag, gw, nwg, c0, c1);
    stamp_pass(6);
    grid_barrier(A, ++nb * n);
    stamp_bar();
  }
  if (usable) tp_tiles_pass<kBF16>(A, T, tag, gw, nwg, d0, d1);
  stamp_pass(7);
  grid_barrier(A, ++nb * n);
  stamp_bar();
  const bool failed = (__ldcg(&cur(A).error) & (uint32_t)(ERR_BARRIER | ERR_COPY_WAIT)) != 0u;
  tp_settle_pass<kBF16>(A, T, tag, gw, nwg, failed);
  stamp_pass(5);
}

}  // namespace specv
