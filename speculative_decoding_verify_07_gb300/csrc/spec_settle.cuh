// spec_verify, settle code (sm_103a): what one warp does with a unit once
// every tile of it has been reduced.
//
//   greedy and unfiltered units: merge the A records in tile order -- max,
//     first argmax, the softmax sum rescaled to the unit max; greedy units
//     and unfiltered bonus positions are settled at once (the bonus draw
//     merges the tiles' level-1 block races and races the winning block's
//     entries); a drafted unfiltered unit takes its accept test and
//     publishes its state for the B tiles; after the B pass its B records
//     are merged (alpha and the residual draw).
//   small top-k units: every A tile lists the 8 largest entries of its
//     tile in the total order, the smallest of them last.  A tile whose
//     smallest listed entry is below the K-th entry of the merged lists holds
//     no further top-K entry, so the merged lists give the top-K set; other
//     tiles are re-read from L2.  Top-p, the accept test, alpha and the draw
//     run on the sorted list.
//
// Every record poll is bounded; a unit whose records do not all arrive, or
// one of whose tiles gave up a wait, is settled as invalid with
// SPEC_F_TIMEOUT.  The last settled unit of a row resolves the accept chain
// and writes the row's outputs.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_common.cuh"

namespace specv {

constexpr unsigned kSettleFull = 0xffffffffu;
// Record tiles a lane loads before merging any of them: A records in
// fin_stats, B records in fin_b (one batch each at V = 151936).
constexpr int kFinBatchA = 2;
constexpr int kFinBatchB = 4;

// The state of a drafted unfiltered unit as tagged words (lanes 0..7).
__device__ __forceinline__ void publish_state(const Args& A, uint32_t tag, int u, UnitState st) {
  const int lane = threadIdx.x & 31;
  const uint32_t v = lane_word8(lane, __float_as_uint(st.m), __float_as_uint(st.invZ), __float_as_uint(st.lnZ),
                                __float_as_uint(st.lp_x), (uint32_t)st.accept, st.flags, st.invalid, (uint32_t)st.am);
  if (lane < kStateWords) __stcg(A.ust + (size_t)u * kStateWords + lane, tagw(tag, v));
  __syncwarp();
}

// Warp loop guard for polling a set of words: true while another pass is
// needed (not all lanes saw the tag); gives up after kSpinLimit passes and
// sets *timed_out.
__device__ __forceinline__ bool poll_again(const Args& A, bool ok, long long& spins, bool* timed_out) {
  if (__all_sync(kSettleFull, ok)) return false;
  if (++spins > kSpinLimit) {
    if ((threadIdx.x & 31) == 0) atomicOr(&cur(A).error, (uint32_t)ERR_RECORD_WAIT);
    *timed_out = true;
    return false;
  }
  __nanosleep(64);
  return true;
}

// The draft token of the unit and its logit and q (inputs, loaded before
// the records are merged so that the loads are in flight meanwhile).
struct Pre {
  int x, valid;
  float lx, qx;
};

template <bool kBF16>
__device__ __forceinline__ Pre load_pre(const Args& A, int u, int row, int pos) {
  Pre pr;
  pr.x = -1;
  pr.valid = 0;
  pr.lx = 0.f;
  pr.qx = 0.f;
  if (pos < A.k) {
    pr.x = A.drafts[(size_t)row * A.k + pos];
    pr.valid = pr.x >= 0 && pr.x < A.V;
    if (pr.valid) {
      pr.lx = load_logit(A, kBF16, (size_t)u * A.V + pr.x);
      pr.qx = A.q[((size_t)row * A.k + pos) * (size_t)A.V + pr.x];
    }
  }
  return pr;
}

// Accept test of the draft at (row, pos) from prefetched operands: accept iff
// u*q(x) < p(x), the sign of u*q - p taken exactly by one fma; greedy:
// p(x) = 1 if x is the argmax, else 0.
__device__ __forceinline__ AcceptInfo accept_pre(const Args& A, int row, int pos, const Pre& pr, bool greedy, int am,
                                                 float m, float c, float Zs) {
  AcceptInfo ai;
  ai.x = pr.x;
  ai.valid = pr.valid != 0;
  ai.lx = pr.lx;
  ai.qx = pr.qx;
  ai.px = 0.f;
  if (ai.valid) ai.px = greedy ? (ai.x == am ? 1.0f : 0.0f) : ex2((ai.lx - m) * c) / Zs;
  const float u = accept_uniform(A, row, pos);
  const float d = fmaf(u, ai.qx, -ai.px);
  ai.accept = d < 0.0f;
  ai.margin = (ai.px > 0.0f && ai.px < 1.0f && fabsf(d) < kMargin);
  return ai;
}

// First index of the row maximum, by one warp (only for a draw that found
// no positive weight, which a valid row does not produce).
template <bool kBF16>
__device__ __noinline__ int row_argmax(const Args& A, size_t lrow) {
  const int lane = threadIdx.x & 31;
  const int G = (A.V + 7) / 8;
  unsigned long long best = 0;
  for (int g = lane; g < G; g += 32) {
    float v[8];
    load_group<kBF16>(A, lrow, g, true, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (g * 8 + i >= A.V) continue;
      const unsigned long long k = key64(okey(v[i]), (uint32_t)(g * 8 + i));
      best = k > best ? k : best;
    }
  }
  return (int)key64_idx(warp_max_u64(best));
}

// Draw from p over a whole row by one warp (the fallback when a residual is
// empty): each lane sums the weights of its own blocks (level 1), then the
// winning block's entries race (level 2).
template <bool kBF16>
__device__ __noinline__ uint32_t warp_draw_p(const Args& A, int row, int pos, float m, float c, bool* margin) {
  const int lane = threadIdx.x & 31;
  const size_t lrow = ((size_t)row * (A.k + 1) + pos) * (size_t)A.V;
  const int nblk = ceil_div(A.V, kRaceBlock);
  const int G = (A.V + 7) / 8;
  Race r1;
  race_init(r1);
  for (int b = lane; b < nblk; b += 32) {
    float W = 0.f;
    for (int g = b * (kRaceBlock / 8); g < (b + 1) * (kRaceBlock / 8) && g < G; ++g) {
      float v[8];
      load_group<kBF16>(A, lrow, g, true, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) W += (g * 8 + j < A.V) ? ex2((v[j] - m) * c) : 0.f;
    }
    if (W > 0.f) race_consider(r1, W, 0.f, (uint32_t)b, block_word(A, row, pos, (uint32_t)b));
  }
  warp_race_merge(r1);
  if (r1.s1 < 0.f) {
    *margin = false;
    return 0xffffffffu;
  }
  const Race l2 = race_in_block<kBF16>(A, row, pos, r1.v1, m, c, 1.f, RW_P, nullptr);
  *margin = draw_margin(r1) || draw_margin(l2);
  return l2.v1;
}

// ---------------------------------------------------------------------------
// Greedy and unfiltered units.
// ---------------------------------------------------------------------------
// Merges the A records.  Greedy units and bonus positions are settled here;
// a drafted unfiltered unit publishes its state: its B records are merged
// later (fin_b).
template <bool kBF16>
__device__ __noinline__ void fin_stats(const Args& A, uint32_t tag, int u, int row, int pos, RowCfg cfg,
                                       Pre pr, bool late) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const bool has_q = pos < A.k;
  const bool greedy = cfg.type == UT_GREEDY;
  const bool bonus = !greedy && !has_q;
  const int NT = ceil_div(A.V, G::EA);
  const u64* R = A.rec + (size_t)u * A.NTA * kRecWords;
  const size_t lrow = (size_t)u * A.V;
  // one pass over the records: each lane keeps its max, the first tile
  // holding it, and its share of the softmax sum relative to that max
  bool nan = false, tmo = false, timed_out = false;
  float m = -INFINITY, zl = 0.f;
  int cm = 0x7fffffff;
  // words 0..7 of a batch of each lane's tiles (word 1 only for greedy
  // units, words 3..7 only for bonus positions); with one batch they stay
  // held for the bonus merge below
  u64 w[kFinBatchA][8];
#pragma unroll
  for (int i = 0; i < kFinBatchA; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) w[i][j] = 0ull;
  {
    long long spins = 0;
    bool ok;
    do {
      ok = true;
      nan = false;
      tmo = false;
      m = -INFINITY;
      zl = 0.f;
      cm = 0x7fffffff;
      for (int c0 = 0; c0 < NT; c0 += 32 * kFinBatchA) {
        // the batch's words are all in flight before the first is used
#pragma unroll
        for (int i = 0; i < kFinBatchA; ++i) {
          const int c = c0 + 32 * i + lane;
#pragma unroll
          for (int j = 0; j < 8; ++j) w[i][j] = 0ull;
          if (c < NT) {
            const u64* r = R + (size_t)c * kRecWords;
            w[i][0] = __ldcg(r);
            w[i][2] = __ldcg(r + 2);
            if (greedy) w[i][1] = __ldcg(r + 1);
            if (bonus) {
#pragma unroll
              for (int j = 3; j < 8; ++j) w[i][j] = __ldcg(r + j);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < kFinBatchA; ++i) {
          const int c = c0 + 32 * i + lane;
          if (c >= NT) continue;
          ok = ok && tag_ok(w[i][0], tag) && tag_ok(w[i][2], tag);
          if (greedy) ok = ok && tag_ok(w[i][1], tag);
          if (bonus) {
#pragma unroll
            for (int j = 3; j < 8; ++j) ok = ok && tag_ok(w[i][j], tag);
          }
          const float mc = wf(w[i][0]), zc = wf(w[i][2]);
          if (wu(w[i][0]) == kTimeoutNaN) {
            tmo = true;
          } else if (mc != mc) {
            nan = true;
          } else if (mc > -INFINITY) {
            if (mc > m) {
              zl = (m > -INFINITY ? zl * ex2((m - mc) * cfg.c) : 0.f) + zc;
              m = mc;
              cm = c;
            } else {
              zl += zc * ex2((mc - m) * cfg.c);
            }
          }
        }
      }
    } while (poll_again(A, ok, spins, &timed_out));
  }
  TLP(u, 1);
  nan = __any_sync(kSettleFull, nan);
  tmo = __any_sync(kSettleFull, tmo) || timed_out;
  const float mw = warp_max_f(m);
  const int cfirst = (int)warp_min_u32((m == mw && cm != 0x7fffffff) ? (uint32_t)cm : 0xffffffffu);
  const bool invalid = tmo || nan || !(mw > -INFINITY) || !(mw < INFINITY);
  const uint32_t base_flags = cfg.bad_param ? SPEC_F_BAD_PARAM : 0u;
  if (invalid) {
    const uint32_t f = tmo ? SPEC_F_TIMEOUT : SPEC_F_NAN;
    if (cfg.type == UT_DENSE && has_q) {
      // the B tiles skip an invalid unit
      UnitState z;
      memset(&z, 0, sizeof(z));
      z.invalid = 1;
      z.flags = f;
      publish_state(A, tag, u, z);
    }
    commit_record(A, tag, u, row, empty_record(f));
    return;
  }
  const float m_lane = m;
  m = mw;
  // the softmax sum rescaled to the unit max (fixed lane order)
  const float Z = warp_sum(cm != 0x7fffffff ? zl * ex2((m_lane - m) * cfg.c) : 0.f);
  const float lnZ = logf(Z);
  if (greedy) {
    const int am = (int)wu(__ldcg(R + (size_t)cfirst * kRecWords + 1));
    TLP(u, 2);
    UnitRecord rec = empty_record(base_flags);
    if (lane == 0) {
      bool need_draw = !has_q;
      float q_am = 0.f;
      if (has_q) {
        const AcceptInfo ai = accept_pre(A, row, pos, pr, true, am, m, cfg.c, 1.f);
        if (!ai.valid) rec.flags |= SPEC_F_BAD_TOKEN;
        rec.accept = ai.accept ? 1 : 0;
        rec.lp_x = ai.valid ? (ai.lx - m) - lnZ : 0.f;
        q_am = A.q[((size_t)row * A.k + pos) * (size_t)A.V + am];
        rec.alpha = fminf(1.0f, q_am);
        need_draw = !ai.accept;
      }
      if (need_draw) {
        rec.y = am;
        rec.lp_y = -lnZ;
        if (has_q && !(1.0f - q_am > 0.0f)) rec.draw_flags |= SPEC_F_RESIDUAL_EMPTY;
      }
    }
    TLP(u, 3);
    publish_desc(A, tag, u, DESC_GREEDY, m, 0.f, 0u, (uint32_t)am);
    commit_record(A, tag, u, row, rec);
    return;
  }
  if (bonus) {
    // merge the tiles' block races (scaled to the unit max), then race the
    // entries of the winning block
    Race a;
    race_init(a);
    const bool held = NT <= 32 * kFinBatchA;   // w holds every tile's words
    for (int c0 = 0; c0 < NT; c0 += 32 * kFinBatchA) {
      u64 x[kFinBatchA][6];   // words 0 and 3..7 of the batch's tiles
#pragma unroll
      for (int i = 0; i < kFinBatchA; ++i) {
        const int c = c0 + 32 * i + lane;
#pragma unroll
        for (int j = 0; j < 6; ++j) x[i][j] = 0ull;
        if (held) {
          x[i][0] = w[i][0];
#pragma unroll
          for (int j = 1; j < 6; ++j) x[i][j] = w[i][2 + j];
        } else if (c < NT) {
          const u64* r = R + (size_t)c * kRecWords;
          x[i][0] = __ldcg(r);
#pragma unroll
          for (int j = 1; j < 6; ++j) x[i][j] = __ldcg(r + 2 + j);
        }
      }
#pragma unroll
      for (int i = 0; i < kFinBatchA; ++i) {
        if (c0 + 32 * i + lane >= NT) continue;
        const float mc = wf(x[i][0]);
        const float sc = mc > -INFINITY ? ex2((mc - m) * cfg.c) : 0.f;
        Race b;
        b.s1 = wf(x[i][1]);
        b.t1 = wf(x[i][2]);
        b.s2 = wf(x[i][3]);
        b.t2 = wf(x[i][4]);
        b.v1 = wu(x[i][5]);
        b.s1lo = 0.f;
        race_scale(b, sc);
        race_merge(a, b);
      }
    }
    warp_race_merge(a);
    TLP(u, 2);
    float ly = 0.f;
    // (every entry of the block weighs: the rolled loop's out-of-line
    // updates beat the inline steps here even for a warp's last task)
    const Race l2 = race_in_block<kBF16>(A, row, pos, a.v1, m, cfg.c, 1.f, RW_BONUS, nullptr, &ly);
    TLP(u, 3);
    uint32_t y = l2.v1;
    const bool drawn = l2.s1 >= 0.f && y < (uint32_t)A.V;
    if (!drawn) y = (uint32_t)row_argmax<kBF16>(A, lrow);
    UnitRecord rec = empty_record(base_flags);
    if (lane == 0) {
      rec.y = (int32_t)y;
      rec.lp_y = ((drawn ? ly : load_logit(A, kBF16, lrow + y)) - m) * cfg.invT - lnZ;
      if (draw_margin(a) || draw_margin(l2)) rec.draw_flags |= SPEC_F_MARGIN_DRAW;
    }
    TLP(u, 4);
    publish_desc(A, tag, u, DESC_ALL, m, 1.0f / Z, 0u, 0u);
    commit_record(A, tag, u, row, rec);
    return;
  }
  // drafted: accept test, then publish the state for the B tiles
  AcceptInfo ai;
  if (lane == 0) ai = accept_pre(A, row, pos, pr, false, -1, m, cfg.c, Z);
  UnitState st;
  st.m = m;
  st.invZ = 1.0f / Z;
  st.lnZ = lnZ;
  st.accept = __shfl_sync(kSettleFull, (lane == 0 && ai.accept) ? 1 : 0, 0);
  st.lp_x = __shfl_sync(kSettleFull, lane == 0 ? (ai.valid ? (ai.lx - m) * cfg.invT - lnZ : 0.f) : 0.f, 0);
  st.flags = __shfl_sync(kSettleFull,
                         lane == 0 ? base_flags | (ai.valid ? 0u : SPEC_F_BAD_TOKEN) | (ai.margin ? SPEC_F_MARGIN_ACCEPT : 0u)
                                   : 0u, 0);
  st.invalid = 0;
  st.am = -1;
  publish_state(A, tag, u, st);
}

// The unit state words of a drafted unfiltered unit, as loaded.
struct StateWords {
  u64 w[kStateWords];
};

// The unit state words of a drafted unfiltered unit.
__device__ __forceinline__ void state_load(const Args& A, int u, u64 (&w)[kStateWords]) {
#pragma unroll
  for (int i = 0; i < kStateWords; ++i) w[i] = __ldcg(A.ust + (size_t)u * kStateWords + i);
}
__device__ __forceinline__ bool state_ok(const u64 (&w)[kStateWords], uint32_t tag) {
  bool ok = true;
#pragma unroll
  for (int i = 0; i < kStateWords; ++i) ok = ok && tag_ok(w[i], tag);
  return ok;
}
__device__ __forceinline__ UnitState state_of(const u64 (&w)[kStateWords]) {
  UnitState st;
  st.m = wf(w[0]);
  st.invZ = wf(w[1]);
  st.lnZ = wf(w[2]);
  st.lp_x = wf(w[3]);
  st.accept = (int32_t)wu(w[4]);
  st.flags = wu(w[5]);
  st.invalid = wu(w[6]);
  st.am = (int32_t)wu(w[7]);
  return st;
}

// A drafted unfiltered unit after its B tiles: alpha from the tiles' sums,
// and after a rejection the residual draw from the tiles' level-1 races.
// The state was published before any B tile of the unit ran, so it is
// read without a wait.
template <bool kBF16>
__device__ __noinline__ void fin_b(const Args& A, uint32_t tag, int u, int row, int pos, RowCfg cfg,
                                   StateWords sw0, bool late) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  u64 sw[kStateWords];
#pragma unroll
  for (int i = 0; i < kStateWords; ++i) sw[i] = sw0.w[i];
  bool timed_out = false;
  {
    long long spins = 0;
    while (poll_again(A, state_ok(sw, tag), spins, &timed_out)) state_load(A, u, sw);
  }
  const UnitState st = state_of(sw);
  if (timed_out) {
    commit_record(A, tag, u, row, empty_record(SPEC_F_TIMEOUT));
    return;
  }
  if (st.invalid) return;   // its record was committed with the state
  const int NT = ceil_div(A.V, G::EB);
  const u64* R = A.brec + (size_t)u * A.NTB * kBRecWords;
  const bool need_race = !st.accept;
  float al = 0.f;
  bool tmo = false;
  Race a;
  race_init(a);
  {
    long long spins = 0;
    bool ok;
    do {
      ok = true;
      al = 0.f;
      tmo = false;
      race_init(a);
      // each lane's tiles lane, lane + 32, ... in batches of kFinBatchB:
      // the batch's words are all in flight before the first is merged
      for (int c0 = 0; c0 < NT; c0 += 32 * kFinBatchB) {
        u64 w[kFinBatchB][6];
#pragma unroll
        for (int i = 0; i < kFinBatchB; ++i) {
          const int c = c0 + 32 * i + lane;
#pragma unroll
          for (int j = 0; j < 6; ++j) w[i][j] = 0ull;
          if (c < NT) {
            const u64* r = R + (size_t)c * kBRecWords;
            w[i][0] = __ldcg(r);
            if (need_race) {
#pragma unroll
              for (int j = 1; j < 6; ++j) w[i][j] = __ldcg(r + j);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < kFinBatchB; ++i) {
          if (c0 + 32 * i + lane >= NT) continue;
          ok = ok && tag_ok(w[i][0], tag);
          if (wu(w[i][0]) == kTimeoutNaN) tmo = true;
          al += wf(w[i][0]);
          if (need_race) {
#pragma unroll
            for (int j = 1; j < 6; ++j) ok = ok && tag_ok(w[i][j], tag);
            Race rb;
            rb.s1 = wf(w[i][1]);
            rb.t1 = wf(w[i][2]);
            rb.s2 = wf(w[i][3]);
            rb.t2 = wf(w[i][4]);
            rb.v1 = wu(w[i][5]);
            rb.s1lo = 0.f;
            race_merge(a, rb);
          }
        }
      }
    } while (poll_again(A, ok, spins, &timed_out));
  }
  TLP(u, 6);
  if (__any_sync(kSettleFull, tmo) || timed_out) {
    commit_record(A, tag, u, row, empty_record(SPEC_F_TIMEOUT));
    return;
  }
  const float alpha_v = warp_sum(al);
  uint32_t draw_flags = 0;
  uint32_t y = 0xffffffffu;
  float ly = 0.f;
  bool drawn = false;   // ly holds the logit of y
  if (need_race) {
    warp_race_merge(a);
    if (a.s1 >= 0.f) {
      const Race l2 = late ? race_in_block<kBF16, true>(A, row, pos, a.v1, st.m, cfg.c, st.invZ, RW_RESIDUAL, nullptr, &ly)
                           : race_in_block<kBF16>(A, row, pos, a.v1, st.m, cfg.c, st.invZ, RW_RESIDUAL, nullptr, &ly);
      y = l2.v1;
      drawn = l2.s1 >= 0.f && y < (uint32_t)A.V;
      if (draw_margin(a) || draw_margin(l2)) draw_flags |= SPEC_F_MARGIN_DRAW;
    } else {
      draw_flags |= SPEC_F_RESIDUAL_EMPTY;
      bool mg = false;
      y = warp_draw_p<kBF16>(A, row, pos, st.m, cfg.c, &mg);
      if (mg) draw_flags |= SPEC_F_MARGIN_DRAW;
    }
    if (y >= (uint32_t)A.V) y = (uint32_t)row_argmax<kBF16>(A, (size_t)u * A.V);
  }
  TLP(u, 7);
  UnitRecord rec = empty_record(st.flags);
  if (lane == 0) {
    rec.accept = st.accept;
    rec.lp_x = st.lp_x;
    rec.alpha = alpha_v;
    if (need_race) {
      rec.y = (int32_t)y;
      rec.lp_y = ((drawn ? ly : load_logit(A, kBF16, (size_t)u * A.V + y)) - st.m) * cfg.invT - st.lnZ;
      rec.draw_flags = draw_flags;
    }
  }
  commit_record(A, tag, u, row, rec);
}

// First bin (from bin 0) where the running count over hist[0..256) reaches
// `need` (>= 1); 256 when the total is below it.  *before = the count of the
// bins before it.  Lane l scans bins 8l..8l+7.
__device__ __forceinline__ int warp_select_bin(const uint32_t* hist, uint32_t need, uint32_t* before) {
  const int lane = threadIdx.x & 31;
  uint32_t h[8], own = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = hist[8 * lane + i];
    own += h[i];
  }
  uint32_t inc = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kSettleFull, inc, o);
    if (lane >= o) inc += y;
  }
  const unsigned ball = __ballot_sync(kSettleFull, inc >= need);
  if (!ball) {
    *before = __shfl_sync(kSettleFull, inc, 31);
    return 256;
  }
  const int src = __ffs(ball) - 1;
  int bin = 0;
  uint32_t acc = inc - own;
  if (lane == src) {
    bin = 8 * lane + 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (acc + h[i] >= need) {
        bin = 8 * lane + i;
        break;
      }
      acc += h[i];
    }
  }
  *before = __shfl_sync(kSettleFull, acc, src);
  return __shfl_sync(kSettleFull, bin, src);
}

// Exclusive warp scan of a count; *total = the warp's sum.
__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t x, uint32_t* total) {
  const int lane = threadIdx.x & 31;
  uint32_t inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kSettleFull, inc, o);
    if (lane >= o) inc += y;
  }
  *total = __shfl_sync(kSettleFull, inc, 31);
  return inc - x;
}

// Descending bitonic sort of s[0..n) (n <= 256) in shared memory by one warp,
// padded with zeros to a power of two >= 32; rolled loops keep it small.
static __device__ __noinline__ void warp_sort_desc(u64* s, int n) {
  const int lane = threadIdx.x & 31;
  if (n <= 64) {
    // in registers: lane holds entries lane and lane + 32; a pair at stride
    // 32 is in one lane, other pairs are one shuffle apart.  The pair's
    // lower entry keeps the larger key iff the pair's run descends.
    u64 x0 = lane < n ? s[lane] : 0ull, x1 = lane + 32 < n ? s[lane + 32] : 0ull;
#pragma unroll 1
    for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll 1
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        if (stride == 32) {
          const u64 hi = x0 > x1 ? x0 : x1, lo = x0 > x1 ? x1 : x0;
          x0 = hi;   // size 64: one descending run
          x1 = lo;
        } else {
          const u64 o0 = __shfl_xor_sync(kSettleFull, x0, stride), o1 = __shfl_xor_sync(kSettleFull, x1, stride);
          const bool lower = (lane & stride) == 0;
          const bool k0 = lower == ((lane & size) == 0), k1 = lower == (((lane + 32) & size) == 0);
          x0 = k0 ? (o0 > x0 ? o0 : x0) : (o0 < x0 ? o0 : x0);
          x1 = k1 ? (o1 > x1 ? o1 : x1) : (o1 < x1 ? o1 : x1);
        }
      }
    }
    __syncwarp();
    s[lane] = x0;
    s[lane + 32] = x1;
    __syncwarp();
    return;
  }
  int N = 32;
  while (N < n) N <<= 1;
  for (int i = n + lane; i < N; i += 32) s[i] = 0ull;
  __syncwarp();
#pragma unroll 1
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll 1
      for (int q = lane; q < (N >> 1); q += 32) {
        const int lo = 2 * q - (q & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const u64 a = s[lo], b = s[hi];
        if ((a < b) == desc) {
          s[lo] = b;
          s[hi] = a;
        }
      }
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------------------
// Small top-k, one warp.
// ---------------------------------------------------------------------------
constexpr int kSel = 128;                  // candidates held for the sort (>= kTopkSmall)

// Scratch of one settle warp.
struct TopkScratch {
  u64 cand[kMaxListCand];                  // the A tiles' lists as total-order keys (0 = none)
  uint32_t hist[256];
  u64 sel[kSel];                           // the selected candidates
  float qsel[kSel];                        // q of the selected candidates
  uint8_t cflag[kMaxListCand / kList];     // per tile: bit 0 NaN, bit 1 partial list, bit 2 timeout
};
static_assert(kTopkSmall <= 256 && kTopkSmall % 32 == 0, "the list is held 32 entries per round");

// Calls fn(g, v) on every lane for groups 8 entries g = g0 + step * 32 + lane
// (g < g1; lanes past the end get g = -1 and -inf values), loading four steps
// ahead.
template <bool kBF16, typename F>
__device__ __forceinline__ void sweep_range(const Args& A, size_t lrow, int g0, int g1, F fn) {
  const int lane = threadIdx.x & 31;
  for (int base = g0; base < g1; base += 128) {
    float v[4][8];
    int g[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      g[s] = base + 32 * s + lane;
      if (g[s] < g1) {
        load_group<kBF16>(A, lrow, g[s], true, v[s]);
      } else {
        g[s] = -1;
#pragma unroll
        for (int i = 0; i < 8; ++i) v[s][i] = -INFINITY;
      }
    }
#pragma unroll
    for (int s = 0; s < 4; ++s)
      if (base + 32 * s < g1) fn(g[s], v[s]);
  }
}

// Appends, in the order of the calls, the entries whose bit is set in `keep`
// (8 per lane, entries 8g..8g+7) to sel[*n ...] (up to kSel); *n counts all.
__device__ __forceinline__ void append_entries(u64* sel, uint32_t* n, int g, uint32_t keep, const uint32_t* keys) {
  uint32_t tot = 0;
  uint32_t p = *n + warp_excl_scan((uint32_t)__popc(keep), &tot);
  *n += tot;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if ((keep >> i) & 1u) {
      if (p < (uint32_t)kSel) sel[p] = key64(keys[i], (uint32_t)(g * 8 + i));
      ++p;
    }
}

// Exact top-K (or every finite entry, when fewer) of the whole row into
// sel[], by radix passes over the row (8 bits at a time from the top), then
// the entries above the K-th key and the first ties in index order.  For rows
// whose lists cannot settle the unit (masses of ties).  Returns the count.
template <bool kBF16>
__device__ __noinline__ int select_k_row(const Args& A, TopkScratch& S, size_t lrow, int K) {
  const int lane = threadIdx.x & 31;
  const int G = (A.V + 7) / 8;
  const uint32_t T32 = okey(-INFINITY) + 1u;          // finite entries
  uint32_t prefix = 0u, mask = 0u, need = (uint32_t)K;
  bool all = false;
  const int lowest = kBF16 ? 16 : 0;        // bf16 keys are fixed by their top 16 bits
  for (int shift = 24; shift >= lowest; shift -= 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) S.hist[8 * lane + i] = 0u;
    __syncwarp();
    sweep_range<kBF16>(A, lrow, 0, G, [&](int g, const float* v) {
      if (g < 0) return;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t key = okey(v[i]);
        if (g * 8 + i < A.V && key >= T32 && (key & mask) == prefix)
          atomicAdd(&S.hist[255u - ((key >> shift) & 255u)], 1u);   // bin 0 = the top byte value
      }
    });
    __syncwarp();
    uint32_t before = 0;
    const int b = warp_select_bin(S.hist, need, &before);
    __syncwarp();
    if (b == 256) {            // fewer than K finite entries: all of them
      all = true;
      break;
    }
    need -= before;
    prefix |= (uint32_t)(255 - b) << shift;
    mask |= 255u << shift;
  }
  const uint32_t tkey = all ? T32 : (kBF16 ? full_key<true>(prefix >> 16) : prefix);
  uint32_t n_out = 0, ties_seen = 0;
  sweep_range<kBF16>(A, lrow, 0, G, [&](int g, const float* v) {
    uint32_t gt = 0, eq = 0;
    uint32_t keys[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      keys[i] = okey(v[i]);
      const bool in = g >= 0 && g * 8 + i < A.V;
      gt |= (in && (all ? keys[i] >= tkey : keys[i] > tkey)) ? (1u << i) : 0u;
      eq |= (in && !all && keys[i] == tkey) ? (1u << i) : 0u;
    }
    uint32_t te = 0;
    uint32_t r = ties_seen + warp_excl_scan((uint32_t)__popc(eq), &te);
    ties_seen += te;
    uint32_t keep = gt;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((eq >> i) & 1u) {
        if (r < need) keep |= 1u << i;
        ++r;
      }
    append_entries(S.sel, &n_out, g, keep, keys);
  });
  __syncwarp();
  return (int)min(n_out, (uint32_t)kSel);
}

static_assert(kList == 8, "list slot q mod 8 of tile q / 8");

static_assert(kSel >= kTopkSmall, "the selection holds the K largest");
static_assert(sizeof(TopkScratch) <= kSlot, "top-k settle scratch exceeds a stream buffer");
static_assert(kTopkSmall * 8 <= 256 * 4, "the sorted keys fit the histogram area");

// The exact top-K of a small top-k unit when a tile may hold more top-K
// entries than it listed (a full list ending above kappa, or one marked
// partial): those tiles are re-read (their entries at or above kappa join
// the listed entries at or above kappa of the other tiles), or, when that
// gives more than kSel entries (masses of ties), the whole row by radix
// passes.  One warp; the lists are in S.cand and S.cflag.  Leaves the K (or
// all, when fewer) largest sorted in S.sel with their q in S.qsel; returns
// their count.
template <bool kBF16>
__device__ __noinline__ int topk_rescan(const Args& A, TopkScratch& S, int NT, int NL, u64 kappa, int K, size_t lrow,
                                        size_t qrow, bool has_q) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  int n_k = 0;
  uint32_t n = 0;
  bool exact = true;
  for (int base = 0; base < NL; base += 32) {
    const int q = base + lane;
    const u64 k = q < NL ? S.cand[q] : 0ull;
    const int ch = q / kList;
    const u64 last = q < NL ? S.cand[ch * kList + kList - 1] : 0ull;
    const bool safe_ch = q < NL && (S.cflag[ch] & 2u) == 0 && !(last != 0ull && last > kappa);
    const bool in = safe_ch && k != 0ull && k >= kappa;
    const unsigned ball = __ballot_sync(kSettleFull, in);
    const uint32_t p = n + __popc(ball & ((1u << lane) - 1u));
    if (in && p < (uint32_t)kSel) S.sel[p] = k;
    n += __popc(ball);
  }
  const uint32_t T = max((uint32_t)(kappa >> 32), okey(-INFINITY) + 1u);
  for (int ch = 0; ch < NT; ++ch) {
    const u64 last = S.cand[ch * kList + kList - 1];
    if (!((S.cflag[ch] & 2u) != 0 || (last != 0ull && last > kappa))) continue;
    const int g0 = ch * (G::EA / 8);
    const int g1 = min(ceil_div(A.V, 8), g0 + G::EA / 8);
    sweep_range<kBF16>(A, lrow, g0, g1, [&](int g, const float* v) {
      uint32_t keep = 0;
      uint32_t keys[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        keys[i] = okey(v[i]);
        const bool inr = g >= 0 && g * 8 + i < A.V && keys[i] >= T && key64(keys[i], (uint32_t)(g * 8 + i)) >= kappa;
        keep |= inr ? (1u << i) : 0u;
      }
      append_entries(S.sel, &n, g, keep, keys);
    });
  }
  __syncwarp();
  if (n <= (uint32_t)kSel) {
    warp_sort_desc(S.sel, (int)n);
    n_k = min((int)n, K);
  } else {
    exact = false;
  }
  if (!exact) {
    const int nn = select_k_row<kBF16>(A, S, lrow, K);
    warp_sort_desc(S.sel, nn);
    n_k = min(nn, K);
  }
  for (int i = lane; i < n_k; i += 32) S.qsel[i] = has_q ? A.q[qrow + key64_idx(S.sel[i])] : 0.f;
  __syncwarp();
  return n_k;
}

// The rest of a small top-k settle, by one warp, from the kept entries in
// the total order (keys lk[0..n_k), their q in lq): prefix sums for top-p,
// alpha, the accept test, the two-level race over the kept entries, the
// unit record.  S.sel is scratch here (lk and lq are read first).
template <bool kBF16>
__device__ __noinline__ void topk_tail(const Args& A, uint32_t tag, TopkScratch& S, int u, int row, int pos,
                                       RowCfg cfg, Pre pr, const u64* lk, const float* lq, int n_k, float m, int am) {
  const int lane = threadIdx.x & 31;
  const bool has_q = pos < A.k;
  const float c = cfg.c;
  pr.x = __shfl_sync(kSettleFull, pr.x, 0);
  pr.valid = __shfl_sync(kSettleFull, pr.valid, 0);
  pr.lx = __shfl_sync(kSettleFull, pr.lx, 0);
  pr.qx = __shfl_sync(kSettleFull, pr.qx, 0);
  // the list in shared memory (in the candidate area, no longer needed):
  // entry i holds index, logit, e = exp2((l - m) c), q, prefix sum of e
  // (entries 32 r + lane in rounds r: rolled loops keep the code small)
  uint32_t* Li = reinterpret_cast<uint32_t*>(S.cand);
  float* Lv = reinterpret_cast<float*>(Li + kTopkSmall);
  float* Le = Lv + kTopkSmall;
  float* Lq = Le + kTopkSmall;
  float* Lc = Lq + kTopkSmall;
  float* Lw = Lc + kTopkSmall;   // race weights
  float* Lu = Lw + kTopkSmall;   // their margin weights
  static_assert(7 * kTopkSmall * 4 <= sizeof(u64) * kMaxListCand, "list arrays exceed the candidate area");
  const int nr = (n_k + 31) >> 5;
  float run = 0.f;
#pragma unroll 1
  for (int r = 0; r < nr; ++r) {
    const int i = 32 * r + lane;
    const bool in = i < n_k;
    const u64 key = in ? lk[i] : 0ull;
    const float v = in ? from_okey((uint32_t)(key >> 32)) : 0.f;
    const float e = in ? ex2((v - m) * c) : 0.f;
    // inclusive prefix sums in the total order (fixed order)
    float inc = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(kSettleFull, inc, o);
      if (lane >= o) inc += y;
    }
    if (in) {
      Li[i] = key64_idx(key);
      Lv[i] = v;
      Le[i] = e;
      Lq[i] = lq[i];
      Lc[i] = run + inc;
    }
    run += __shfl_sync(kSettleFull, inc, 31);
  }
  __syncwarp();
  TLP(u, 4);
  const float Zk = Lc[n_k - 1];
  uint32_t flags = cfg.bad_param ? SPEC_F_BAD_PARAM : 0u;
  int n_s = n_k;
  if (cfg.P < 1.0f) {
    const float target = cfg.P * Zk;
#pragma unroll 1
    for (int r = 0; r < nr; ++r) {
      const int i = 32 * r + lane;
      const unsigned ball = __ballot_sync(kSettleFull, i < n_k && Lc[i] >= target);
      if (ball) {
        n_s = 32 * r + __ffs(ball);
        break;
      }
    }
    const float at = Lc[n_s - 1] / Zk;
    const float bef = n_s >= 2 ? Lc[n_s - 2] / Zk : 0.f;
    if (fabsf(at - cfg.P) < kMargin || fabsf(cfg.P - bef) < kMargin) flags |= SPEC_F_MARGIN_TOPP;
  }
  const float Zs = Lc[n_s - 1];
  const float invZ = 1.0f / Zs;
  const float lnZ = logf(Zs);
  const int sr = (n_s + 31) >> 5;
  float alpha_v = 0.f;
  AcceptInfo ai;
  ai.valid = true;
  ai.accept = false;
  ai.margin = false;
  ai.lx = 0.f;
  bool need_race = !has_q;
  if (has_q) {
    float a = 0.f, ex = -1.f;
#pragma unroll 1
    for (int r = 0; r < sr; ++r) {
      const int i = 32 * r + lane;
      if (i < n_s) {
        a += fminf(Le[i] * invZ, Lq[i]);
        if (Li[i] == (uint32_t)pr.x) ex = Le[i];
      }
    }
    alpha_v = warp_sum(a);
    const unsigned hb = __ballot_sync(kSettleFull, ex >= 0.f);
    const float exx = hb ? __shfl_sync(kSettleFull, ex, __ffs(hb) - 1) : 0.f;
    ai.x = pr.x;
    ai.valid = pr.valid != 0;
    ai.px = hb ? exx / Zs : 0.f;
    ai.qx = pr.qx;
    ai.lx = pr.lx;
    const float uu = accept_uniform(A, row, pos);
    const float d = fmaf(uu, ai.qx, -ai.px);
    ai.accept = d < 0.0f;
    ai.margin = (ai.px > 0.0f && ai.px < 1.0f && fabsf(d) < kMargin);
    need_race = !ai.accept;
  }
  TLP(u, 5);
  // the draw: the two-level race over the kept entries (blocks by index)
  uint32_t draw_flags = 0;
  uint32_t y = 0xffffffffu;
  if (need_race) {
#pragma unroll 1
    for (int attempt = 0; attempt < 2; ++attempt) {
      const bool resid = has_q && attempt == 0;   // attempt 1: an empty residual, draw from p
#pragma unroll 1
      for (int r = 0; r < sr; ++r) {
        const int i = 32 * r + lane;
        if (i < n_s) {
          const float p = Le[i] * invZ;
          const float w = resid ? fmaxf(p - Lq[i], 0.f) : p;
          Lw[i] = w;
          Lu[i] = w + (resid ? 2.0f * Lq[i] : 0.f);
        }
      }
      __syncwarp();
      // level 1: a block's weights summed in list order; the block's first
      // entry with weight races for it
      Race r1;
      race_init(r1);
#pragma unroll 1
      for (int r = 0; r < sr; ++r) {
        const int i = 32 * r + lane;
        const bool mine = i < n_s && Lw[i] > 0.f;
        const uint32_t bl = mine ? Li[i] / kRaceBlock : 0xffffffffu;
        float W = 0.f, WU = 0.f;
        bool owner = mine;
#pragma unroll 1
        for (int j = 0; j < n_s; ++j) {
          const float wj = Lw[j];
          if (wj > 0.f && Li[j] / kRaceBlock == bl) {
            W += wj;
            WU += Lu[j];
            owner = owner && j >= i;
          }
        }
        if (owner) race_consider(r1, W, WU - W, bl, block_word(A, row, pos, bl));
      }
      warp_race_merge(r1);
      if (r1.s1 < 0.f) {
        draw_flags |= SPEC_F_RESIDUAL_EMPTY;
        continue;
      }
      // level 2: the entries of the winning block
      Race r2;
      race_init(r2);
#pragma unroll 1
      for (int r = 0; r < sr; ++r) {
        const int i = 32 * r + lane;
        if (i < n_s && Lw[i] > 0.f && Li[i] / kRaceBlock == r1.v1)
          race_consider(r2, Lw[i], Lu[i] - Lw[i], Li[i], race_word(A, row, pos, Li[i]));
      }
      warp_race_merge(r2);
      y = r2.v1;
      if (draw_margin(r1) || draw_margin(r2)) draw_flags |= SPEC_F_MARGIN_DRAW;
      break;
    }
  }
  TLP(u, 6);
  // the logit of the drawn entry, from the list
  float vy = m;
  {
    float vv = 0.f;
    bool own = false;
#pragma unroll 1
    for (int r = 0; r < nr; ++r) {
      const int i = 32 * r + lane;
      if (i < n_k && Li[i] == y) {
        vv = Lv[i];
        own = true;
      }
    }
    const unsigned ob = __ballot_sync(kSettleFull, own);
    if (ob) vy = __shfl_sync(kSettleFull, vv, __ffs(ob) - 1);
  }
  UnitRecord rec = empty_record(flags);
  if (lane == 0) {
    if (has_q) {
      if (!ai.valid) rec.flags |= SPEC_F_BAD_TOKEN;
      if (ai.margin) rec.flags |= SPEC_F_MARGIN_ACCEPT;
      rec.accept = ai.accept ? 1 : 0;
      rec.lp_x = ai.valid ? (ai.lx - m) * cfg.invT - lnZ : 0.f;
      rec.alpha = alpha_v;
    }
    if (need_race) {
      const bool ok = y < (uint32_t)A.V;
      rec.y = ok ? (int32_t)y : am;
      rec.lp_y = ((ok ? vy : m) - m) * cfg.invT - lnZ;
      rec.draw_flags = draw_flags;
    }
  }
  TLP(u, 7);
  publish_desc(A, tag, u, DESC_THRESH, m, invZ, (uint32_t)(lk[n_s - 1] >> 32), Li[n_s - 1]);
  commit_record(A, tag, u, row, rec);
}

// The value keys of the listed entries, CR per lane (candidate 32 r + lane
// in round r; 0 for an empty slot), held in registers for the bisection.
template <int CR>
struct KeyRounds {
  uint32_t k[CR];
};
template <int CR>
__device__ __forceinline__ uint32_t count_key_ge(const KeyRounds<CR>& K, uint32_t t) {
  uint32_t n = 0;
#pragma unroll
  for (int r = 0; r < CR; ++r) n += K.k[r] >= t ? 1u : 0u;
  return __reduce_add_sync(kSettleFull, n);
}

// The K-th largest listed entry in the total order (0 when fewer than K are
// listed), by bisection on the value key within [lo, hi] (lo at or below it,
// hi the largest), then on the index among the entries at that key.
template <bool kBF16, int CR>
__device__ __noinline__ u64 kth_listed(const u64* cand, int NL, uint32_t K, uint32_t lo, uint32_t hi,
                                       uint32_t* tmp) {
  const int lane = threadIdx.x & 31;
  KeyRounds<CR> R;
#pragma unroll
  for (int r = 0; r < CR; ++r) {
    const int q = 32 * r + lane;
    R.k[r] = q < NL ? (uint32_t)(cand[q] >> 32) : 0u;
  }
  if (count_key_ge(R, 1u) < K) return 0ull;
  uint32_t tkey;
  if (kBF16) {
    // bf16 keys are fixed by their top 16 bits
    uint32_t l = lo >> 16, h = hi >> 16;
    while (l < h) {
      const uint32_t mid = l + ((h - l + 1u) >> 1);
      if (count_key_ge(R, max(mid << 16, 1u)) >= K) l = mid;
      else h = mid - 1u;
    }
    tkey = full_key<true>(l);
  } else {
    uint32_t l = max(lo, 1u), h = hi;
    while (l < h) {
      const uint32_t mid = l + (uint32_t)(((u64)h - l + 1ull) >> 1);
      if (count_key_ge(R, mid) >= K) l = mid;
      else h = mid - 1u;
    }
    tkey = l;
  }
  const uint32_t n_gt = tkey == 0xffffffffu ? 0u : count_key_ge(R, tkey + 1u);
  const uint32_t need = K - n_gt;   // entries at the key, smallest indices first
  const uint32_t n_eq = count_key_ge(R, tkey) - n_gt;
  uint32_t low = 0xffffffffu;
  for (int q = lane; q < NL; q += 32)
    if ((uint32_t)(cand[q] >> 32) == tkey) low = min(low, (uint32_t)cand[q]);
  low = __reduce_min_sync(kSettleFull, low);
  if (n_eq == need) return ((u64)tkey << 32) | low;   // every entry at the key is kept
  if (n_eq <= 32u) {
    // bf16 values tie often: gather the entries at the key (tmp, 32 words)
    // and take the one with need - 1 larger low words (0xffffffff - index)
    uint32_t n = 0;
    for (int q0 = 0; q0 < NL; q0 += 32) {
      const int q = q0 + lane;
      const u64 k = q < NL ? cand[q] : 0ull;
      const bool in = (uint32_t)(k >> 32) == tkey;
      const unsigned ball = __ballot_sync(kSettleFull, in);
      const uint32_t p = n + __popc(ball & ((1u << lane) - 1u));
      if (in && p < 32u) tmp[p] = (uint32_t)k;
      n += __popc(ball);
    }
    __syncwarp();
    const uint32_t my = (uint32_t)lane < n_eq ? tmp[lane] : 0u;
    uint32_t rk = 0;
    for (uint32_t j = 0; j < n_eq; ++j) rk += tmp[j] > my ? 1u : 0u;
    const unsigned win = __ballot_sync(kSettleFull, (uint32_t)lane < n_eq && rk == need - 1u);
    const uint32_t lw = __shfl_sync(kSettleFull, my, __ffs(win) - 1);
    __syncwarp();
    return ((u64)tkey << 32) | lw;
  }
  // the need-th largest low word (0xffffffff - index) among the entries at tkey
  uint32_t l = low, h = 0xffffffffu;
  while (l < h) {
    const uint32_t mid = l + (uint32_t)(((u64)h - l + 1ull) >> 1);
    uint32_t n = 0;
    for (int q = lane; q < NL; q += 32)
      n += ((uint32_t)(cand[q] >> 32) == tkey && (uint32_t)cand[q] >= mid) ? 1u : 0u;
    if (__reduce_add_sync(kSettleFull, n) >= need) l = mid;
    else h = mid - 1u;
  }
  return ((u64)tkey << 32) | l;
}

// Settle a small top-k unit with one warp; S is scratch in shared memory
// (one of the warp's stream buffers).
//   1. The tiles' lists into S.cand (candidate q: tile q / 8, slot q mod 8),
//      loaded 10 candidates a lane at a time.
//   2. tau: the ceil(K / 8)-th largest value key among the last entries of
//      full lists -- that many lists hold 8 entries at or above it, so the
//      K-th listed entry is at or above it.  The listed entries at or above
//      tau (a few more than K) are gathered with their q, each one's rank
//      among them is counted, and the K first go to their places, which
//      sorts them; kappa is the K-th.  A tile whose list is full and ends
//      above kappa, or is marked partial, may hold more top-K entries: then
//      such tiles are re-read (topk_rescan).
//   3. Top-p, alpha, the accept test and the draw (topk_tail).
template <bool kBF16>
__device__ __noinline__ void topk_settle(const Args& A, uint32_t tag, TopkScratch& S, int u, int row, int pos,
                                         RowCfg cfg, Pre pr) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const bool has_q = pos < A.k;
  const int NT = ceil_div(A.V, G::EA);
  const int NL = NT * kList;
  const u64* R = A.rec + (size_t)u * A.NTA * kRecWords;
  const size_t lrow = (size_t)u * A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const int K = cfg.K;

  // 1. the lists
  uint32_t allf = 0;
  bool timed_out = false;
  {
    long long spins = 0;
    bool ok;
    do {
      ok = true;
      uint32_t fl = 0;
      // ten candidates a lane at a time: one round trip for a bf16 row of
      // V <= 163840 (40 tiles)
      constexpr int kB = 10;
#pragma unroll 1
      for (int q0 = 0; q0 < NL; q0 += 32 * kB) {
        u64 wk[kB], wi[kB];
#pragma unroll
        for (int i = 0; i < kB; ++i) {
          const int q = q0 + 32 * i + lane;
          wk[i] = 0ull;
          wi[i] = 0ull;
          if (q < NL) {
            const u64* r = R + (size_t)(q >> 3) * kRecWords + 2 * (q & 7);
            wk[i] = __ldcg(r);
            wi[i] = __ldcg(r + 1);
          }
        }
#pragma unroll
        for (int i = 0; i < kB; ++i) {
          const int q = q0 + 32 * i + lane;
          if (q < NL) {
            ok = ok && tag_ok(wk[i], tag) && tag_ok(wi[i], tag);
            const uint32_t key = (uint32_t)wk[i], iw = (uint32_t)wi[i];
            fl |= iw & (kListNaN | kListPartial | kListTimeout);
            S.cand[q] = key ? key64(key, (uint32_t)((q >> 3) * G::EA) + (iw & kListIdx)) : 0ull;
            if ((q & 7) == 0) S.cflag[q >> 3] = (uint8_t)((iw & kListPartial) ? 2u : 0u);
          }
        }
      }
      allf = __reduce_or_sync(kSettleFull, fl);
    } while (poll_again(A, ok, spins, &timed_out));
  }
  __syncwarp();
  TLP(u, 1);
  if ((allf & kListTimeout) || timed_out) {
    commit_record(A, tag, u, row, empty_record(SPEC_F_TIMEOUT));
    return;
  }
  // the maximum and the count of listed entries
  u64 top = 0ull;
  uint32_t cnt = 0;
  for (int q = lane; q < NL; q += 32) {
    const u64 k = S.cand[q];
    top = k > top ? k : top;
    cnt += k ? 1u : 0u;
  }
  top = warp_max_u64(top);
  cnt = __reduce_add_sync(kSettleFull, cnt);
  const float m = from_okey((uint32_t)(top >> 32));
  if ((allf & kListNaN) || top == 0ull || !(m > -INFINITY) || !(m < INFINITY)) {
    commit_record(A, tag, u, row, empty_record(SPEC_F_NAN));
    return;
  }
  const int am = (int)key64_idx(top);
  TLS(u, 0);

  // 2. tau (a lower bound of the K-th listed value key), kappa by bisection
  // above it, the K entries at or above kappa (in S.sel) with their q, ranked
  uint32_t tau = 1u;
  {
    uint32_t v[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int ch = lane + 32 * i;
      v[i] = ch < NT ? (uint32_t)(S.cand[ch * kList + kList - 1] >> 32) : 0u;
    }
    static_assert(kMaxListCand / kList <= 96, "three list ends per lane");
    const int need = (K + kList - 1) / kList;
#pragma unroll 1
    for (int i = 0; i < need; ++i) {
      const uint32_t lm = max(v[0], max(v[1], v[2]));
      const uint32_t M = __reduce_max_sync(kSettleFull, lm);
      tau = max(M, 1u);
      if (M == 0u) break;
      // one occurrence leaves: the first lane holding it, its first slot
      const int src = __ffs(__ballot_sync(kSettleFull, lm == M)) - 1;
      if (lane == src) {
        if (v[0] == M) v[0] = 0u;
        else if (v[1] == M) v[1] = 0u;
        else v[2] = 0u;
      }
    }
  }
  // candidates a lane holds: a small top-k unit has at most kMaxListCand / kList
  // tiles of fp32 logits, half as many of bf16
  constexpr int CR = (kBF16 ? kMaxListCand / 2 : kMaxListCand) / 32;
  static_assert(Geo<true>::EA == 2 * Geo<false>::EA, "bf16 tiles hold twice the entries");
  TLS(u, 1);
  const u64 kappa = kth_listed<kBF16, CR>(S.cand, NL, (uint32_t)K, tau, (uint32_t)(top >> 32),
                                          reinterpret_cast<uint32_t*>(S.qsel));
  TLS(u, 2);
  const int n_k = (int)min(cnt, (uint32_t)K);
  {
    uint32_t n = 0;
    for (int q0 = 0; q0 < NL; q0 += 32) {
      const int q = q0 + lane;
      const u64 k = q < NL ? S.cand[q] : 0ull;
      const bool in = k != 0ull && k >= kappa;
      const unsigned ball = __ballot_sync(kSettleFull, in);
      const uint32_t p = n + __popc(ball & ((1u << lane) - 1u));
      if (in && p < (uint32_t)kSel) S.sel[p] = k;
      n += __popc(ball);
    }
  }
  __syncwarp();
  TLS(u, 3);
  u64* sorted = reinterpret_cast<u64*>(S.hist);
  {
    // q of the gathered entries (in flight while they are ranked)
    u64 mk[kSel / 32];
    float mq[kSel / 32];
    uint32_t rk[kSel / 32];
#pragma unroll
    for (int r = 0; r < kSel / 32; ++r) {
      const int i = 32 * r + lane;
      mk[r] = i < n_k ? S.sel[i] : 0ull;
      const uint32_t v = key64_idx(mk[r]);
      mq[r] = (has_q && mk[r] && v < (uint32_t)A.V) ? __ldcg(A.q + qrow + v) : 0.f;
      rk[r] = 0u;
    }
#pragma unroll 2
    for (int j = 0; j < n_k; ++j) {
      const u64 kj = S.sel[j];
#pragma unroll
      for (int r = 0; r < kSel / 32; ++r) rk[r] += kj > mk[r] ? 1u : 0u;
    }
#pragma unroll
    for (int r = 0; r < kSel / 32; ++r)
      if (mk[r]) {
        sorted[rk[r]] = mk[r];
        S.qsel[rk[r]] = mq[r];
      }
  }
  __syncwarp();
  TLS(u, 4);
  bool unsafe = false;
  for (int ch = lane; ch < NT; ch += 32) {
    const u64 last = S.cand[ch * kList + kList - 1];
    unsafe |= (S.cflag[ch] & 2u) != 0 || (last != 0ull && last > kappa);
  }
  unsafe = __any_sync(kSettleFull, unsafe);
  TLP(u, 2);
  if (unsafe) {
    const int nr = topk_rescan<kBF16>(A, S, NT, NL, kappa, K, lrow, qrow, has_q);
    topk_tail<kBF16>(A, tag, S, u, row, pos, cfg, pr, S.sel, S.qsel, nr, m, am);
  } else {
    topk_tail<kBF16>(A, tag, S, u, row, pos, cfg, pr, sorted, S.qsel, n_k, m, am);
  }
}

}  // namespace specv
