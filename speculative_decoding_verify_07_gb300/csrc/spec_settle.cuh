// spec_verify, settle code (sm_103a): what one warp does with a unit whose
// chunk records are complete.
//
//   greedy and unfiltered units: merge the chunk records in chunk order --
//     max, first argmax, the softmax sum rescaled to the unit max; greedy
//     units and unfiltered bonus positions are settled at once (the bonus
//     draw merges the chunks' level-1 block races and races the winning
//     block's entries); a drafted unfiltered unit takes its accept test and
//     publishes its state for the B items.
//   small top-k units: every top-K entry lies in a 64-entry super-group
//     whose maximum is among the K largest super-group maxima, so the K-th
//     largest maximum bounds the candidates.  A histogram of the maxima's
//     distances from the unit maximum gives that bound in one pass; the
//     candidates are gathered from L2, the first K of the total order
//     selected exactly and sorted, and top-p, the accept test, alpha and the
//     draw run on that list.
//
// The last settled unit of a row resolves the accept chain and writes the
// row's outputs.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify_common.cuh"

namespace specv {

constexpr unsigned kSettleFull = 0xffffffffu;

// The draft token of the unit and its logit and q (inputs).
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
  const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)pos, (uint32_t)row, 0u), A.key0, A.key1);
  const float u = uniform_of(w.x);
  const float d = fmaf(u, ai.qx, -ai.px);
  ai.accept = d < 0.0f;
  ai.margin = (ai.px > 0.0f && ai.px < 1.0f && fabsf(d) < kMargin);
  return ai;
}

template <bool kBF16>
__device__ __noinline__ void fin_stats(const Args& A, int u, int row, int pos, const RowCfg& cfg) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const bool has_q = pos < A.k;
  const int NC = ceil_div(A.V, G::EA);
  const ChunkRec* R = A.crec + (size_t)u * A.NCA;
  const Pre pr = load_pre<kBF16>(A, u, row, pos);   // lane 0's copy is the one used
  // one pass over the records: each lane keeps its max, the first chunk
  // holding it, and its share of the softmax sum relative to that max
  bool nan = false;
  float m = -INFINITY, zl = 0.f;
  int cm = 0x7fffffff;
  for (int c = lane; c < NC; c += 32) {
    const float mc = __ldcg(&R[c].m);
    const float zc = __ldcg(&R[c].z);
    if (mc != mc) {
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
  nan = __any_sync(kSettleFull, nan);
  const float mw = warp_max_f(m);
  const int cfirst = (int)warp_min_u32((m == mw && cm != 0x7fffffff) ? (uint32_t)cm : 0xffffffffu);
  const bool invalid = nan || !(mw > -INFINITY) || !(mw < INFINITY);
  const uint32_t base_flags = cfg.bad_param ? SPEC_F_BAD_PARAM : 0u;
  if (invalid) {
    if (lane == 0) {
      if (cfg.type == UT_DENSE && has_q) {
        UnitState st;
        memset(&st, 0, sizeof(st));
        st.invalid = 1;
        A.ust[u] = st;
        store_release(&A.ready[u], 1u);
      }
      commit_record(A, u, row, empty_record(SPEC_F_NAN));
    }
    __syncwarp();
    return;
  }
  const float m_lane = m;
  m = mw;
  const int am = (int)__ldcg(&R[cfirst].amax);
  // the softmax sum rescaled to the unit max (fixed lane order)
  const float Z = warp_sum(cm != 0x7fffffff ? zl * ex2((m_lane - m) * cfg.c) : 0.f);
  const float lnZ = logf(Z);
  if (cfg.type == UT_GREEDY) {
    if (lane == 0) {
      UnitRecord rec = empty_record(base_flags);
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
      commit_record(A, u, row, rec);
    }
    __syncwarp();
    return;
  }
  // unfiltered
  if (!has_q) {
    // bonus: merge the chunks' block races (scaled to the unit max), then
    // race the entries of the winning block
    Race a;
    race_init(a);
    for (int c = lane; c < NC; c += 32) {
      const float mc = __ldcg(&R[c].m);
      const float sc = mc > -INFINITY ? ex2((mc - m) * cfg.c) : 0.f;
      Race b;
      b.s1 = __ldcg(&R[c].s1);
      b.t1 = __ldcg(&R[c].t1);
      b.s2 = __ldcg(&R[c].s2);
      b.t2 = __ldcg(&R[c].t2);
      b.v1 = __ldcg(&R[c].v1);
      b.s1lo = 0.f;
      race_scale(b, sc);
      race_merge(a, b);
    }
    warp_race_merge(a);
    const Race l2 = race_in_block<kBF16>(A, row, pos, a.v1, m, cfg.c, 1.f, RW_BONUS, nullptr);
    if (lane == 0) {
      UnitRecord rec = empty_record(base_flags);
      const uint32_t y = l2.v1 < (uint32_t)A.V ? l2.v1 : (uint32_t)am;
      rec.y = (int32_t)y;
      rec.lp_y = (load_logit(A, kBF16, (size_t)u * A.V + y) - m) * cfg.invT - lnZ;
      if (draw_margin(a) || draw_margin(l2)) rec.draw_flags |= SPEC_F_MARGIN_DRAW;
      commit_record(A, u, row, rec);
    }
    __syncwarp();
    return;
  }
  // drafted: accept test, then publish the state for the B items
  if (lane == 0) {
    const AcceptInfo ai = accept_pre(A, row, pos, pr, false, am, m, cfg.c, Z);
    UnitState st;
    st.m = m;
    st.invZ = 1.0f / Z;
    st.lnZ = lnZ;
    st.accept = ai.accept ? 1 : 0;
    st.lp_x = ai.valid ? (ai.lx - m) * cfg.invT - lnZ : 0.f;
    st.flags = base_flags | (ai.valid ? 0u : SPEC_F_BAD_TOKEN) | (ai.margin ? SPEC_F_MARGIN_ACCEPT : 0u);
    st.invalid = 0;
    st.am = am;
    A.ust[u] = st;
    store_release(&A.ready[u], 1u);
  }
  __syncwarp();
}


// ---------------------------------------------------------------------------
// Small top-k, one warp.
// ---------------------------------------------------------------------------
constexpr int kCandCap = 256;              // candidates held for the sort path

// Scratch of one warp: its two stream buffers.
struct TopkScratch {
  uint16_t sg[kMaxNsmTopk];                // super-group max keys (16-bit), then qualifying super-group ids
  uint32_t hist[256];
  unsigned long long cand[kCandCap];
};
static_assert(sizeof(TopkScratch) <= 2 * kSlot, "top-k scratch exceeds a warp's stream buffers");

// The list phase reuses the super-group area.
struct ListArrays {
  uint32_t blk[kTopkSmall];
  float w[kTopkSmall];
  float wu[kTopkSmall];
};
static_assert(sizeof(ListArrays) <= sizeof(uint16_t) * kMaxNsmTopk, "list arrays exceed the super-group area");

__device__ __forceinline__ uint32_t k16(float v) { return okey(v) >> 16; }

// Smallest order key whose weight exp2((v - m) c) is positive (the weight is
// monotone in the key); every lane computes the same.
__device__ __forceinline__ uint32_t positive_key(float m, float c, uint32_t km) {
  uint32_t lo = 0u, hi = km;
  while (lo < hi) {
    const uint32_t mid = lo + ((hi - lo) >> 1);
    if (ex2((from_okey(mid) - m) * c) > 0.f) hi = mid;
    else lo = mid + 1u;
  }
  return lo;
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

// Calls fn(g, v) on every lane for the groups of 8 entries of the listed
// super-groups (4 super-groups per warp step, lane l on group 8 * id + (l & 7);
// g < 0 on lanes past the list).  Steps are loaded four at a time.
template <bool kBF16, typename F>
__device__ __forceinline__ void sweep_groups(const Args& A, size_t lrow, const uint16_t* ids, int n_sg, F fn) {
  const int lane = threadIdx.x & 31;
  for (int base = 0; base < n_sg; base += 16) {
    float v[4][8];
    int g[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int j = base + 4 * s + (lane >> 3);
      g[s] = j < n_sg ? (int)ids[j] * 8 + (lane & 7) : -1;
      if (g[s] >= 0) {
        load_group<kBF16>(A, lrow, g[s], true, v[s]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[s][i] = -INFINITY;
      }
    }
#pragma unroll
    for (int s = 0; s < 4; ++s)
      if (base + 4 * s < n_sg) fn(g[s], v[s]);
  }
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

// Bitonic sort, descending, of 32 * R keys held R per lane (element
// lane * R + r in register r).
template <int R>
__device__ __forceinline__ void warp_bitonic_desc(unsigned long long (&a)[R]) {
  const int lane = threadIdx.x & 31;
  constexpr int N = 32 * R;
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < R) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int r2 = r ^ stride;
          if (r2 > r) {
            const int i = lane * R + r;
            const bool desc = (i & size) == 0;
            const unsigned long long x = a[r], y = a[r2];
            const bool sw = desc ? (x < y) : (x > y);
            a[r] = sw ? y : x;
            a[r2] = sw ? x : y;
          }
        }
      } else {
        const int lx = stride / R;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int i = lane * R + r;
          const unsigned long long o = __shfl_xor_sync(kSettleFull, a[r], lx);
          const bool desc = (i & size) == 0;
          const bool lower = (i & stride) == 0;
          const bool keep_max = desc == lower;
          a[r] = keep_max ? (o > a[r] ? o : a[r]) : (o < a[r] ? o : a[r]);
        }
      }
    }
  }
}

// Sort cand[0..n) (n <= 32 R, kept keys > 0) in place, descending.
template <int R>
__device__ __forceinline__ void sort_cands(unsigned long long* cand, int n) {
  const int lane = threadIdx.x & 31;
  unsigned long long a[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = lane * R + r;
    a[r] = i < n ? cand[i] : 0ull;
  }
  warp_bitonic_desc<R>(a);
  __syncwarp();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = lane * R + r;
    if (i < n) cand[i] = a[r];
  }
  __syncwarp();
}

// Exact selection when more than kCandCap candidates pass the bound: the
// K-th largest candidate key by radix passes over the listed super-groups
// (8 bits at a time from the top), then the entries above it and the first
// ties in index order, K in all, into cand[].
template <bool kBF16>
__device__ __noinline__ void select_k_exact(const Args& A, TopkScratch& S, size_t lrow, int n_sg, uint32_t T32,
                                            int K) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0u, mask = 0u, need = (uint32_t)K;
  const int lowest = kBF16 ? 16 : 0;        // bf16 keys are fixed by their top 16 bits
  for (int shift = 24; shift >= lowest; shift -= 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) S.hist[8 * lane + i] = 0u;
    __syncwarp();
    sweep_groups<kBF16>(A, lrow, S.sg, n_sg, [&](int g, const float* v) {
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
    need -= before;
    prefix |= (uint32_t)(255 - min(b, 255)) << shift;
    mask |= 255u << shift;
    __syncwarp();
  }
  uint32_t tkey = prefix;
  if (kBF16) tkey = full_key<true>(prefix >> 16);
  // `need` ties at tkey (in index order) complete the K entries above it
  uint32_t n_out = 0, ties_seen = 0;
  sweep_groups<kBF16>(A, lrow, S.sg, n_sg, [&](int g, const float* v) {
    uint32_t gt = 0, eq = 0;
    uint32_t keys[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      keys[i] = okey(v[i]);
      const bool in = g >= 0 && g * 8 + i < A.V;
      gt |= (in && keys[i] > tkey) ? (1u << i) : 0u;
      eq |= (in && keys[i] == tkey) ? (1u << i) : 0u;
    }
    uint32_t te = 0;
    const uint32_t tbase = ties_seen + warp_excl_scan((uint32_t)__popc(eq), &te);
    ties_seen += te;
    // keep the ties of rank < need
    uint32_t keep = gt;
    uint32_t r = tbase;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((eq >> i) & 1u) {
        if (r < need) keep |= 1u << i;
        ++r;
      }
    uint32_t tk = 0;
    uint32_t pos = n_out + warp_excl_scan((uint32_t)__popc(keep), &tk);
    n_out += tk;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((keep >> i) & 1u) {
        if (pos < (uint32_t)kCandCap) S.cand[pos] = key64(keys[i], (uint32_t)(g * 8 + i));
        ++pos;
      }
  });
  __syncwarp();
}

// Settle a small top-k unit with one warp.
template <bool kBF16>
__device__ __noinline__ void topk_settle(const Args& A, TopkScratch& S, int u, int row, int pos, const RowCfg& cfg) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const bool has_q = pos < A.k;
  const int nsm = ceil_div(A.V, G::EA) * G::SPI;
  const size_t lrow = (size_t)u * A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const float c = cfg.c;
  // the accept test's operands are in flight while the list is built (lane 0)
  Pre pr;
  pr.x = -1;
  pr.valid = 0;
  pr.lx = 0.f;
  pr.qx = 0.f;
  if (lane == 0) pr = load_pre<kBF16>(A, u, row, pos);

  // 1. super-group maxima -> 16-bit keys; the unit max; NaN
  const float4* src = reinterpret_cast<const float4*>(A.smax + (size_t)u * A.NSM);
  float mf = -INFINITY;
  bool nan = false;
  for (int base = 0; base < nsm; base += 4 * 128) {
    float4 x[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int i = base + s * 128 + lane * 4;
      x[s] = i < nsm ? __ldcg(src + (i >> 2)) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int i = base + s * 128 + lane * 4;
      if (i >= nsm) continue;
      const float e[4] = {x[s].x, x[s].y, x[s].z, x[s].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        nan |= e[j] != e[j];
        mf = fmaxf(mf, e[j]);
        S.sg[i + j] = (uint16_t)k16(e[j]);
      }
    }
  }
  nan = __any_sync(kSettleFull, nan);
  const float m = warp_max_f(mf);
  if (nan || !(m > -INFINITY) || !(m < INFINITY)) {
    if (lane == 0) commit_record(A, u, row, empty_record(SPEC_F_NAN));
    __syncwarp();
    return;
  }
  const uint32_t km = okey(m);
  const uint32_t km16 = km >> 16;
  const uint32_t kpos = positive_key(m, c, km);
  const uint32_t kpos16 = kpos >> 16;
#pragma unroll
  for (int i = 0; i < 8; ++i) S.hist[8 * lane + i] = 0u;
  __syncwarp();

  // 2. tau16: the K-th largest positive super-group key, from a histogram of
  // distances to the unit max (the 255th bin lumps the rest)
  for (int s = lane; s < nsm; s += 32) {
    const uint32_t kk = S.sg[s];
    if (kk >= kpos16) atomicAdd(&S.hist[min(km16 - kk, 255u)], 1u);
  }
  __syncwarp();
  uint32_t before = 0;
  const int b = warp_select_bin(S.hist, (uint32_t)cfg.K, &before);
  uint32_t tau16;
  if (b == 256) {
    tau16 = kpos16;                          // fewer than K positive super-groups: all qualify
  } else if (b < 255) {
    tau16 = km16 - (uint32_t)b;
  } else {
    // the K-th lies in the lumped tail: bisect the 16-bit key space
    uint32_t lo = kpos16, hi = km16;           // count(key >= lo) >= K holds
    while (lo < hi) {
      const uint32_t mid = lo + ((hi - lo + 1u) >> 1);
      uint32_t cnt = 0;
      for (int s = lane; s < nsm; s += 32) cnt += S.sg[s] >= mid ? 1u : 0u;
      cnt = __reduce_add_sync(kSettleFull, cnt);
      if (cnt >= (uint32_t)cfg.K) lo = mid;
      else hi = mid - 1u;
    }
    tau16 = lo;
  }
  tau16 = max(tau16, kpos16);
  const uint32_t T32 = max(tau16 << 16, kpos);

  // 3. the qualifying super-groups, ids in increasing order (in place)
  int n_sg = 0;
  for (int base = 0; base < nsm; base += 32) {
    const int s = base + lane;
    const bool q = s < nsm && (uint32_t)S.sg[s] >= tau16;
    const unsigned ball = __ballot_sync(kSettleFull, q);
    __syncwarp();
    if (q) S.sg[n_sg + __popc(ball & ((1u << lane) - 1u))] = (uint16_t)s;
    n_sg += __popc(ball);
    __syncwarp();
  }

  // 4. candidates: entries with key >= T32 of those super-groups
  uint32_t n_c = 0;
  sweep_groups<kBF16>(A, lrow, S.sg, n_sg, [&](int g, const float* v) {
    uint32_t hit = 0;
    uint32_t keys[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      keys[i] = okey(v[i]);
      hit |= (g >= 0 && g * 8 + i < A.V && keys[i] >= T32) ? (1u << i) : 0u;
    }
    uint32_t tot = 0;
    uint32_t p = n_c + warp_excl_scan((uint32_t)__popc(hit), &tot);
    n_c += tot;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((hit >> i) & 1u) {
        if (p < (uint32_t)kCandCap) S.cand[p] = key64(keys[i], (uint32_t)(g * 8 + i));
        ++p;
      }
  });
  __syncwarp();
  int n_k;
  if (n_c <= (uint32_t)kCandCap) {
    if (n_c <= 128) sort_cands<4>(S.cand, (int)n_c);
    else sort_cands<8>(S.cand, (int)n_c);
    n_k = min((int)n_c, cfg.K);
  } else {
    select_k_exact<kBF16>(A, S, lrow, n_sg, T32, cfg.K);
    n_k = cfg.K;
    sort_cands<4>(S.cand, n_k);
  }

  // 5. the list: lane l holds entries 4l..4l+3 of the first n_k
  ListArrays& L = *reinterpret_cast<ListArrays*>(S.sg);
  uint32_t idx[4];
  float val[4], e[4], qv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = 4 * lane + j;
    const unsigned long long key = i < n_k ? S.cand[i] : 0ull;
    idx[j] = key64_idx(key);
    val[j] = from_okey((uint32_t)(key >> 32));
    qv[j] = 0.f;
    if (has_q && i < n_k) qv[j] = A.q[qrow + idx[j]];   // in flight while the list is settled
    e[j] = i < n_k ? ex2((val[j] - m) * c) : 0.f;
  }
  const int am = (int)__shfl_sync(kSettleFull, idx[0], 0);
  pr.x = __shfl_sync(kSettleFull, pr.x, 0);
  pr.valid = __shfl_sync(kSettleFull, pr.valid, 0);
  pr.lx = __shfl_sync(kSettleFull, pr.lx, 0);
  pr.qx = __shfl_sync(kSettleFull, pr.qx, 0);
  // inclusive prefix sums in the total order (fixed order)
  float cum[4];
  cum[0] = e[0];
  cum[1] = cum[0] + e[1];
  cum[2] = cum[1] + e[2];
  cum[3] = cum[2] + e[3];
  float inc = cum[3];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kSettleFull, inc, o);
    if (lane >= o) inc += y;
  }
  const float off = inc - cum[3];
#pragma unroll
  for (int j = 0; j < 4; ++j) cum[j] += off;
  auto cum_at = [&](int i) {      // cum of entry i (every lane)
    const int j = i & 3;
    const float x = j == 0 ? cum[0] : (j == 1 ? cum[1] : (j == 2 ? cum[2] : cum[3]));
    return __shfl_sync(kSettleFull, x, i >> 2);
  };
  const float Zk = cum_at(n_k - 1);
  uint32_t flags = cfg.bad_param ? SPEC_F_BAD_PARAM : 0u;
  int n_s = n_k;
  if (cfg.P < 1.0f) {
    const float target = cfg.P * Zk;
    int first = 4;
#pragma unroll
    for (int j = 3; j >= 0; --j)
      if (4 * lane + j < n_k && cum[j] >= target) first = j;
    const unsigned ball = __ballot_sync(kSettleFull, first < 4);
    if (ball) {
      const int sl = __ffs(ball) - 1;
      n_s = 4 * sl + __shfl_sync(kSettleFull, first, sl) + 1;
    }
    const float at = cum_at(n_s - 1) / Zk;
    const float bef = n_s >= 2 ? cum_at(n_s - 2) / Zk : 0.f;
    if (fabsf(at - cfg.P) < kMargin || fabsf(cfg.P - bef) < kMargin) flags |= SPEC_F_MARGIN_TOPP;
  }
  const float Zs = cum_at(n_s - 1);
  const float invZ = 1.0f / Zs;
  const float lnZ = logf(Zs);
  float p[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) p[j] = 4 * lane + j < n_s ? e[j] * invZ : 0.f;
  float alpha_v = 0.f;
  AcceptInfo ai;
  ai.valid = true;
  ai.accept = false;
  ai.margin = false;
  ai.lx = 0.f;
  bool need_race = !has_q;
  if (has_q) {
    float a = 0.f, ex = -1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (4 * lane + j < n_s) {
        a += fminf(p[j], qv[j]);
        if (idx[j] == (uint32_t)pr.x) ex = e[j];
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
    const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)pos, (uint32_t)row, 0u), A.key0, A.key1);
    const float uu = uniform_of(w.x);
    const float d = fmaf(uu, ai.qx, -ai.px);
    ai.accept = d < 0.0f;
    ai.margin = (ai.px > 0.0f && ai.px < 1.0f && fabsf(d) < kMargin);
    need_race = !ai.accept;
  }
  // 6. the draw: the two-level race over the kept entries (blocks by index)
  uint32_t draw_flags = 0;
  uint32_t y = 0xffffffffu;
  if (need_race) {
    for (int attempt = 0; attempt < 2; ++attempt) {
      const bool use_p = attempt == 1;          // empty residual: draw from p
      float w[4], tq[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool mine = 4 * lane + j < n_s;
        w[j] = mine ? ((has_q && !use_p) ? fmaxf(p[j] - qv[j], 0.f) : p[j]) : 0.f;
        tq[j] = (mine && has_q && !use_p) ? 2.0f * qv[j] : 0.f;
        if (4 * lane + j < kTopkSmall) {
          L.blk[4 * lane + j] = idx[j] / kRaceBlock;
          L.w[4 * lane + j] = w[j];
          L.wu[4 * lane + j] = w[j] + tq[j];
        }
      }
      __syncwarp();
      // level 1: the first kept entry of each block races for its block, with
      // the block's weights summed in list order
      Race r1;
      race_init(r1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 4 * lane + j;
        if (!(w[j] > 0.f)) continue;
        const uint32_t bb = idx[j] / kRaceBlock;
        bool rep = true;
        float W = 0.f, U = 0.f;
        for (int t = 0; t < n_s; ++t) {
          if (L.blk[t] == bb && L.w[t] > 0.f) {
            if (t < i) rep = false;
            W += L.w[t];
            U += L.wu[t];
          }
        }
        if (rep) race_consider(r1, W, U - W, bb, block_word(A, row, pos, bb));
      }
      warp_race_merge(r1);
      __syncwarp();
      if (r1.s1 < 0.f) {
        draw_flags |= SPEC_F_RESIDUAL_EMPTY;
        continue;
      }
      // level 2: the entries of the winning block
      Race r2;
      race_init(r2);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (w[j] > 0.f && idx[j] / kRaceBlock == r1.v1)
          race_consider(r2, w[j], tq[j], idx[j], race_word(A, row, pos, idx[j]));
      warp_race_merge(r2);
      y = r2.v1;
      if (draw_margin(r1) || draw_margin(r2)) draw_flags |= SPEC_F_MARGIN_DRAW;
      break;
    }
  }
  // the logit of the drawn entry, from the list
  float vy = m;
  {
    float vv = 0.f;
    bool own = false;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (4 * lane + j < n_k && idx[j] == y) {
        vv = val[j];
        own = true;
      }
    const unsigned ob = __ballot_sync(kSettleFull, own);
    if (ob) vy = __shfl_sync(kSettleFull, vv, __ffs(ob) - 1);
  }
  if (lane == 0) {
    UnitRecord rec = empty_record(flags);
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
    commit_record(A, u, row, rec);
  }
  __syncwarp();
}

}  // namespace specv
