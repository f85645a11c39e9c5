// spec_verify, unit kernel (sm_103a): one CTA settles one (row, position)
// unit from the stats kernel's records, all units in parallel.
//
//   greedy and unfiltered units (one warp): merge the chunk records in chunk
//     order -- max, first argmax, the softmax sum rescaled to the unit max;
//     greedy units and unfiltered bonus positions are settled at once (the
//     bonus draw merges the chunks' level-1 block races and races the winning
//     block's entries); a drafted unfiltered unit takes its accept test,
//     publishes its state and lists itself for the B pass.
//   small top-k units (the CTA): every top-K entry lies in a 64-entry
//     super-group whose maximum is among the K largest super-group maxima, so
//     the K-th largest maximum bounds the candidates; they are gathered from
//     L2, sorted exactly, and top-p, the accept test, alpha and the draw run
//     on the list.
//   general units (the CTA): passes over the row (spec_general.cuh).
//
// The last settled unit of a row resolves the accept chain and writes the
// row's outputs.  The kernel starts while the stats kernel finishes and waits
// for its records (programmatic dependent launch).
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "spec_general.cuh"
#include "spec_host.h"
#include "spec_verify_common.cuh"

namespace specv {

constexpr int kMergeCap = 4096;            // finaliser buffer: candidates + super-group maxima
constexpr int kGPC = 1024;                 // qualifying super-groups held
constexpr unsigned kFull = 0xffffffffu;
static_assert(kMaxNsmTopk * 4 <= kMergeCap / 2 * 8, "super-group maxima exceed the buffer");

// The draft token of the unit and its logit and q, read before the stats
// kernel's records are awaited (they are inputs).
struct Pre {
  int x, valid;
  float lx, qx;
};

struct alignas(16) UnitShm {
  GenShm g;
  Pre pre;
  uint32_t cand_count;
  float gmax[kGPC];
  float list_e[kTopkSmall];
  float list_cum[kTopkSmall];
  float list_w[kTopkSmall];
  float list_u[kTopkSmall];
  unsigned long long cand[kMergeCap];
};

// Bitonic sort of s[0..n) in descending order (n a power of two), one CTA.
__device__ void bitonic_desc(unsigned long long* s, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (n >> 1); i += kThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long a = s[lo], b = s[hi];
        if ((a < b) == desc) {
          s[lo] = b;
          s[hi] = a;
        }
      }
      __syncthreads();
    }
  }
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
__device__ __noinline__ void fin_stats(const Args& A, int u, int row, int pos, const RowCfg& cfg, const Pre& pr) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const bool has_q = pos < A.k;
  const int NC = ceil_div(A.V, G::EA);
  const ChunkRec* R = A.crec + (size_t)u * A.NCA;
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
  nan = __any_sync(kFull, nan);
  const float mw = warp_max_f(m);
  const int cfirst = (int)warp_min_u32((m == mw && cm != 0x7fffffff) ? (uint32_t)cm : 0xffffffffu);
  const bool invalid = nan || !(mw > -INFINITY) || !(mw < INFINITY);
  const uint32_t base_flags = cfg.bad_param ? SPEC_F_BAD_PARAM : 0u;
  if (invalid) {
    if (lane == 0) {
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
    A.dlist[atomicAdd(&A.ws->n_dense, 1u)] = (uint32_t)u;
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Small top-k: the sorted candidate list in S.cand[0..n_k) (the first n_k
// entries of the total order) settles the unit.  CTA-wide; n_k <= 128.
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ __noinline__ void list_unit(const Args& A, UnitShm& S, int u, int row, int pos, const RowCfg& cfg, float m,
                          int am, int n_k) {
  const bool has_q = pos < A.k;
  const size_t lrow = (size_t)u * A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const int t = threadIdx.x;
  float e = 0.f;
  uint32_t idx = 0;
  float q_pre = 0.f;
  if (t < n_k) {
    const unsigned long long key = S.cand[t];
    idx = key64_idx(key);
    if (has_q) q_pre = A.q[qrow + idx];   // in flight while the list is settled
    e = ex2((from_okey((uint32_t)(key >> 32)) - m) * cfg.c);
    S.list_e[t] = e;
  }
  {
    // inclusive prefix sum in the total order (fixed order)
    float inc = e;
    const int lane = t & 31, w = t >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) S.g.wred[w] = inc;
    __syncthreads();
    float off = 0.f;
    for (int i = 0; i < w; ++i) off += S.g.wred[i];
    if (t < n_k) S.list_cum[t] = off + inc;
    __syncthreads();
  }
  const float Zk = S.list_cum[n_k - 1];
  uint32_t flags = cfg.bad_param ? SPEC_F_BAD_PARAM : 0u;
  int n_s = n_k;
  if (cfg.P < 1.0f) {
    const float target = cfg.P * Zk;
    if (t == 0) S.g.bci[4] = n_k - 1;
    __syncthreads();
    const bool hit = t < n_k && S.list_cum[t] >= target;
    const unsigned ball = __ballot_sync(0xffffffffu, hit);
    if ((t & 31) == 0 && ball) atomicMin(&S.g.bci[4], (t & ~31) + __ffs(ball) - 1);
    __syncthreads();
    n_s = S.g.bci[4] + 1;
    const float at = S.list_cum[n_s - 1] / Zk;
    const float before = n_s >= 2 ? S.list_cum[n_s - 2] / Zk : 0.f;
    if (fabsf(at - cfg.P) < kMargin || fabsf(cfg.P - before) < kMargin) flags |= SPEC_F_MARGIN_TOPP;
  }
  const float Zs = S.list_cum[n_s - 1];
  const float invZ = 1.0f / Zs;
  const float lnZ = logf(Zs);
  const bool mine = t < n_s;
  const float p = mine ? e * invZ : 0.f;
  const float qv = mine ? q_pre : 0.f;
  int x = -1;
  if (has_q) {
    x = S.pre.x;
    if (t == 0) S.g.bci[5] = -1;
    __syncthreads();
    if (mine && idx == (uint32_t)x) S.g.bci[5] = t;
    __syncthreads();
  }
  const float alpha_v = has_q ? block_sum(S.g, mine ? fminf(p, qv) : 0.f) : 0.f;
  bool need_race = !has_q;
  AcceptInfo ai;
  ai.valid = true;
  ai.accept = false;
  ai.margin = false;
  ai.lx = 0.f;
  if (has_q) {
    const int xi = S.g.bci[5];
    ai.x = x;
    ai.valid = x >= 0 && x < A.V;
    ai.px = xi >= 0 ? S.list_e[xi] / Zs : 0.f;
    ai.qx = S.pre.qx;
    ai.lx = S.pre.lx;
    const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)pos, (uint32_t)row, 0u), A.key0, A.key1);
    const float uu = uniform_of(w.x);
    const float d = fmaf(uu, ai.qx, -ai.px);
    ai.accept = d < 0.0f;
    ai.margin = (ai.px > 0.0f && ai.px < 1.0f && fabsf(d) < kMargin);
    need_race = !ai.accept;
  }
  // the draw: the two-level race over the kept entries (blocks by index)
  uint32_t draw_flags = 0;
  uint32_t y = 0xffffffffu;
  if (need_race) {
    for (int attempt = 0; attempt < 2; ++attempt) {
      const bool use_p = attempt == 1;          // empty residual: draw from p
      const float w = (has_q && !use_p) ? fmaxf(p - qv, 0.f) : p;
      const float tq = (has_q && !use_p) ? 2.0f * qv : 0.f;
      if (t < kTopkSmall) {
        S.list_w[t] = mine ? w : 0.f;
        S.list_u[t] = mine ? w + tq : 0.f;
      }
      __syncthreads();
      // level 1: the first kept entry of each block races for its block, with
      // the block's weights summed in list order
      Race r1;
      race_init(r1);
      if (mine && w > 0.f) {
        const uint32_t b = idx / kRaceBlock;
        bool rep = true;
        float W = 0.f, U = 0.f;
        for (int j = 0; j < n_s; ++j) {
          const uint32_t bj = key64_idx(S.cand[j]) / kRaceBlock;
          if (bj == b && S.list_w[j] > 0.f) {
            if (j < t) rep = false;
            W += S.list_w[j];
            U += S.list_u[j];
          }
        }
        if (rep) race_consider(r1, W, U - W, b, block_word(A, row, pos, b));
      }
      const Race g1 = block_race(S.g, r1);
      if (g1.s1 < 0.f) {
        draw_flags |= SPEC_F_RESIDUAL_EMPTY;
        continue;
      }
      // level 2: the entries of the winning block
      Race r2;
      race_init(r2);
      if (mine && w > 0.f && idx / kRaceBlock == g1.v1) race_consider(r2, w, tq, idx, race_word(A, row, pos, idx));
      const Race g2 = block_race(S.g, r2);
      y = g2.v1;
      if (draw_margin(g1) || draw_margin(g2)) draw_flags |= SPEC_F_MARGIN_DRAW;
      break;
    }
  }
  if (t == 0) {
    UnitRecord rec = empty_record(flags);
    if (has_q) {
      if (!ai.valid) rec.flags |= SPEC_F_BAD_TOKEN;
      if (ai.margin) rec.flags |= SPEC_F_MARGIN_ACCEPT;
      rec.accept = ai.accept ? 1 : 0;
      rec.lp_x = ai.valid ? (ai.lx - m) * cfg.invT - lnZ : 0.f;
      rec.alpha = alpha_v;
    }
    if (need_race) {
      const uint32_t yy = y < (uint32_t)A.V ? y : (uint32_t)am;
      rec.y = (int32_t)yy;
      rec.lp_y = (load_logit(A, kBF16, lrow + yy) - m) * cfg.invT - lnZ;
      rec.draw_flags = draw_flags;
    }
    commit_record(A, u, row, rec);
  }
  __syncthreads();
}


// Small top-k finaliser: every top-K entry lies in a 64-entry super-group
// whose maximum is among the K largest super-group maxima, so the K-th
// largest super-group maximum tau bounds the candidates: the entries >= tau
// of the super-groups whose maximum reaches tau (at least K of them, and at
// most 64 per such super-group).  They are gathered from L2, sorted exactly,
// and the first K settle the unit.
template <bool kBF16>
__device__ __noinline__ void finalize_topk(const Args& A, UnitShm& S, int u, int row, int pos, const RowCfg& cfg) {
  const int nsm = ceil_div(A.V, Geo<kBF16>::EA) * Geo<kBF16>::SPI;
  const float* src = A.smax + (size_t)u * A.NSM;
  float* sm = reinterpret_cast<float*>(S.cand + kMergeCap / 2);    // second half of the buffer
  unsigned long long* cand = S.cand;                               // first half
  const int G = (A.V + 7) / 8;
  const size_t lrow = (size_t)u * A.V;
  // maxima into shared memory; the unit max; NaN
  unsigned long long best = 0;
  bool nan_seen = false;
  for (int base = threadIdx.x; base < nsm; base += 8 * kThreads) {
    float xs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = base + i * kThreads;
      xs[i] = s < nsm ? __ldcg(src + s) : -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = base + i * kThreads;
      if (s >= nsm) continue;
      sm[s] = xs[i];
      if (xs[i] != xs[i]) nan_seen = true;
      else {
        const unsigned long long kk = ((unsigned long long)okey(xs[i]) << 32) | (0xffffffffu - (uint32_t)s);
        best = kk > best ? kk : best;
      }
    }
  }
  if (nan_seen) best = ~0ull;
  best = block_max_u64(S.g, best);
  const float m = from_okey((uint32_t)(best >> 32));
  if (best == ~0ull || best == 0 || !(m > -INFINITY) || !(m < INFINITY)) {
    if (threadIdx.x == 0) commit_record(A, u, row, empty_record(SPEC_F_NAN));
    __syncthreads();
    return;
  }
  const uint32_t km = kf<kBF16>(m);
  uint32_t tau = 0u;
  if (cfg.K < nsm) {
    unsigned long long need = (unsigned long long)cfg.K;
    auto each = [&](auto fn) {
      for (int s = threadIdx.x; s < nsm; s += kThreads) fn(km - kf<kBF16>(sm[s]));
    };
    tau = km - kth_distance(S.g, each, need, kBF16 ? 0 : 16, kBF16 ? 16 : 32);
  }
  // list the qualifying super-groups, then gather their entries >= tau
  int* sg = reinterpret_cast<int*>(S.gmax);   // up to kGPC super-group ids
  if (threadIdx.x == 0) {
    S.cand_count = 0;
    S.g.bci[6] = 0;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  for (int base = 0; base < nsm; base += kThreads) {
    const int s = base + threadIdx.x;
    const bool ok = s < nsm && kf<kBF16>(sm[s]) >= tau;
    const unsigned b = __ballot_sync(0xffffffffu, ok);
    int off = 0;
    if (lane == 0 && b) off = atomicAdd(&S.g.bci[6], __popc(b));
    off = __shfl_sync(0xffffffffu, off, 0);
    if (ok) {
      const int slot = off + __popc(b & ((1u << lane) - 1u));
      if (slot < kGPC) sg[slot] = s;
    }
  }
  __syncthreads();
  const int nsg = S.g.bci[6];
  bool ovf = nsg > kGPC;
  if (!ovf) {
    for (int base = 0; base < nsg * 8; base += kThreads) {
      const int e = base + threadIdx.x;
      const int g = e < nsg * 8 ? sg[e >> 3] * 8 + (e & 7) : G;   // super-group s covers groups 8s..8s+7
      float v[8];
      if (g < G) load_group<kBF16>(A, lrow, g, true, v);
      int ups = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) ups += (g < G && g * 8 + j < A.V && kf<kBF16>(v[j]) >= tau) ? 1 : 0;
      // one shared atomic per warp: an exclusive scan of the lanes' counts
      int inc = ups;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      uint32_t off = 0;
      if (lane == 31 && inc) off = atomicAdd(&S.cand_count, (uint32_t)inc);
      off = __shfl_sync(0xffffffffu, off, 31) + (uint32_t)(inc - ups);
      if (ups) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (g * 8 + j < A.V && kf<kBF16>(v[j]) >= tau) {
            if (off < (uint32_t)(kMergeCap / 2)) cand[off] = key64(okey(v[j]), (uint32_t)(g * 8 + j));
            ++off;
          }
        }
      }
    }
  }
  __syncthreads();
  const uint32_t count = S.cand_count;
  ovf = ovf || count > (uint32_t)(kMergeCap / 2);
  if (ovf) {
    unit_general<kBF16>(A, S.g, u, row, pos, cfg);
    return;
  }
  int n = 1;
  while (n < (int)count) n <<= 1;
  for (int i = (int)count + threadIdx.x; i < n; i += kThreads) cand[i] = 0ull;
  __syncthreads();
  bitonic_desc(cand, n);
  const int am = (int)key64_idx(cand[0]);
  list_unit<kBF16>(A, S, u, row, pos, cfg, m, am, min((int)count, cfg.K));
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads) unit_kernel(const Args A) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  UnitShm& S = *reinterpret_cast<UnitShm*>(smem_raw);
  const int u = blockIdx.x;
  const int row = u / (A.k + 1), pos = u - row * (A.k + 1);
  const RowCfg cfg = classify(A.params[row], A.V);
  // the B pass may be scheduled now; it waits for this grid's results
  pdl_trigger();
  // the draft token, its logit and q are inputs: read them before waiting
  if (threadIdx.x == 0) {
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
    S.pre = pr;
  }
  // the stats kernel's records
  pdl_wait();
  __syncthreads();
  if (cfg.type == UT_GENERAL) {
    unit_general<kBF16>(A, S.g, u, row, pos, cfg);
  } else if (cfg.type == UT_TOPK) {
    finalize_topk<kBF16>(A, S, u, row, pos, cfg);
  } else if (threadIdx.x < 32) {
    fin_stats<kBF16>(A, u, row, pos, cfg, S.pre);
  }
}

template <bool kBF16>
int launch_units(const Args& A, cudaStream_t stream) {
  static std::mutex mu;
  static bool ready[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
      if (cudaFuncSetAttribute(unit_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sizeof(UnitShm)) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_E_CUDA;
      }
      ready[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)A.U);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(UnitShm);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, unit_kernel<kBF16>, A) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  return SPEC_OK;
}

template int launch_units<true>(const Args&, cudaStream_t);
template int launch_units<false>(const Args&, cudaStream_t);

}  // namespace specv
