// spec_verify, general path: rows whose kept set needs a global threshold
// search (top-p without a small top-k, or a top-k above the candidate-list
// limit).  One settle group (256 threads) settles one (row, position) unit
// in passes over its logit row (the first from HBM, later ones mostly from L2): max and argmax, an
// exact rank select for top-k, a fixed-point mass histogram refined to the
// exact top-p crossing key, the tie rank by index, Z over the kept set, the
// accept test, alpha, and the two-level exponential race for the draw.  The
// settle groups take these units before any other.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_common.cuh"

namespace specv {

// Shared memory of a settle group on the general path.
struct alignas(16) GenShm {
  uint32_t hist[2][256];
  uint32_t mlo[2][256];
  uint32_t mhi[2][256];
  unsigned long long total[256];
  unsigned long long bc64[8];
  float wred[kWarps * 8];
  float bcf[8];
  int bci[16];
  int ring_fail;
};

// One pass over a unit's row by the group: fn(g, v) for every group g of 8
// entries (thread t takes groups t, t + kThreads, ...), kGenBatch groups of
// a thread loaded before any is used, so that the pass is bound by
// bandwidth rather than by one load's latency per group.  Groups past the
// row hold -inf (the callers check g * 8 + i < V as well).
constexpr int kGenBatch = 4;
template <bool kBF16, typename F>
__device__ __forceinline__ void gsweep(const Args& A, size_t lrow, int G, F fn) {
  for (int g0 = ctid(); g0 < G; g0 += kThreads * kGenBatch) {
    float v[kGenBatch][8];
#pragma unroll
    for (int b = 0; b < kGenBatch; ++b) {
      const int g = g0 + b * kThreads;
      if (g < G) {
        load_group<kBF16>(A, lrow, g, true, v[b]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[b][i] = -INFINITY;
      }
    }
#pragma unroll
    for (int b = 0; b < kGenBatch; ++b) {
      const int g = g0 + b * kThreads;
      if (g < G) fn(g, v[b]);
    }
  }
}

// The group's ring of shared-memory chunks: a pass over a row streams it
// through kGRing slots of kGSlot bytes by bulk copies (several chunks in
// flight), so that a pass is bound by the SM's bandwidth rather than by one
// load's latency per group.
constexpr int kGRing = 5;
constexpr int kGSlot = 32768;
struct GenRing {
  unsigned char* buf;          // kGRing slots of kGSlot bytes
  unsigned long long* bar;     // one mbarrier per slot
  int* fail;                   // shared: set when a thread's chunk wait gave up
  uint32_t seq;                // chunks taken so far (every thread keeps the same count)
  bool ok;                     // false once a chunk's wait gave up (the same in every thread)
};

// Entries of a chunk: logits only, or logits and q (a multiple of 256, so
// that a warp's 32 groups of a round are one race block).
template <bool kBF16>
__device__ __forceinline__ int chunk_entries(bool with_q) {
  return with_q ? (kGSlot / ((kBF16 ? 2 : 4) + 4)) / kRaceBlock * kRaceBlock : kGSlot / (kBF16 ? 2 : 4);
}

// One pass over a unit's row (and its q row with with_q), through the ring:
// fn(g, v, qv) for every group g of 8 entries, in rounds in which thread t
// takes group t of each 256 (every thread calls fn in every round, so fn may
// use warp collectives; groups past the row get -inf logits and zero q, and
// the callers check g * 8 + i < V per entry).  Needs 16-byte aligned rows
// (vec_logits, and vec_q with q).
template <bool kBF16, typename F>
__device__ __forceinline__ void csweep(const Args& A, GenRing& R, size_t lrow, size_t qrow, bool with_q, F fn) {
  constexpr int es = kBF16 ? 2 : 4;
  const int EC = chunk_entries<kBF16>(with_q);
  const int nch = (A.V + EC - 1) / EC;
  const uint32_t base = R.seq;
  const unsigned char* lg = reinterpret_cast<const unsigned char*>(A.logits);
  auto issue = [&](int c) {
    const uint32_t sq = base + (uint32_t)c;
    const int slot = (int)(sq % kGRing);
    const int e0 = c * EC, n = min(EC, A.V - e0);
    const uint32_t bl = (uint32_t)(n * es), bq = with_q ? (uint32_t)(n * 4) : 0u;
    unsigned char* dst = R.buf + (size_t)slot * kGSlot;
    fence_proxy_async();
    mbar_arrive_expect_tx(&R.bar[slot], bl + bq);
    bulk_g2s(dst, lg + (lrow + (size_t)e0) * es, bl, &R.bar[slot]);
    if (bq) bulk_g2s(dst + (size_t)EC * es, A.q + qrow + e0, bq, &R.bar[slot]);
  };
  if (ctid() == 0)
    for (int c = 0; c < min(nch, kGRing); ++c) issue(c);
  const int GC = EC / 8;   // groups per chunk
  for (int c = 0; c < nch; ++c) {
    const uint32_t sq = base + (uint32_t)c;
    const int slot = (int)(sq % kGRing);
    const uint32_t par = (sq / kGRing) & 1u;
    long long spins = 0;
    bool got = R.ok;
    while (got && !mbar_try_wait(&R.bar[slot], par)) {
      if (++spins > kSpinLimit) {
        atomicOr(&cur(A).error, (uint32_t)ERR_COPY_WAIT);
        *R.fail = 1;
        got = false;
      }
      if (spins > 64) __nanosleep(32);
    }
    const unsigned char* src = R.buf + (size_t)slot * kGSlot;
    const float* qsrc = reinterpret_cast<const float*>(src + (size_t)EC * es);
    const int n = min(EC, A.V - c * EC);
    const int ng = (n + 7) / 8;
    for (int r0 = 0; r0 < ng; r0 += kThreads) {
      const int lgi = r0 + ctid();
      const int g = lgi < ng ? c * GC + lgi : (1 << 27);   // past the row: g * 8 >= V
      float v[8], qv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[i] = -INFINITY;
        qv[i] = 0.f;
      }
      if (lgi < ng && got) {
        if (kBF16) {
          const uint4 w = *reinterpret_cast<const uint4*>(src + (size_t)lgi * 16);
          v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
          v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
        } else {
          const float4 a = *reinterpret_cast<const float4*>(src + (size_t)lgi * 32);
          const float4 b = *reinterpret_cast<const float4*>(src + (size_t)lgi * 32 + 16);
          v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
        if (with_q) {
          const float4 a = *reinterpret_cast<const float4*>(qsrc + (size_t)lgi * 8);
          const float4 b = *reinterpret_cast<const float4*>(qsrc + (size_t)lgi * 8 + 4);
          qv[0] = a.x; qv[1] = a.y; qv[2] = a.z; qv[3] = a.w; qv[4] = b.x; qv[5] = b.y; qv[6] = b.z; qv[7] = b.w;
        }
        // entries past the row in its last group
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (g * 8 + i >= A.V) {
            v[i] = -INFINITY;
            qv[i] = 0.f;
          }
      }
      fn(g, v, qv);
    }
    csync();   // every thread is done with the slot (and sees a failed wait)
    R.ok = R.ok && *R.fail == 0;
    if (ctid() == 0 && c + kGRing < nch && R.ok) issue(c + kGRing);
  }
  R.seq = base + (uint32_t)nch;
}

// A pass over the row: through the ring when the rows allow bulk copies,
// else with batched plain loads.
template <bool kBF16, typename F>
__device__ __forceinline__ void row_pass(const Args& A, GenRing& R, size_t lrow, F fn) {
  if (A.vec_logits && R.ok) {
    csweep<kBF16>(A, R, lrow, 0, false, [&](int g, const float* v, const float*) { fn(g, v); });
  } else {
    gsweep<kBF16>(A, lrow, (A.V + 7) / 8, fn);
  }
}

// ---------------------------------------------------------------------------
// Block reductions (fixed combination order, so results are reproducible).
// Each returns its result in every thread.
// ---------------------------------------------------------------------------
__device__ float block_sum(GenShm& S, float a) {
  a = warp_sum(a);
  const int w = ctid() >> 5, l = ctid() & 31;
  if (l == 0) S.wred[w] = a;
  csync();
  if (ctid() == 0) {
    float x = 0.f;
    for (int i = 0; i < kWarps; ++i) x += S.wred[i];
    S.bcf[7] = x;
  }
  csync();
  const float r = S.bcf[7];
  csync();
  return r;
}

// Exclusive prefix sum of x over the CTA in thread order; *total = the sum.
__device__ int block_exclusive_scan(GenShm& S, int x, int* total) {
  const int w = ctid() >> 5, l = ctid() & 31;
  int inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (l >= o) inc += y;
  }
  int* ws = S.bci;   // kWarps <= 16 entries
  if (l == 31) ws[w] = inc;
  csync();
  int off = 0, tot = 0;
  for (int i = 0; i < kWarps; ++i) {
    if (i < w) off += ws[i];
    tot += ws[i];
  }
  csync();
  *total = tot;
  return off + inc - x;
}

__device__ unsigned long long block_max_u64(GenShm& S, unsigned long long v) {
  v = warp_max_u64(v);
  const int w = ctid() >> 5, l = ctid() & 31;
  unsigned long long* buf = reinterpret_cast<unsigned long long*>(S.wred);
  if (l == 0) buf[w] = v;
  csync();
  if (ctid() == 0) {
    unsigned long long x = 0;
    for (int i = 0; i < kWarps; ++i) x = buf[i] > x ? buf[i] : x;
    S.bc64[7] = x;
  }
  csync();
  const unsigned long long r = S.bc64[7];
  csync();
  return r;
}

__device__ unsigned long long block_sum_u64(GenShm& S, unsigned long long v) {
  v = warp_sum_u64(v);
  const int w = ctid() >> 5, l = ctid() & 31;
  unsigned long long* buf = reinterpret_cast<unsigned long long*>(S.wred);
  if (l == 0) buf[w] = v;
  csync();
  if (ctid() == 0) {
    unsigned long long x = 0;
    for (int i = 0; i < kWarps; ++i) x += buf[i];
    S.bc64[7] = x;
  }
  csync();
  const unsigned long long r = S.bc64[7];
  csync();
  return r;
}

__device__ uint2 block_minmax_u32(GenShm& S, uint32_t mn, uint32_t mx) {
  uint32_t a = ~mn, b = mx;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  uint32_t* wb = reinterpret_cast<uint32_t*>(S.wred);
  if ((ctid() & 31) == 0) {
    wb[2 * (ctid() >> 5)] = a;
    wb[2 * (ctid() >> 5) + 1] = b;
  }
  csync();
  if (ctid() == 0) {
    uint32_t aa = 0, bb = 0;
    for (int i = 0; i < kWarps; ++i) {
      aa = max(aa, wb[2 * i]);
      bb = max(bb, wb[2 * i + 1]);
    }
    S.bci[12] = (int)~aa;
    S.bci[13] = (int)bb;
  }
  csync();
  const uint2 r = make_uint2((uint32_t)S.bci[12], (uint32_t)S.bci[13]);
  csync();
  return r;
}

__device__ Race block_race(GenShm& S, Race r) {
  warp_race_merge(r);
  const int w = ctid() >> 5, l = ctid() & 31;
  float* f = S.wred;
  if (l == 0) {
    f[w * 5 + 0] = r.s1;
    f[w * 5 + 1] = r.t1;
    f[w * 5 + 2] = r.s2;
    f[w * 5 + 3] = r.t2;
    f[w * 5 + 4] = __uint_as_float(r.v1);
  }
  csync();
  // every warp merges the warps' results itself (lanes 0..kWarps-1; the
  // winner and runner-up do not depend on the merge order)
  Race o;
  race_init(o);
  if (l < kWarps) {
    o.s1 = f[l * 5 + 0];
    o.t1 = f[l * 5 + 1];
    o.s2 = f[l * 5 + 2];
    o.t2 = f[l * 5 + 3];
    o.v1 = __float_as_uint(f[l * 5 + 4]);
  }
  warp_race_merge(o);
  o.s1lo = 0.f;
  csync();
  return o;
}

// Histogram selection on S.total (bin 0 = the top of the order): the bin
// where the cumulative weight from bin 0 reaches `need`, and the weight of
// the bins before it.  Warp 0 scans; the result is broadcast.
__device__ void select_from_bin0(GenShm& S, unsigned long long need, int* out_bin,
                                 unsigned long long* out_above) {
  if (ctid() < 32) {
    const int lane = ctid();
    unsigned long long own = 0;
    for (int i = 0; i < 8; ++i) own += S.total[8 * lane + i];
    unsigned long long inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const unsigned long long exc = inc - own;
    const unsigned ball = __ballot_sync(0xffffffffu, inc >= need);
    const int src = ball ? (__ffs(ball) - 1) : 31;
    if (lane == src) {
      unsigned long long above = exc;
      int chosen = 8 * lane + 7;
      for (int i = 0; i < 8; ++i) {
        const unsigned long long t = S.total[8 * lane + i];
        if (above + t >= need || i == 7) {
          chosen = 8 * lane + i;
          break;
        }
        above += t;
      }
      S.bci[2] = chosen;
      S.bc64[1] = above;
    }
  }
  csync();
  *out_bin = S.bci[2];
  *out_above = S.bc64[1];
  csync();
}

// ---------------------------------------------------------------------------
// Rank select on distances from the maximum (one settle group).  Values are described
// by d = key(max) - key(v) >= 0 in the order-key space, so the largest values
// have the smallest distances.  Finds the distance of the value at 1-based
// rank `need` (counting multiplicity) among the values `each` enumerates.
// The first histogram gives every distance below 255 << s0 its own bin and
// lumps the tail without an atomic; the chosen bin is refined 8 bits at a
// time; a rank in the tail falls back to a top-down radix over all bits.  On
// return `need` is the rank inside the group at exactly that distance.
// ---------------------------------------------------------------------------
template <typename Each>
__device__ uint32_t kth_distance(GenShm& S, Each each, unsigned long long& need, int s0, int dbits) {
  auto reduce = [&](int slot) {
    S.total[ctid()] = S.hist[slot][ctid()];
    csync();
  };
  int hs = 0;
  {
    const int slot = hs++ & 1;
    S.hist[slot][ctid()] = 0;
    csync();
    const uint32_t lim = 255u << s0;
    each([&](uint32_t d) {
      if (d < lim) atomicAdd(&S.hist[slot][d >> s0], 1u);
    });
    csync();
    reduce(slot);
    int b;
    unsigned long long below;
    select_from_bin0(S, need, &b, &below);
    if (b < 255) {
      need -= below;
      uint32_t base = (uint32_t)b << s0;
      for (int s = s0 - 8; s >= 0; s -= 8) {
        const int sl = hs++ & 1;
        S.hist[sl][ctid()] = 0;
        csync();
        const uint32_t span = 1u << (s + 8);
        each([&](uint32_t d) {
          if (d >= base && d - base < span) atomicAdd(&S.hist[sl][(d - base) >> s], 1u);
        });
        csync();
        reduce(sl);
        int bb;
        unsigned long long bl;
        select_from_bin0(S, need, &bb, &bl);
        need -= bl;
        base += (uint32_t)bb << s;
      }
      return base;
    }
  }
  uint32_t prefix = 0u, mask = 0u;
  for (int shift = dbits - 8; shift >= 0; shift -= 8) {
    const int slot = hs++ & 1;
    S.hist[slot][ctid()] = 0;
    csync();
    each([&](uint32_t d) {
      if ((d & mask) == prefix) atomicAdd(&S.hist[slot][(d >> shift) & 255u], 1u);
    });
    csync();
    reduce(slot);
    int b;
    unsigned long long below;
    select_from_bin0(S, need, &b, &below);
    need -= below;
    prefix |= (uint32_t)b << shift;
    mask |= 255u << shift;
  }
  return prefix;
}

// Exact fixed-point mass accumulation with native 32-bit shared atomics: the
// low word wraps, and the atomic that wraps it carries one into the high word.
__device__ __forceinline__ void mass_add(uint32_t* lo, uint32_t* hi, unsigned long long fx) {
  const uint32_t l = (uint32_t)fx;
  const uint32_t h = (uint32_t)(fx >> 32);
  const uint32_t old = atomicAdd(lo, l);
  const uint32_t carry = (old + l < old) ? 1u : 0u;
  if (h + carry) atomicAdd(hi, h + carry);
}
__device__ __forceinline__ unsigned long long mass_fixed(float e) {
  return __float2ull_rz(e * 1099511627776.0f);   // e * 2^40, e in [0, 1]
}

// Level 1 over a whole row, one settle group: every warp-row of 32 groups is one race
// block.  Returns the winning block's race state (v1 = block) in every thread.
template <bool kBF16>
__device__ Race race_blocks_row(const Args& A, GenShm& S, GenRing& R, int row, int pos, float m, float c, float invZ,
                                int mode, const Thresh* th) {
  const size_t lrow = ((size_t)row * (A.k + 1) + pos) * (size_t)A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const int G = (A.V + 7) / 8;
  const int lane = ctid() & 31, wp = ctid() >> 5;
  Race r;
  race_init(r);
  const bool with_q = mode == RW_RESIDUAL;
  if (A.vec_logits && (!with_q || A.vec_q) && R.ok) {
    // a warp's 32 groups of a round are one race block
    csweep<kBF16>(A, R, lrow, qrow, with_q, [&](int g, const float* v, const float* qv) {
      float w8 = 0.f, u8 = 0.f;
      if (g * 8 < A.V) {
        float w[8], tq[8];
        group_weights(A, g, v, qv, m, c, invZ, mode, th, w, tq);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (w[j] > 0.f) {
            w8 += w[j];
            u8 += w[j] + tq[j];
          }
      }
      const float W = warp_sum(w8), U = warp_sum(u8);
      const int g0 = __shfl_sync(0xffffffffu, g, 0);
      if (lane == 0 && W > 0.f) {
        const uint32_t bk = (uint32_t)(g0 / (kRaceBlock / 8));
        race_consider(r, W, U - W, bk, block_word(A, row, pos, bk));
      }
    });
    return block_race(S, r);
  }
  constexpr int QB = kGenBatch / 2;   // groups in flight: logits and q
  for (int base0 = 0; base0 < G; base0 += kThreads * QB) {
    float v[QB][8], qv[QB][8];
#pragma unroll
    for (int b = 0; b < QB; ++b) {
      const int g = base0 + b * kThreads + ctid();
#pragma unroll
      for (int j = 0; j < 8; ++j) qv[b][j] = 0.f;
      if (g < G) {
        load_group<kBF16>(A, lrow, g, true, v[b]);
        if (mode == RW_RESIDUAL) load_q8(A, qrow, g * 8, qv[b]);
      }
    }
#pragma unroll
    for (int b = 0; b < QB; ++b) {
      const int base = base0 + b * kThreads;
      const int g = base + ctid();
      float w8 = 0.f, u8 = 0.f;
      if (g < G) {
        float w[8], tq[8];
        group_weights(A, g, v[b], qv[b], m, c, invZ, mode, th, w, tq);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (w[j] > 0.f) {
            w8 += w[j];
            u8 += w[j] + tq[j];
          }
      }
      const float W = warp_sum(w8), U = warp_sum(u8);
      if (lane == 0 && W > 0.f) {
        const uint32_t bk = (uint32_t)(base / (kRaceBlock / 8) + wp);
        race_consider(r, W, U - W, bk, block_word(A, row, pos, bk));
      }
    }
  }
  return block_race(S, r);
}

// The full two-level draw over a row by one settle group; returns the drawn entry
// (or 0xffffffff when every weight is 0) and sets *margin.
template <bool kBF16>
__device__ uint32_t draw_row(const Args& A, GenShm& S, GenRing& R, int row, int pos, float m, float c, float invZ,
                             int mode, const Thresh* th, bool* margin) {
  const Race l1 = race_blocks_row<kBF16>(A, S, R, row, pos, m, c, invZ, mode, th);
  if (l1.s1 < 0.f) {
    *margin = false;
    return 0xffffffffu;
  }
  if (ctid() < 32) {
    const Race l2 = race_in_block<kBF16>(A, row, pos, l1.v1, m, c, invZ, mode, th);
    if (ctid() == 0) {
      S.bci[8] = (int)l2.v1;
      S.bci[9] = (draw_margin(l1) || draw_margin(l2)) ? 1 : 0;
    }
  }
  csync();
  const uint32_t y = (uint32_t)S.bci[8];
  *margin = S.bci[9] != 0;
  csync();
  return y;
}

// ---------------------------------------------------------------------------
// The general path: one settle group settles a unit whose kept set needs a global
// threshold (top-p without a small top-k, or a large top-k), in passes over
// the logit row (the first from HBM, later ones mostly from L2).  The kept
// set is a prefix of the total order, described by a Thresh.
// ---------------------------------------------------------------------------

// Index of the n-th (1-based) entry of the row, in index order, whose order
// key is tkey; 0xffffffff when there are fewer.
template <bool kBF16>
__device__ uint32_t nth_tie_index(const Args& A, GenShm& S, size_t lrow, uint32_t tkey, unsigned long long n) {
  const int G = (A.V + 7) / 8;
  constexpr int NB = kGenBatch;   // a thread takes NB consecutive groups a round
  unsigned long long need = n;
  uint32_t found = 0xffffffffu;
  for (int base = 0; base < G; base += kThreads * NB) {
    const int g0 = base + ctid() * NB;
    float v[NB][8];
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (g0 + b < G) load_group<kBF16>(A, lrow, g0 + b, true, v[b]);
    int c = 0;
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (g0 + b < G) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if ((g0 + b) * 8 + i < A.V && okey(v[b][i]) == tkey) ++c;
      }
    int rowtot = 0;
    const int exc = block_exclusive_scan(S, c, &rowtot);
    if (c > 0 && need > (unsigned long long)exc && need <= (unsigned long long)(exc + c)) {
      int want = (int)(need - exc);
      for (int b = 0; b < NB && want > 0; ++b) {
        const int g = g0 + b;
        if (g >= G) break;
        for (int i = 0; i < 8; ++i) {
          if (g * 8 + i < A.V && okey(v[b][i]) == tkey && --want == 0) {
            S.bci[10] = g * 8 + i;
            break;
          }
        }
      }
    }
    csync();
    if (need <= (unsigned long long)rowtot) {
      found = (uint32_t)S.bci[10];
      csync();
      break;
    }
    need -= (unsigned long long)rowtot;
    csync();
  }
  return found;
}

template <bool kBF16>
__device__ __noinline__ void unit_general(const Args& A, GenShm& S, GenRing& R, uint32_t tag, int u, int row,
                                          int pos, RowCfg cfg) {
  const size_t lrow = (size_t)u * A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const bool has_q = pos < A.k;
  const int G = (A.V + 7) / 8;
  // pass 1: max, argmax, NaN
  unsigned long long best = 0;
  bool nan_seen = false;
  row_pass<kBF16>(A, R, lrow, [&](int g, const float* v) {
    const float gm = group_max(v);
    if (gm != gm) {
      nan_seen = true;
    } else if (best == 0 || gm > from_okey((uint32_t)(best >> 32))) {
      int first = 0;
#pragma unroll
      for (int i = 7; i >= 0; --i)
        if (v[i] == gm) first = i;
      best = key64(okey(gm), (uint32_t)(g * 8 + first));
    }
  });
  if (nan_seen) best = ~0ull;
  best = block_max_u64(S, best);
  if (ctid() < 32) TLP(u, 1);
  const float m = from_okey((uint32_t)(best >> 32));
  const int am = (int)key64_idx(best);
  if (best == 0 || !(m > -INFINITY) || !(m < INFINITY)) {
    if (ctid() < 32) commit_record(A, tag, u, row, empty_record(SPEC_F_NAN));
    csync();
    return;
  }
  uint32_t flags = cfg.bad_param ? SPEC_F_BAD_PARAM : 0u;
  const float c = cfg.c;
  const uint32_t km = kf<kBF16>(m);

  // top-k threshold
  Thresh th;
  th.tkey = 0u;
  th.tidx = 0xffffffffu;
  if (cfg.K > 0) {
    unsigned long long need = (unsigned long long)cfg.K;
    auto each = [&](auto fn) {
      row_pass<kBF16>(A, R, lrow, [&](int g, const float* v) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (g * 8 + i < A.V) fn(km - kf<kBF16>(v[i]));
      });
    };
    const uint32_t d = kth_distance(S, each, need, kBF16 ? 0 : 16, kBF16 ? 16 : 32);
    th.tkey = full_key<kBF16>(km - d);
    th.tidx = nth_tie_index<kBF16>(A, S, lrow, th.tkey, need);
  }
  const bool topp = cfg.P < 1.0f;

  // Z pass over the top-k set; with top-p also a fixed-point mass histogram
  // binned by log2 of the weight in steps of 1/8 (the last bin in registers).
  const int hslot = 0;
  S.mlo[hslot][ctid()] = 0;
  S.mhi[hslot][ctid()] = 0;
  csync();
  unsigned long long tail = 0;
  float z0 = 0.f, z1 = 0.f;
  row_pass<kBF16>(A, R, lrow, [&](int g, const float* v) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float x = (v[i] - m) * c;
      const bool in = (g * 8 + i < A.V) && (cfg.K == 0 || kept(th, okey(v[i]), (uint32_t)(g * 8 + i)));
      const float e = in ? ex2(x) : 0.f;
      if (i & 1) z1 += e; else z0 += e;
      if (topp && e > 0.f) {
        const int bin = __float2int_rz(fminf(-x * 8.0f, 255.0f));
        const unsigned long long fx = mass_fixed(e);
        if (bin < 255) mass_add(&S.mlo[hslot][bin], &S.mhi[hslot][bin], fx);
        else tail += fx;
      }
    }
  });
  float Zs;
  if (ctid() < 32) TLP(u, 2);
  if (topp) {
    csync();
    tail = block_sum_u64(S, tail);
    if (ctid() == 0) {
      S.mlo[hslot][255] = (uint32_t)tail;
      S.mhi[hslot][255] = (uint32_t)(tail >> 32);
    }
    csync();
    S.total[ctid()] = ((unsigned long long)S.mhi[hslot][ctid()] << 32) + S.mlo[hslot][ctid()];
    csync();
    const unsigned long long zk = block_sum_u64(S, S.total[ctid()]);
    const unsigned long long target = (unsigned long long)ceil((double)cfg.P * (double)zk);
    int b;
    unsigned long long above;
    select_from_bin0(S, target, &b, &above);
    // key range of bin b
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    row_pass<kBF16>(A, R, lrow, [&](int g, const float* v) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (g * 8 + i >= A.V) continue;
        const uint32_t key = okey(v[i]);
        if (cfg.K > 0 && !kept(th, key, (uint32_t)(g * 8 + i))) continue;
        const float x = (v[i] - m) * c;
        if (!(ex2(x) > 0.f)) continue;
        if (__float2int_rz(fminf(-x * 8.0f, 255.0f)) == b) {
          kmin = min(kmin, key);
          kmax = max(kmax, key);
        }
      }
    });
    const uint2 mm = block_minmax_u32(S, kmin, kmax);
    if (ctid() < 32) TLP(u, 3);
    uint32_t lo = mm.x, hi = mm.y;
    unsigned long long rem = target - above;
    int hs = 1;
    while (hi > lo) {
      const uint32_t span = hi - lo;
      const int nbits = 32 - __clz(span);
      const int shift = nbits > 8 ? nbits - 8 : 0;
      const int slot = hs++ & 1;
      S.mlo[slot][ctid()] = 0;
      S.mhi[slot][ctid()] = 0;
      csync();
      row_pass<kBF16>(A, R, lrow, [&](int g, const float* v) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (g * 8 + i >= A.V) continue;
          const uint32_t key = okey(v[i]);
          if (key < lo || key > hi) continue;
          if (cfg.K > 0 && !kept(th, key, (uint32_t)(g * 8 + i))) continue;
          const uint32_t bin = (hi - key) >> shift;
          mass_add(&S.mlo[slot][bin], &S.mhi[slot][bin], mass_fixed(ex2((v[i] - m) * c)));
        }
      });
      csync();
      S.total[ctid()] = ((unsigned long long)S.mhi[slot][ctid()] << 32) + S.mlo[slot][ctid()];
      csync();
      int sb;
      unsigned long long ab;
      select_from_bin0(S, rem, &sb, &ab);
      rem -= ab;
      above += ab;
      const uint32_t nhi = hi - ((uint32_t)sb << shift);
      const uint32_t span_lo = ((uint32_t)(sb + 1) << shift) - 1u;
      const uint32_t nlo = (hi - lo > span_lo) ? max(lo, hi - span_lo) : lo;
      hi = nhi;
      lo = max(nlo, lo);
      if (shift == 0) lo = hi;
    }
    const uint32_t tkey = hi;
    if (ctid() < 32) TLP(u, 4);
    const float et = ex2((from_okey(tkey) - m) * c);
    const unsigned long long efx = mass_fixed(et);
    unsigned long long n_need = efx ? (rem + efx - 1) / efx : 1ull;
    if (n_need == 0) n_need = 1;
    // with a top-k threshold at the same key, the ties top-k keeps are a
    // prefix of the ties in index order, so the rank carries over
    th.tidx = nth_tie_index<kBF16>(A, S, lrow, tkey, n_need);
    th.tkey = tkey;
    if (ctid() < 32) TLP(u, 5);
    const unsigned long long zs_fx = above + n_need * efx;
    Zs = (float)((double)zs_fx * (1.0 / 1099511627776.0));
    const double at = (double)zs_fx / (double)zk;
    const double bef = (double)(zs_fx - efx) / (double)zk;
    if (fabs(at - (double)cfg.P) < 1e-6 || fabs((double)cfg.P - bef) < 1e-6) flags |= SPEC_F_MARGIN_TOPP;
  } else {
    Zs = block_sum(S, z0 + z1);
  }
  const float invZ = 1.0f / Zs;
  const float lnZ = logf(Zs);

  // accept test (every thread computes the same)
  AcceptInfo ai;
  ai.accept = false;
  ai.valid = true;
  ai.margin = false;
  ai.lx = 0.f;
  bool need_race = !has_q;
  if (has_q) {
    ai = accept_test(A, row, pos, kBF16, false, am, m, c, Zs, &th);
    need_race = !ai.accept;
  }
  // alpha pass
  float al0 = 0.f, al1 = 0.f;
  if (has_q) {
    auto acc = [&](int g, const float* v, const float* qv) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const bool in = (g * 8 + i < A.V) && kept(th, okey(v[i]), (uint32_t)(g * 8 + i));
        const float p = in ? ex2((v[i] - m) * c) * invZ : 0.f;
        if (i & 1) al1 += fminf(p, qv[i]); else al0 += fminf(p, qv[i]);
      }
    };
    if (A.vec_logits && A.vec_q && R.ok) {
      csweep<kBF16>(A, R, lrow, qrow, true, acc);
    } else {
      for (int g = ctid(); g < G; g += kThreads) {
        float v[8], qv[8];
        load_group<kBF16>(A, lrow, g, true, v);
        load_q8(A, qrow, g * 8, qv);
        acc(g, v, qv);
      }
    }
  }
  const float alpha_v = has_q ? block_sum(S, al0 + al1) : 0.f;
  if (ctid() < 32) TLP(u, 6);
  // the draw: residual after a rejection, p at the bonus position
  uint32_t draw_flags = 0;
  uint32_t y = 0xffffffffu;
  if (need_race) {
    bool mg = false;
    y = draw_row<kBF16>(A, S, R, row, pos, m, c, invZ, has_q ? RW_RESIDUAL : RW_BONUS, &th, &mg);
    if (y == 0xffffffffu) {
      draw_flags |= SPEC_F_RESIDUAL_EMPTY;
      y = draw_row<kBF16>(A, S, R, row, pos, m, c, invZ, RW_P, &th, &mg);
    }
    if (mg) draw_flags |= SPEC_F_MARGIN_DRAW;
  }
  if (ctid() < 32) TLP(u, 7);
  if (!R.ok) {
    // a chunk's copy gave up: the unit's results are not trusted
    if (ctid() < 32) commit_record(A, tag, u, row, empty_record(SPEC_F_TIMEOUT));
    csync();
    return;
  }
  UnitRecord rec = empty_record(flags);
  if (ctid() == 0) {
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
  }
  if (ctid() < 32) {
    publish_desc(A, tag, u, DESC_THRESH, m, invZ, th.tkey, th.tidx);
    commit_record(A, tag, u, row, rec);
  }
  csync();
}

}  // namespace specv
