// spec_verify: batched speculative-decoding verify sampler for sm_103a.
//
// Method: inclusionAI/AReno PR #550, "feat(engine): MTP training loss and
// speculative decoding for bailing_v3", "What does this PR do?" Phase 2
// (sampler-equivalent target distribution, exact chain rejection sampling,
// unchanged logprobs), table "Per-step optimizations" (Gumbel-max draws,
// one-pass logprobs, no host syncs) and table "On-policy accept probability"
// (alpha = sum min(p, q)).  Ties follow InfiniTensor/InfiniLM PR #588, "feat:
// add mtp draft models for speculative decoding", section 4.1 (exact bf16
// ties flip argmax between kernel paths, so the order is defined: larger
// logit first, then smaller index).
//
// Execution model: one persistent grid of independent CTAs (several per SM)
// pulls work items from two counters in the workspace.  A "unit" is one
// (row, position); its vocabulary is cut into chunks of 8192 entries.
//
//   A items (unit, chunk): stream the chunk from HBM once and reduce it to a
//     chunk record: max and argmax, the softmax sum relative to the chunk
//     max, the exponential-race partial of an unfiltered bonus position, and
//     for small top-k the chunk's own sorted top-K list.  An atomic ticket
//     per unit makes the CTA that finishes the last chunk the unit's
//     finaliser: it merges the chunk records in chunk order (deterministic),
//     and settles greedy, small top-k and bonus units completely; for a
//     position with a draft over an unfiltered distribution it decides the
//     accept test and publishes the unit state.
//   B items (unit, chunk), only for such drafted unfiltered positions: wait
//     (bounded) for the unit state, then re-read the chunk (L2) and stream q
//     for alpha = sum min(p, q) and, after a rejection, the residual race.
//     The last chunk's CTA merges and settles the unit.
//   Units with a kept set that needs a global threshold search (top-p
//     without a small top-k, or a large top-k) are settled by one CTA in
//     passes over the row (the general path).
//
// Every A item is claimed before any B item, and A items never wait, so the
// B items' waits always end.  A per-row ticket makes the last settled unit of
// a row resolve the accept chain and write the row's outputs.  All
// reductions use a fixed order, and no floating-point atomics are used, so
// results are bit-reproducible.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/spec_verify.h"
#include "spec_device.cuh"
#include "spec_host.h"

namespace specv {

constexpr int kChunk = 8192;               // vocabulary entries per chunk
constexpr int kGPC = kChunk / 8;           // groups of 8 entries per chunk
constexpr int kGPT = kGPC / kThreads;      // groups per thread
constexpr int kTopkSmall = 128;            // top_k <= this keeps per-chunk lists
constexpr int kMergeCap = 4096;            // finaliser buffer: candidates + super-group maxima
constexpr int kSPC = kGPC / 8;             // 64-entry super-groups per chunk
constexpr int kMaxNCTopk = kMergeCap / kSPC;         // chunks whose maxima fit half the buffer (as floats)
constexpr long long kSpinLimit = 1ll << 24;
constexpr int kClaim = 1;                  // items claimed per atomic
constexpr int kRaceBlock = 256;            // entries per block of the two-level race

enum { UT_GREEDY = 0, UT_TOPK = 1, UT_DENSE = 2, UT_GENERAL = 3 };

struct WsHeader {
  uint32_t a_next;        // next A item
  uint32_t b_next;        // next B item
  uint32_t ctas_done;     // CTAs that left the kernel
  uint32_t error;         // bit 0: a bounded wait gave up
  uint32_t pad[60];
};

struct ChunkRec {         // 48 bytes, one per (unit, chunk)
  float m;                // chunk max (NaN when the chunk holds a NaN)
  uint32_t amax;          // first index of the chunk max
  float z;                // sum of exp((l - m_chunk) * c)
  uint32_t nlist;         // unused
  float s1, t1, s2, t2;   // race partial relative to the chunk max (bonus units)
  uint32_t v1;
  uint32_t overflow;      // unused
  uint32_t pad[2];
};

struct UnitState {        // 48 bytes: what the B items of a drafted unfiltered unit need
  float m, invZ, lnZ, lp_x;
  int32_t accept;
  uint32_t flags;         // BAD_TOKEN | MARGIN_ACCEPT | BAD_PARAM of this unit
  uint32_t invalid;       // the unit is invalid (NaN); its record is already written
  int32_t am;
  uint32_t pad[4];
};

struct BRec {             // 32 bytes per (unit, chunk)
  float alpha, s1, t1, s2, t2;
  uint32_t v1;
  uint32_t pad[2];
};

struct UnitRecord {       // 32 bytes, one per unit, read by the row finaliser
  uint32_t flags;
  int32_t accept;
  float lp_x;
  float alpha;
  int32_t y;
  float lp_y;
  uint32_t draw_flags;
  uint32_t pad;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t row_ticket, a_ticket, b_ticket, ready, crec, ust, brec, urec, smax, total;
};

__host__ __device__ inline Layout ws_layout(int B, int k, int V) {
  const size_t U = (size_t)B * (k + 1);
  const size_t NC = ((size_t)V + kChunk - 1) / kChunk;
  Layout L;
  size_t off = sizeof(WsHeader);
  L.row_ticket = off; off = align_up(off + (size_t)B * 4, 256);
  L.a_ticket = off; off = align_up(off + U * 4, 256);
  L.b_ticket = off; off = align_up(off + U * 4, 256);
  L.ready = off; off = align_up(off + U * 4, 256);
  L.crec = off; off = align_up(off + U * NC * sizeof(ChunkRec), 256);
  L.ust = off; off = align_up(off + U * sizeof(UnitState), 256);
  L.brec = off; off = align_up(off + U * NC * sizeof(BRec), 256);
  L.urec = off; off = align_up(off + U * sizeof(UnitRecord), 256);
  L.smax = off; off = align_up(off + U * NC * kSPC * 4, 256);
  L.total = off;
  return L;
}

struct Args {
  const void* logits;
  const float* q;
  const int32_t* drafts;
  const spec_params_t* params;
  int32_t* tokens;
  int32_t* accept_len;
  float* logprobs;
  float* alpha;
  uint32_t* flags;
  WsHeader* ws;
  uint32_t* row_ticket;
  uint32_t* a_ticket;
  uint32_t* b_ticket;
  uint32_t* ready;
  ChunkRec* crec;
  UnitState* ust;
  BRec* brec;
  UnitRecord* urec;
  float* smax;
  uint32_t key0, key1;
  int B, k, V, NC, U;
  int NA, NB;
  int n_ctas;
  int vec_logits;
  int vec_q;
};

// Shared memory of one CTA (dynamic).
struct alignas(16) Shm {
  uint32_t hist[2][256];
  uint32_t mlo[2][256];
  uint32_t mhi[2][256];
  unsigned long long total[256];
  unsigned long long bc64[8];
  float wred[kWarps * 8];
  float bcf[8];
  int bci[16];
  uint32_t cand_count;
  float gmax[kGPC];
  float list_e[kTopkSmall];
  float list_cum[kTopkSmall];
  float list_w[kTopkSmall];
  float list_u[kTopkSmall];
  float bm[32], bw[32], bu[32], ba[32];   // per race block of a chunk: max, weight, margin weight, alpha
  uint32_t bi[32];                        // per race block: first index of the max
  unsigned long long cand[kMergeCap];
};

// ---------------------------------------------------------------------------
// Row configuration.
// ---------------------------------------------------------------------------
struct RowCfg {
  int type;
  bool bad_param;
  int K;        // active top-k (0 = off)
  float P;      // active top-p (1 = off)
  float c;      // log2(e) / T (log2(e) for greedy)
  float invT;   // 1 / T (1 for greedy)
};

__device__ __forceinline__ RowCfg classify(const spec_params_t& prm, int V, int NC) {
  RowCfg r;
  const float T = prm.temperature;
  const float P = prm.top_p;
  const bool T_ok = (T == 0.0f) || (isfinite(T) && T >= 1.17549435e-38f);
  const bool P_ok = isfinite(P) && P > 0.0f && P <= 1.0f;
  r.bad_param = !(T_ok && P_ok);
  const bool greedy = r.bad_param || T == 0.0f;
  r.K = (prm.top_k > 0 && prm.top_k < V) ? prm.top_k : 0;
  r.P = (greedy || P >= 1.0f) ? 1.0f : P;
  r.c = greedy ? kLog2e : kLog2e / T;
  r.invT = greedy ? 1.0f : 1.0f / T;
  if (greedy) r.type = UT_GREEDY;
  else if (r.K > 0 && r.K <= kTopkSmall && NC <= kMaxNCTopk) r.type = UT_TOPK;
  else if (r.K == 0 && r.P >= 1.0f) r.type = UT_DENSE;
  else r.type = UT_GENERAL;
  return r;
}

// ---------------------------------------------------------------------------
// Block reductions (fixed combination order, so results are reproducible).
// Each returns its result in every thread.
// ---------------------------------------------------------------------------
__device__ float block_sum(Shm& S, float a) {
  a = warp_sum(a);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) S.wred[w] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float x = 0.f;
    for (int i = 0; i < kWarps; ++i) x += S.wred[i];
    S.bcf[7] = x;
  }
  __syncthreads();
  const float r = S.bcf[7];
  __syncthreads();
  return r;
}

__device__ unsigned long long block_max_u64(Shm& S, unsigned long long v) {
  v = warp_max_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  unsigned long long* buf = reinterpret_cast<unsigned long long*>(S.wred);
  if (l == 0) buf[w] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long x = 0;
    for (int i = 0; i < kWarps; ++i) x = buf[i] > x ? buf[i] : x;
    S.bc64[7] = x;
  }
  __syncthreads();
  const unsigned long long r = S.bc64[7];
  __syncthreads();
  return r;
}

__device__ unsigned long long block_sum_u64(Shm& S, unsigned long long v) {
  v = warp_sum_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  unsigned long long* buf = reinterpret_cast<unsigned long long*>(S.wred);
  if (l == 0) buf[w] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long x = 0;
    for (int i = 0; i < kWarps; ++i) x += buf[i];
    S.bc64[7] = x;
  }
  __syncthreads();
  const unsigned long long r = S.bc64[7];
  __syncthreads();
  return r;
}

__device__ uint2 block_minmax_u32(Shm& S, uint32_t mn, uint32_t mx) {
  uint32_t a = ~mn, b = mx;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  uint32_t* wb = reinterpret_cast<uint32_t*>(S.wred);
  if ((threadIdx.x & 31) == 0) {
    wb[2 * (threadIdx.x >> 5)] = a;
    wb[2 * (threadIdx.x >> 5) + 1] = b;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t aa = 0, bb = 0;
    for (int i = 0; i < kWarps; ++i) {
      aa = max(aa, wb[2 * i]);
      bb = max(bb, wb[2 * i + 1]);
    }
    S.bci[12] = (int)~aa;
    S.bci[13] = (int)bb;
  }
  __syncthreads();
  const uint2 r = make_uint2((uint32_t)S.bci[12], (uint32_t)S.bci[13]);
  __syncthreads();
  return r;
}

__device__ Race block_race(Shm& S, Race r) {
  warp_race_merge(r);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  float* f = S.wred;
  if (l == 0) {
    f[w * 5 + 0] = r.s1;
    f[w * 5 + 1] = r.t1;
    f[w * 5 + 2] = r.s2;
    f[w * 5 + 3] = r.t2;
    f[w * 5 + 4] = __uint_as_float(r.v1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Race a;
    race_init(a);
    for (int i = 0; i < kWarps; ++i) {
      Race b;
      b.s1 = f[i * 5 + 0];
      b.t1 = f[i * 5 + 1];
      b.s2 = f[i * 5 + 2];
      b.t2 = f[i * 5 + 3];
      b.v1 = __float_as_uint(f[i * 5 + 4]);
      b.s1lo = 0.f;
      race_merge(a, b);
    }
    S.bcf[0] = a.s1;
    S.bcf[1] = a.t1;
    S.bcf[2] = a.s2;
    S.bcf[3] = a.t2;
    S.bci[0] = (int)a.v1;
  }
  __syncthreads();
  Race o;
  o.s1 = S.bcf[0];
  o.t1 = S.bcf[1];
  o.s2 = S.bcf[2];
  o.t2 = S.bcf[3];
  o.v1 = (uint32_t)S.bci[0];
  o.s1lo = 0.f;
  __syncthreads();
  return o;
}

// Histogram selection on S.total (bin 0 = the top of the order): the bin
// where the cumulative weight from bin 0 reaches `need`, and the weight of
// the bins before it.  Warp 0 scans; the result is broadcast.
__device__ void select_from_bin0(Shm& S, unsigned long long need, int* out_bin,
                                 unsigned long long* out_above) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
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
  __syncthreads();
  *out_bin = S.bci[2];
  *out_above = S.bc64[1];
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Rank select on distances from the maximum (one CTA).  Values are described
// by d = key(max) - key(v) >= 0 in the order-key space, so the largest values
// have the smallest distances.  Finds the distance of the value at 1-based
// rank `need` (counting multiplicity) among the values `each` enumerates.
// The first histogram gives every distance below 255 << s0 its own bin and
// lumps the tail without an atomic; the chosen bin is refined 8 bits at a
// time; a rank in the tail falls back to a top-down radix over all bits.  On
// return `need` is the rank inside the group at exactly that distance.
// ---------------------------------------------------------------------------
template <typename Each>
__device__ uint32_t kth_distance(Shm& S, Each each, unsigned long long& need, int s0, int dbits) {
  auto reduce = [&](int slot) {
    S.total[threadIdx.x] = S.hist[slot][threadIdx.x];
    __syncthreads();
  };
  int hs = 0;
  {
    const int slot = hs++ & 1;
    S.hist[slot][threadIdx.x] = 0;
    __syncthreads();
    const uint32_t lim = 255u << s0;
    each([&](uint32_t d) {
      if (d < lim) atomicAdd(&S.hist[slot][d >> s0], 1u);
    });
    __syncthreads();
    reduce(slot);
    int b;
    unsigned long long below;
    select_from_bin0(S, need, &b, &below);
    if (b < 255) {
      need -= below;
      uint32_t base = (uint32_t)b << s0;
      for (int s = s0 - 8; s >= 0; s -= 8) {
        const int sl = hs++ & 1;
        S.hist[sl][threadIdx.x] = 0;
        __syncthreads();
        const uint32_t span = 1u << (s + 8);
        each([&](uint32_t d) {
          if (d >= base && d - base < span) atomicAdd(&S.hist[sl][(d - base) >> s], 1u);
        });
        __syncthreads();
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
    S.hist[slot][threadIdx.x] = 0;
    __syncthreads();
    each([&](uint32_t d) {
      if ((d & mask) == prefix) atomicAdd(&S.hist[slot][(d >> shift) & 255u], 1u);
    });
    __syncthreads();
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

template <bool kBF16>
__device__ __forceinline__ uint32_t kf(float v) {
  return kBF16 ? (okey(v) >> 16) : okey(v);
}
template <bool kBF16>
__device__ __forceinline__ uint32_t full_key(uint32_t k) {
  if (!kBF16) return k;
  return (k << 16) | ((k & 0x8000u) ? 0u : 0xffffu);
}

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

// ---------------------------------------------------------------------------
// Loading logits and draft probabilities.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float load_logit(const Args& A, bool bf16, size_t off) {
  if (bf16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(A.logits)[off] << 16);
  return reinterpret_cast<const float*>(A.logits)[off];
}

// Eight values of group g (entries 8g..8g+7) of a logit row; entries past V
// read as -inf.  keep: leave the lines in L2 for a later re-read.
template <bool kBF16>
__device__ __forceinline__ void load_group(const Args& A, size_t lrow, int g, bool keep, float v[8]) {
  const int e0 = g * 8;
  if (kBF16) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(A.logits) + lrow;
    uint4 w;
    if (A.vec_logits && e0 + 8 <= A.V) {
      const uint4* p4 = reinterpret_cast<const uint4*>(p + e0);
      w = keep ? __ldcg(p4) : __ldcs(p4);
    } else {
      uint32_t h[8];
      for (int i = 0; i < 8; ++i) h[i] = (e0 + i < A.V) ? p[e0 + i] : 0xff80u;
      w = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
    }
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
    v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
    v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
  } else {
    const float* p = reinterpret_cast<const float*>(A.logits) + lrow;
    if (A.vec_logits && e0 + 8 <= A.V) {
      const float4* p4 = reinterpret_cast<const float4*>(p + e0);
      const float4 a = keep ? __ldcg(p4) : __ldcs(p4);
      const float4 b = keep ? __ldcg(p4 + 1) : __ldcs(p4 + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
      for (int i = 0; i < 8; ++i) v[i] = (e0 + i < A.V) ? p[e0 + i] : -INFINITY;
    }
  }
}

__device__ __forceinline__ void load_q8(const Args& A, size_t qrow, int e0, float qv[8]) {
  const float* p = A.q + qrow;
  if (A.vec_q && e0 + 8 <= A.V) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p + e0));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p + e0 + 4));
    qv[0] = a.x; qv[1] = a.y; qv[2] = a.z; qv[3] = a.w;
    qv[4] = b.x; qv[5] = b.y; qv[6] = b.z; qv[7] = b.w;
  } else {
    for (int i = 0; i < 8; ++i) qv[i] = (e0 + i < A.V) ? p[e0 + i] : 0.f;
  }
}

__device__ __forceinline__ float group_max(const float v[8]) {
  return max_nan(max_nan(max_nan(v[0], v[1]), max_nan(v[2], v[3])),
                 max_nan(max_nan(v[4], v[5]), max_nan(v[6], v[7])));
}

// ---------------------------------------------------------------------------
// Records and the per-row finalize.
// ---------------------------------------------------------------------------
__device__ void finalize_row(const Args& A, int row) {
  const int k = A.k;
  const UnitRecord* R = A.urec + (size_t)row * (k + 1);
  uint32_t uflags = 0;
  bool invalid = false;
  for (int j = 0; j <= k; ++j) {
    const uint32_t f = __ldcg(&R[j].flags);
    uflags |= f & (SPEC_F_NAN | SPEC_F_BAD_PARAM | SPEC_F_BAD_TOKEN | SPEC_F_MARGIN_TOPP);
    invalid |= (f & SPEC_F_NAN) != 0;
  }
  int32_t* tok = A.tokens + (size_t)row * (k + 1);
  float* lp = A.logprobs + (size_t)row * (k + 1);
  if (invalid) {
    for (int j = 0; j <= k; ++j) {
      tok[j] = -1;
      lp[j] = 0.f;
    }
    for (int j = 0; j < k; ++j) A.alpha[(size_t)row * k + j] = 0.f;
    A.accept_len[row] = 0;
    A.flags[row] = SPEC_F_NAN;
    return;
  }
  int a = k;
  for (int j = 0; j < k; ++j) {
    uflags |= __ldcg(&R[j].flags) & SPEC_F_MARGIN_ACCEPT;
    if (!__ldcg(&R[j].accept)) {
      a = j;
      break;
    }
  }
  for (int j = 0; j < a; ++j) {
    tok[j] = A.drafts[(size_t)row * k + j];
    lp[j] = __ldcg(&R[j].lp_x);
  }
  tok[a] = __ldcg(&R[a].y);
  lp[a] = __ldcg(&R[a].lp_y);
  uflags |= __ldcg(&R[a].draw_flags);
  for (int j = a + 1; j <= k; ++j) {
    tok[j] = -1;
    lp[j] = 0.f;
  }
  for (int j = 0; j < k; ++j) A.alpha[(size_t)row * k + j] = __ldcg(&R[j].alpha);
  A.accept_len[row] = a + 1;
  A.flags[row] = uflags;
}

// One thread: publish a unit's record; the last unit of the row finalizes it.
__device__ void commit_record(const Args& A, int u, int row, const UnitRecord& rec) {
  A.urec[u] = rec;
  const uint32_t old = atomic_add_acq_rel(&A.row_ticket[row], 1u);
  if (old == (uint32_t)A.k) {
    finalize_row(A, row);
    A.row_ticket[row] = 0;   // leave the workspace clean for the next call
  }
}

__device__ __forceinline__ UnitRecord empty_record(uint32_t flags) {
  UnitRecord r;
  r.flags = flags;
  r.accept = 0;
  r.lp_x = 0.f;
  r.alpha = 0.f;
  r.y = -1;
  r.lp_y = 0.f;
  r.draw_flags = 0;
  r.pad = 0;
  return r;
}

struct AcceptInfo {
  bool valid, accept, margin;
  int x;
  float px, qx, lx;
};

// Accept test of the draft at (row, pos): accept iff u*q(x) < p(x), with the
// sign of u*q - p taken exactly by one fma.  p(x) = exp((l_x - m) / T) / Z
// when x is kept (kept_th == nullptr keeps everything); greedy: p(x) = 1 if
// x is the argmax, else 0.
struct Thresh {
  uint32_t tkey;
  uint32_t tidx;
};
__device__ __forceinline__ bool kept(const Thresh& t, uint32_t key, uint32_t v) {
  return key > t.tkey || (key == t.tkey && v <= t.tidx);
}

__device__ AcceptInfo accept_test(const Args& A, int row, int pos, bool bf16, bool greedy, int am,
                                  float m, float c, float Zs, const Thresh* kept_th) {
  AcceptInfo ai;
  ai.x = A.drafts[(size_t)row * A.k + pos];
  ai.valid = ai.x >= 0 && ai.x < A.V;
  ai.lx = 0.f;
  ai.px = 0.f;
  ai.qx = 0.f;
  const size_t lrow = ((size_t)row * (A.k + 1) + pos) * (size_t)A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  if (ai.valid) {
    ai.lx = load_logit(A, bf16, lrow + ai.x);
    ai.qx = A.q[qrow + ai.x];
    if (greedy) {
      ai.px = (ai.x == am) ? 1.0f : 0.0f;
    } else {
      const bool in = kept_th ? kept(*kept_th, okey(ai.lx), (uint32_t)ai.x) : true;
      ai.px = in ? ex2((ai.lx - m) * c) / Zs : 0.0f;
    }
  }
  const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)pos, (uint32_t)row, 0u), A.key0, A.key1);
  const float u = uniform_of(w.x);
  const float d = fmaf(u, ai.qx, -ai.px);
  ai.accept = d < 0.0f;
  ai.margin = (ai.px > 0.0f && ai.px < 1.0f && fabsf(d) < kMargin);
  return ai;
}

__device__ __forceinline__ uint32_t race_word(const Args& A, int row, int pos, uint32_t v) {
  const uint4 w = philox4x32_10(make_uint4(v >> 2, (uint32_t)pos, (uint32_t)row, 1u), A.key0, A.key1);
  return word_of(w, v & 3);
}

// Race over the 8 weights of one group (two Philox blocks), skipping empty halves.
__device__ __forceinline__ void race_group(const Args& A, int row, int pos, int e0, const float w[8],
                                           const float tq[8], Race& r) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float* wh = w + 4 * h;
    if (wh[0] > 0.f || wh[1] > 0.f || wh[2] > 0.f || wh[3] > 0.f) {
      const uint32_t blk = (uint32_t)((e0 >> 2) + h);
      const uint4 ww = philox4x32_10(make_uint4(blk, (uint32_t)pos, (uint32_t)row, 1u), A.key0, A.key1);
      if (wh[0] > 0.f) race_consider(r, wh[0], tq[4 * h + 0], blk * 4 + 0, ww.x);
      if (wh[1] > 0.f) race_consider(r, wh[1], tq[4 * h + 1], blk * 4 + 1, ww.y);
      if (wh[2] > 0.f) race_consider(r, wh[2], tq[4 * h + 2], blk * 4 + 2, ww.z);
      if (wh[3] > 0.f) race_consider(r, wh[3], tq[4 * h + 3], blk * 4 + 3, ww.w);
    }
  }
}

__device__ __forceinline__ bool draw_margin(const Race& r) {
  return r.s2 >= 0.f && (r.s1 - r.s2) < kMargin * (r.t1 + r.t2);
}

// The draw is a two-level exponential race: level 1 races the blocks of
// kRaceBlock consecutive entries with their total weights (one Philox word
// per block, stream 2), level 2 races the entries of the winning block
// (stream 1).  Block b then wins with probability W_b / sum W and entry v of
// it with r_v / W_b, so v is drawn with probability r_v / sum r exactly,
// while only one block needs a random number per entry.
__device__ __forceinline__ uint32_t block_word(const Args& A, int row, int pos, uint32_t b) {
  const uint4 w = philox4x32_10(make_uint4(b >> 2, (uint32_t)pos, (uint32_t)row, 2u), A.key0, A.key1);
  return word_of(w, b & 3);
}

enum { RW_BONUS = 0, RW_RESIDUAL = 1, RW_P = 2 };

// Weights of the 8 entries of group g: RW_BONUS / RW_P use exp2((l - m) c)
// (margin weight: the same), RW_RESIDUAL uses max(p - q, 0) with
// p = exp2((l - m) c) * invZ (margin weight p + q).  Entries outside the
// kept set (th) or past V weigh 0.  Returns in w[] and tq[] = margin - w.
template <bool kBF16>
__device__ __forceinline__ void race_weights(const Args& A, size_t lrow, size_t qrow, int g, float m, float c,
                                             float invZ, int mode, const Thresh* th, float w[8], float tq[8]) {
  float v[8], qv[8];
  load_group<kBF16>(A, lrow, g, true, v);
  if (mode == RW_RESIDUAL) {
    load_q8(A, qrow, g * 8, qv);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) qv[j] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const bool in = (g * 8 + j < A.V) && (th == nullptr || kept(*th, okey(v[j]), (uint32_t)(g * 8 + j)));
    const float e = in ? ex2((v[j] - m) * c) : 0.f;
    if (mode == RW_RESIDUAL) {
      const float p = e * invZ;
      w[j] = fmaxf(p - qv[j], 0.f);
      tq[j] = 2.0f * qv[j];
    } else {
      w[j] = e;
      tq[j] = 0.f;
    }
  }
}

// Level 2: the race among the entries of block b, run by one warp (the
// result is in every lane).
template <bool kBF16>
__device__ Race race_in_block(const Args& A, int row, int pos, uint32_t b, float m, float c, float invZ, int mode,
                              const Thresh* th) {
  const int lane = threadIdx.x & 31;
  const size_t lrow = ((size_t)row * (A.k + 1) + pos) * (size_t)A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const int G = (A.V + 7) / 8;
  const int g = (int)b * (kRaceBlock / 8) + lane;
  Race r;
  race_init(r);
  if (g < G) {
    float w[8], tq[8];
    race_weights<kBF16>(A, lrow, qrow, g, m, c, invZ, mode, th, w, tq);
    race_group(A, row, pos, g * 8, w, tq, r);
  }
  warp_race_merge(r);
  return r;
}

// Level 1 over a whole row, one CTA: every warp-row of 32 groups is one race
// block.  Returns the winning block's race state (v1 = block) in every thread.
template <bool kBF16>
__device__ Race race_blocks_row(const Args& A, Shm& S, int row, int pos, float m, float c, float invZ, int mode,
                                const Thresh* th) {
  const size_t lrow = ((size_t)row * (A.k + 1) + pos) * (size_t)A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const int G = (A.V + 7) / 8;
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  Race r;
  race_init(r);
  for (int base = 0; base < G; base += kThreads) {
    const int g = base + threadIdx.x;
    float w8 = 0.f, u8 = 0.f;
    if (g < G) {
      float w[8], tq[8];
      race_weights<kBF16>(A, lrow, qrow, g, m, c, invZ, mode, th, w, tq);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (w[j] > 0.f) {
          w8 += w[j];
          u8 += w[j] + tq[j];
        }
    }
    const float W = warp_sum(w8), U = warp_sum(u8);
    if (lane == 0 && W > 0.f) {
      const uint32_t b = (uint32_t)(base / (kRaceBlock / 8) + wp);
      race_consider(r, W, U - W, b, block_word(A, row, pos, b));
    }
  }
  return block_race(S, r);
}

// The full two-level draw over a row by one CTA; returns the drawn entry
// (or 0xffffffff when every weight is 0) and sets *margin.
template <bool kBF16>
__device__ uint32_t draw_row(const Args& A, Shm& S, int row, int pos, float m, float c, float invZ, int mode,
                             const Thresh* th, bool* margin) {
  const Race l1 = race_blocks_row<kBF16>(A, S, row, pos, m, c, invZ, mode, th);
  if (l1.s1 < 0.f) {
    *margin = false;
    return 0xffffffffu;
  }
  if (threadIdx.x < 32) {
    const Race l2 = race_in_block<kBF16>(A, row, pos, l1.v1, m, c, invZ, mode, th);
    if (threadIdx.x == 0) {
      S.bci[8] = (int)l2.v1;
      S.bci[9] = (draw_margin(l1) || draw_margin(l2)) ? 1 : 0;
    }
  }
  __syncthreads();
  const uint32_t y = (uint32_t)S.bci[8];
  *margin = S.bci[9] != 0;
  __syncthreads();
  return y;
}

// ---------------------------------------------------------------------------
// The general path: one CTA settles a unit whose kept set needs a global
// threshold (top-p without a small top-k, or a large top-k), in passes over
// the logit row (the first from HBM, later ones mostly from L2).  The kept
// set is a prefix of the total order, described by a Thresh.
// ---------------------------------------------------------------------------

// Index of the n-th (1-based) entry of the row, in index order, whose order
// key is tkey; 0xffffffff when there are fewer.
template <bool kBF16>
__device__ uint32_t nth_tie_index(const Args& A, Shm& S, size_t lrow, uint32_t tkey, unsigned long long n) {
  const int G = (A.V + 7) / 8;
  unsigned long long need = n;
  uint32_t found = 0xffffffffu;
  for (int base = 0; base < G; base += kThreads) {
    const int g = base + threadIdx.x;
    int c = 0;
    float v[8];
    if (g < G) {
      load_group<kBF16>(A, lrow, g, true, v);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (g * 8 + i < A.V && okey(v[i]) == tkey) ++c;
    }
    int inc = c;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    int* wsum = reinterpret_cast<int*>(S.wred);
    if (lane == 31) wsum[w] = inc;
    __syncthreads();
    int woff = 0, rowtot = 0;
    for (int i = 0; i < kWarps; ++i) {
      if (i < w) woff += wsum[i];
      rowtot += wsum[i];
    }
    const int exc = woff + inc - c;
    if (c > 0 && need > (unsigned long long)exc && need <= (unsigned long long)(exc + c)) {
      int want = (int)(need - exc);
      for (int i = 0; i < 8; ++i) {
        if (g * 8 + i < A.V && okey(v[i]) == tkey && --want == 0) {
          S.bci[3] = g * 8 + i;
          break;
        }
      }
    }
    __syncthreads();
    if (need <= (unsigned long long)rowtot) {
      found = (uint32_t)S.bci[3];
      __syncthreads();
      break;
    }
    need -= (unsigned long long)rowtot;
    __syncthreads();
  }
  return found;
}

template <bool kBF16>
__device__ void unit_general(const Args& A, Shm& S, int u, int row, int pos, const RowCfg& cfg) {
  const size_t lrow = (size_t)u * A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const bool has_q = pos < A.k;
  const int G = (A.V + 7) / 8;
  // pass 1: max, argmax, NaN
  unsigned long long best = 0;
  bool nan_seen = false;
  for (int g = threadIdx.x; g < G; g += kThreads) {
    float v[8];
    load_group<kBF16>(A, lrow, g, true, v);
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
  }
  if (nan_seen) best = ~0ull;
  best = block_max_u64(S, best);
  const float m = from_okey((uint32_t)(best >> 32));
  const int am = (int)key64_idx(best);
  if (best == 0 || !(m > -INFINITY) || !(m < INFINITY)) {
    if (threadIdx.x == 0) commit_record(A, u, row, empty_record(SPEC_F_NAN));
    __syncthreads();
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
      for (int g = threadIdx.x; g < G; g += kThreads) {
        float v[8];
        load_group<kBF16>(A, lrow, g, true, v);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (g * 8 + i < A.V) fn(km - kf<kBF16>(v[i]));
      }
    };
    const uint32_t d = kth_distance(S, each, need, kBF16 ? 0 : 16, kBF16 ? 16 : 32);
    th.tkey = full_key<kBF16>(km - d);
    th.tidx = nth_tie_index<kBF16>(A, S, lrow, th.tkey, need);
  }
  const bool topp = cfg.P < 1.0f;

  // Z pass over the top-k set; with top-p also a fixed-point mass histogram
  // binned by log2 of the weight in steps of 1/8 (the last bin in registers).
  const int hslot = 0;
  S.mlo[hslot][threadIdx.x] = 0;
  S.mhi[hslot][threadIdx.x] = 0;
  __syncthreads();
  unsigned long long tail = 0;
  float z0 = 0.f, z1 = 0.f;
  for (int g = threadIdx.x; g < G; g += kThreads) {
    float v[8];
    load_group<kBF16>(A, lrow, g, true, v);
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
  }
  float Zs;
  if (topp) {
    __syncthreads();
    tail = block_sum_u64(S, tail);
    if (threadIdx.x == 0) {
      S.mlo[hslot][255] = (uint32_t)tail;
      S.mhi[hslot][255] = (uint32_t)(tail >> 32);
    }
    __syncthreads();
    S.total[threadIdx.x] = ((unsigned long long)S.mhi[hslot][threadIdx.x] << 32) + S.mlo[hslot][threadIdx.x];
    __syncthreads();
    const unsigned long long zk = block_sum_u64(S, S.total[threadIdx.x]);
    const unsigned long long target = (unsigned long long)ceil((double)cfg.P * (double)zk);
    int b;
    unsigned long long above;
    select_from_bin0(S, target, &b, &above);
    // key range of bin b
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int g = threadIdx.x; g < G; g += kThreads) {
      float v[8];
      load_group<kBF16>(A, lrow, g, true, v);
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
    }
    const uint2 mm = block_minmax_u32(S, kmin, kmax);
    uint32_t lo = mm.x, hi = mm.y;
    unsigned long long rem = target - above;
    int hs = 1;
    while (hi > lo) {
      const uint32_t span = hi - lo;
      const int nbits = 32 - __clz(span);
      const int shift = nbits > 8 ? nbits - 8 : 0;
      const int slot = hs++ & 1;
      S.mlo[slot][threadIdx.x] = 0;
      S.mhi[slot][threadIdx.x] = 0;
      __syncthreads();
      for (int g = threadIdx.x; g < G; g += kThreads) {
        float v[8];
        load_group<kBF16>(A, lrow, g, true, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (g * 8 + i >= A.V) continue;
          const uint32_t key = okey(v[i]);
          if (key < lo || key > hi) continue;
          if (cfg.K > 0 && !kept(th, key, (uint32_t)(g * 8 + i))) continue;
          const uint32_t bin = (hi - key) >> shift;
          mass_add(&S.mlo[slot][bin], &S.mhi[slot][bin], mass_fixed(ex2((v[i] - m) * c)));
        }
      }
      __syncthreads();
      S.total[threadIdx.x] = ((unsigned long long)S.mhi[slot][threadIdx.x] << 32) + S.mlo[slot][threadIdx.x];
      __syncthreads();
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
    const float et = ex2((from_okey(tkey) - m) * c);
    const unsigned long long efx = mass_fixed(et);
    unsigned long long n_need = efx ? (rem + efx - 1) / efx : 1ull;
    if (n_need == 0) n_need = 1;
    // with a top-k threshold at the same key, the ties top-k keeps are a
    // prefix of the ties in index order, so the rank carries over
    th.tidx = nth_tie_index<kBF16>(A, S, lrow, tkey, n_need);
    th.tkey = tkey;
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
    for (int g = threadIdx.x; g < G; g += kThreads) {
      float v[8], qv[8];
      load_group<kBF16>(A, lrow, g, true, v);
      load_q8(A, qrow, g * 8, qv);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const bool in = (g * 8 + i < A.V) && kept(th, okey(v[i]), (uint32_t)(g * 8 + i));
        const float p = in ? ex2((v[i] - m) * c) * invZ : 0.f;
        if (i & 1) al1 += fminf(p, qv[i]); else al0 += fminf(p, qv[i]);
      }
    }
  }
  const float alpha_v = has_q ? block_sum(S, al0 + al1) : 0.f;
  // the draw: residual after a rejection, p at the bonus position
  uint32_t draw_flags = 0;
  uint32_t y = 0xffffffffu;
  if (need_race) {
    bool mg = false;
    y = draw_row<kBF16>(A, S, row, pos, m, c, invZ, has_q ? RW_RESIDUAL : RW_BONUS, &th, &mg);
    if (y == 0xffffffffu) {
      draw_flags |= SPEC_F_RESIDUAL_EMPTY;
      y = draw_row<kBF16>(A, S, row, pos, m, c, invZ, RW_P, &th, &mg);
    }
    if (mg) draw_flags |= SPEC_F_MARGIN_DRAW;
  }
  if (threadIdx.x == 0) {
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

// ---------------------------------------------------------------------------
// Small top-k: the sorted candidate list in S.cand[0..n_k) (the first n_k
// entries of the total order) settles the unit.  CTA-wide; n_k <= 128.
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ void list_unit(const Args& A, Shm& S, int u, int row, int pos, const RowCfg& cfg, float m,
                          int am, int n_k) {
  const bool has_q = pos < A.k;
  const size_t lrow = (size_t)u * A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const int t = threadIdx.x;
  float e = 0.f;
  uint32_t idx = 0;
  if (t < n_k) {
    const unsigned long long key = S.cand[t];
    idx = key64_idx(key);
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
    if (lane == 31) S.wred[w] = inc;
    __syncthreads();
    float off = 0.f;
    for (int i = 0; i < w; ++i) off += S.wred[i];
    if (t < n_k) S.list_cum[t] = off + inc;
    __syncthreads();
  }
  const float Zk = S.list_cum[n_k - 1];
  uint32_t flags = cfg.bad_param ? SPEC_F_BAD_PARAM : 0u;
  int n_s = n_k;
  if (cfg.P < 1.0f) {
    const float target = cfg.P * Zk;
    if (t == 0) S.bci[4] = n_k - 1;
    __syncthreads();
    const bool hit = t < n_k && S.list_cum[t] >= target;
    const unsigned ball = __ballot_sync(0xffffffffu, hit);
    if ((t & 31) == 0 && ball) atomicMin(&S.bci[4], (t & ~31) + __ffs(ball) - 1);
    __syncthreads();
    n_s = S.bci[4] + 1;
    const float at = S.list_cum[n_s - 1] / Zk;
    const float before = n_s >= 2 ? S.list_cum[n_s - 2] / Zk : 0.f;
    if (fabsf(at - cfg.P) < kMargin || fabsf(cfg.P - before) < kMargin) flags |= SPEC_F_MARGIN_TOPP;
  }
  const float Zs = S.list_cum[n_s - 1];
  const float invZ = 1.0f / Zs;
  const float lnZ = logf(Zs);
  const bool mine = t < n_s;
  const float p = mine ? e * invZ : 0.f;
  const float qv = (mine && has_q) ? A.q[qrow + idx] : 0.f;
  int x = -1;
  if (has_q) {
    x = A.drafts[(size_t)row * A.k + pos];
    if (t == 0) S.bci[5] = -1;
    __syncthreads();
    if (mine && idx == (uint32_t)x) S.bci[5] = t;
    __syncthreads();
  }
  const float alpha_v = has_q ? block_sum(S, mine ? fminf(p, qv) : 0.f) : 0.f;
  bool need_race = !has_q;
  AcceptInfo ai;
  ai.valid = true;
  ai.accept = false;
  ai.margin = false;
  ai.lx = 0.f;
  if (has_q) {
    const int xi = S.bci[5];
    ai.x = x;
    ai.valid = x >= 0 && x < A.V;
    ai.px = xi >= 0 ? S.list_e[xi] / Zs : 0.f;
    ai.qx = ai.valid ? A.q[qrow + x] : 0.f;
    ai.lx = ai.valid ? load_logit(A, kBF16, lrow + x) : 0.f;
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
      const Race g1 = block_race(S, r1);
      if (g1.s1 < 0.f) {
        draw_flags |= SPEC_F_RESIDUAL_EMPTY;
        continue;
      }
      // level 2: the entries of the winning block
      Race r2;
      race_init(r2);
      if (mine && w > 0.f && idx / kRaceBlock == g1.v1) race_consider(r2, w, tq, idx, race_word(A, row, pos, idx));
      const Race g2 = block_race(S, r2);
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

__device__ __forceinline__ void race_scale(Race& r, float sc) {
  if (r.s1 >= 0.f) r.s1 *= sc;
  if (r.s2 >= 0.f) r.s2 *= sc;
  r.t1 *= sc;
  r.t2 *= sc;
}

// ---------------------------------------------------------------------------
// A items.
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ void finalize_A(const Args& A, Shm& S, int u, int row, int pos, const RowCfg& cfg);

// Claim the unit's ticket (thread 0) and run the finaliser if this chunk was last.
template <bool kBF16>
__device__ __forceinline__ void chunk_done(const Args& A, Shm& S, int u, int row, int pos, const RowCfg& cfg) {
  if (threadIdx.x == 0) {
    const uint32_t t = atomic_add_acq_rel(&A.a_ticket[u], 1u);
    S.bci[1] = (t == (uint32_t)A.NC - 1u) ? 1 : 0;
  }
  __syncthreads();
  const bool last = S.bci[1] != 0;
  __syncthreads();
  if (last) finalize_A<kBF16>(A, S, u, row, pos, cfg);
}

template <bool kBF16>
__device__ void item_A(const Args& A, Shm& S, int item) {
  const int u = item / A.NC;
  const int c = item - u * A.NC;
  const int row = u / (A.k + 1), pos = u - row * (A.k + 1);
  const size_t lrow = (size_t)u * A.V;
  const int gbase = c * kGPC;
  const int G = (A.V + 7) / 8;
  // the chunk loads go out first (kept in L2: drafted unfiltered units re-read them)
  float v[kGPT][8];
#pragma unroll
  for (int i = 0; i < kGPT; ++i) {
    const int g = gbase + threadIdx.x + i * kThreads;
    if (g < G) {
      load_group<kBF16>(A, lrow, g, true, v[i]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[i][j] = -INFINITY;
    }
  }
  const RowCfg cfg = classify(A.params[row], A.V, A.NC);
  if (cfg.type == UT_GENERAL) {
    if (c == 0) unit_general<kBF16>(A, S, u, row, pos, cfg);
    return;
  }
  if (cfg.type == UT_TOPK) {
    // maxima of super-groups of 64 entries (8 consecutive groups held by 8
    // consecutive lanes); NaN propagates.  The finaliser works from these.
    float* dst = A.smax + ((size_t)u * A.NC + c) * kSPC;
#pragma unroll
    for (int i = 0; i < kGPT; ++i) {
      float gm = group_max(v[i]);
      gm = max_nan(gm, __shfl_xor_sync(0xffffffffu, gm, 1));
      gm = max_nan(gm, __shfl_xor_sync(0xffffffffu, gm, 2));
      gm = max_nan(gm, __shfl_xor_sync(0xffffffffu, gm, 4));
      if ((threadIdx.x & 7) == 0) dst[(threadIdx.x >> 3) + i * (kThreads / 8)] = gm;
    }
    __threadfence();   // every writer publishes before the ticket
    __syncthreads();
    chunk_done<kBF16>(A, S, u, row, pos, cfg);
    return;
  }
  // greedy and unfiltered units.  Each warp-row of 32 groups is one race
  // block: its max, first argmax and softmax sum relative to the block max
  // (warp collectives); warp 0 then folds the chunk's 32 blocks in index
  // order and, at an unfiltered bonus position, races them (level 1).
  const bool bonus_race = cfg.type == UT_DENSE && pos == A.k;
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  bool nan_seen = false;
#pragma unroll
  for (int i = 0; i < kGPT; ++i) {
    const int g = gbase + threadIdx.x + i * kThreads;
    const float gm = group_max(v[i]);
    nan_seen |= gm != gm;
    float mb = gm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = max_nan(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    const unsigned ball = __ballot_sync(0xffffffffu, gm == mb);
    int first = 7;
#pragma unroll
    for (int j = 7; j >= 0; --j)
      if (v[i][j] == gm) first = j;
    const uint32_t idx = __shfl_sync(0xffffffffu, (uint32_t)(g * 8 + first), ball ? __ffs(ball) - 1 : 0);
    float s8 = 0.f;
    if (mb > -INFINITY && mb < INFINITY) {
#pragma unroll
      for (int j = 0; j < 8; ++j) s8 += ex2((v[i][j] - mb) * cfg.c);   // padding is -inf -> 0
    }
    const float W = warp_sum(s8);
    if (lane == 0) {
      S.bm[wp + 8 * i] = mb;
      S.bi[wp + 8 * i] = idx;
      S.bw[wp + 8 * i] = W;
    }
  }
  const bool any_nan = __syncthreads_or(nan_seen) != 0;
  if (wp == 0) {
    const float mb = S.bm[lane];
    const float W = S.bw[lane];
    float mc = mb;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mc = max_nan(mc, __shfl_xor_sync(0xffffffffu, mc, o));
    const unsigned ball = __ballot_sync(0xffffffffu, mb == mc);
    const uint32_t idx = __shfl_sync(0xffffffffu, S.bi[lane], ball ? __ffs(ball) - 1 : 0);
    const bool live = mc > -INFINITY && mc < INFINITY;
    const float Ws = (live && mb > -INFINITY) ? W * ex2((mb - mc) * cfg.c) : 0.f;
    const float z = warp_sum(Ws);
    Race r;
    race_init(r);
    if (bonus_race && Ws > 0.f) {
      const uint32_t b = (uint32_t)(c * (kChunk / kRaceBlock) + lane);
      race_consider(r, Ws, 0.f, b, block_word(A, row, pos, b));
    }
    warp_race_merge(r);
    if (lane == 0) {
      ChunkRec rec;
      rec.m = any_nan ? __uint_as_float(0x7fc00000u) : mc;
      rec.amax = idx;
      rec.z = z;
      rec.nlist = 0;
      rec.overflow = 0;
      rec.s1 = r.s1;
      rec.t1 = r.t1;
      rec.s2 = r.s2;
      rec.t2 = r.t2;
      rec.v1 = r.v1;
      rec.pad[0] = rec.pad[1] = 0;
      A.crec[(size_t)u * A.NC + c] = rec;
    }
  }
  chunk_done<kBF16>(A, S, u, row, pos, cfg);
}

// Small top-k finaliser: every top-K entry lies in a 64-entry super-group
// whose maximum is among the K largest super-group maxima, so the K-th
// largest super-group maximum tau bounds the candidates: the entries >= tau
// of the super-groups whose maximum reaches tau (at least K of them, and at
// most 64 per such super-group).  They are gathered from L2, sorted exactly,
// and the first K settle the unit.
template <bool kBF16>
__device__ void finalize_topk(const Args& A, Shm& S, int u, int row, int pos, const RowCfg& cfg) {
  const int nsm = A.NC * kSPC;
  const float* src = A.smax + (size_t)u * A.NC * kSPC;
  float* sm = reinterpret_cast<float*>(S.cand + kMergeCap / 2);    // second half of the buffer
  unsigned long long* cand = S.cand;                               // first half
  const int G = (A.V + 7) / 8;
  const size_t lrow = (size_t)u * A.V;
  // maxima into shared memory; the unit max; NaN
  unsigned long long best = 0;
  bool nan_seen = false;
  for (int s = threadIdx.x; s < nsm; s += kThreads) {
    const float x = __ldcg(src + s);
    sm[s] = x;
    if (x != x) nan_seen = true;
    else {
      const unsigned long long kk = ((unsigned long long)okey(x) << 32) | (0xffffffffu - (uint32_t)s);
      best = kk > best ? kk : best;
    }
  }
  if (nan_seen) best = ~0ull;
  best = block_max_u64(S, best);
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
    tau = km - kth_distance(S, each, need, kBF16 ? 0 : 16, kBF16 ? 16 : 32);
  }
  // list the qualifying super-groups, then gather their entries >= tau
  int* sg = reinterpret_cast<int*>(S.gmax);   // up to kGPC super-group ids
  if (threadIdx.x == 0) {
    S.cand_count = 0;
    S.bci[6] = 0;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < nsm; s += kThreads) {
    if (kf<kBF16>(sm[s]) >= tau) {
      const int slot = atomicAdd(&S.bci[6], 1);
      if (slot < kGPC) sg[slot] = s;
    }
  }
  __syncthreads();
  const int nsg = S.bci[6];
  bool ovf = nsg > kGPC;
  if (!ovf) {
    for (int e = threadIdx.x; e < nsg * 8; e += kThreads) {
      const int s = sg[e >> 3];
      const int g = s * 8 + (e & 7);      // super-group s covers groups 8s..8s+7
      if (g >= G) continue;
      float v[8];
      load_group<kBF16>(A, lrow, g, true, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (g * 8 + j < A.V && kf<kBF16>(v[j]) >= tau) {
          const uint32_t slot = atomicAdd(&S.cand_count, 1u);
          if (slot < (uint32_t)(kMergeCap / 2)) cand[slot] = key64(okey(v[j]), (uint32_t)(g * 8 + j));
        }
      }
    }
  }
  __syncthreads();
  const uint32_t count = S.cand_count;
  ovf = ovf || count > (uint32_t)(kMergeCap / 2);
  if (ovf) {
    unit_general<kBF16>(A, S, u, row, pos, cfg);
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

// The unit's chunk records, merged in chunk order.
template <bool kBF16>
__device__ void finalize_A(const Args& A, Shm& S, int u, int row, int pos, const RowCfg& cfg) {
  if (threadIdx.x == 0) A.a_ticket[u] = 0;
  if (cfg.type == UT_TOPK) {
    finalize_topk<kBF16>(A, S, u, row, pos, cfg);
    return;
  }
  const ChunkRec* R = A.crec + (size_t)u * A.NC;
  const bool has_q = pos < A.k;
  // chunk maxima -> unit max and argmax (the first chunk holding the max)
  bool nan_any = false;
  float m = -INFINITY;
  int am = -1;
  for (int c = 0; c < A.NC; ++c) {
    const float mc = __ldcg(&R[c].m);
    if (mc != mc) {
      nan_any = true;
    } else if (mc > m) {
      m = mc;
      am = (int)__ldcg(&R[c].amax);
    }
  }
  const bool invalid = nan_any || !(m > -INFINITY) || !(m < INFINITY);
  if (invalid) {
    if (threadIdx.x == 0) {
      if (cfg.type == UT_DENSE && has_q) {
        UnitState st;
        memset(&st, 0, sizeof(st));
        st.invalid = 1;
        A.ust[u] = st;
        store_release(&A.ready[u], 1u);
      }
      commit_record(A, u, row, empty_record(SPEC_F_NAN));
    }
    __syncthreads();
    return;
  }
  // the softmax sum rescaled to the unit max
  float Z = 0.f;
  for (int c = 0; c < A.NC; ++c) {
    const float mc = __ldcg(&R[c].m);
    if (mc > -INFINITY) Z += __ldcg(&R[c].z) * ex2((mc - m) * cfg.c);
  }
  const float lnZ = logf(Z);
  const uint32_t base_flags = cfg.bad_param ? SPEC_F_BAD_PARAM : 0u;
  if (cfg.type == UT_GREEDY) {
    if (threadIdx.x == 0) {
      UnitRecord rec = empty_record(base_flags);
      bool need_draw = !has_q;
      float q_am = 0.f;
      if (has_q) {
        const AcceptInfo ai = accept_test(A, row, pos, kBF16, true, am, m, cfg.c, 1.f, nullptr);
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
    __syncthreads();
    return;
  }
  // UT_DENSE
  if (!has_q) {
    // bonus: merge the chunks' block races (scaled to the unit max), then
    // race the entries of the winning block
    Race a;
    race_init(a);
    for (int c = 0; c < A.NC; ++c) {
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
    if (threadIdx.x < 32) {
      const Race l2 = race_in_block<kBF16>(A, row, pos, a.v1, m, cfg.c, 1.f, RW_BONUS, nullptr);
      if (threadIdx.x == 0) {
        UnitRecord rec = empty_record(base_flags);
        const uint32_t y = l2.v1 < (uint32_t)A.V ? l2.v1 : (uint32_t)am;
        rec.y = (int32_t)y;
        rec.lp_y = (load_logit(A, kBF16, (size_t)u * A.V + y) - m) * cfg.invT - lnZ;
        if (draw_margin(a) || draw_margin(l2)) rec.draw_flags |= SPEC_F_MARGIN_DRAW;
        commit_record(A, u, row, rec);
      }
    }
    __syncthreads();
    return;
  }
  // drafted position: accept test, then publish the state for the B items
  if (threadIdx.x == 0) {
    const AcceptInfo ai = accept_test(A, row, pos, kBF16, false, am, m, cfg.c, Z, nullptr);
    UnitState st;
    memset(&st, 0, sizeof(st));
    st.m = m;
    st.invZ = 1.0f / Z;
    st.lnZ = lnZ;
    st.accept = ai.accept ? 1 : 0;
    st.lp_x = ai.valid ? (ai.lx - m) * cfg.invT - lnZ : 0.f;
    st.flags = base_flags | (ai.valid ? 0u : SPEC_F_BAD_TOKEN) | (ai.margin ? SPEC_F_MARGIN_ACCEPT : 0u);
    st.am = am;
    A.ust[u] = st;
    store_release(&A.ready[u], 1u);
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// B items: alpha and the residual race of drafted unfiltered positions.
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ void item_B(const Args& A, Shm& S, int item) {
  const int ub = item / A.NC;
  const int c = item - ub * A.NC;
  const int row = ub / A.k, pos = ub - row * A.k;
  const int u = row * (A.k + 1) + pos;
  const RowCfg cfg = classify(A.params[row], A.V, A.NC);
  if (cfg.type != UT_DENSE) return;
  const size_t lrow = (size_t)u * A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const int gbase = c * kGPC;
  const int G = (A.V + 7) / 8;
  // the loads do not depend on the unit state: issue them before waiting
  float vv[kGPT][8], qq[kGPT][8];
#pragma unroll
  for (int i = 0; i < kGPT; ++i) {
    const int g = gbase + threadIdx.x + i * kThreads;
    if (g < G) {
      load_group<kBF16>(A, lrow, g, false, vv[i]);
      load_q8(A, qrow, g * 8, qq[i]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        vv[i][j] = -INFINITY;
        qq[i][j] = 0.f;
      }
    }
  }
  // wait for the unit state (bounded; every A item was claimed before any B item)
  if (threadIdx.x == 0) {
    long long spins = 0;
    while (load_acquire(&A.ready[u]) == 0u) {
      if (++spins > kSpinLimit) {
        atomicOr(&A.ws->error, 1u);
        break;
      }
      __nanosleep(64);
    }
  }
  __syncthreads();
  const UnitState* sp = A.ust + u;
  const bool invalid = __ldcg(&sp->invalid) != 0;
  const float m = __ldcg(&sp->m);
  const float invZ = __ldcg(&sp->invZ);
  const bool accept = __ldcg(&sp->accept) != 0;
  const int am = __ldcg(&sp->am);
  const bool need_race = !accept;
  // per race block (warp-row): alpha, residual weight and margin weight
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < kGPT; ++i) {
    float a8 = 0.f, w8 = 0.f, u8 = 0.f;
    if (!invalid) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p = ex2((vv[i][j] - m) * cfg.c) * invZ;   // padding: -inf -> 0
        a8 += fminf(p, qq[i][j]);
        const float w = p - qq[i][j];
        if (w > 0.f) {
          w8 += w;
          u8 += p + qq[i][j];
        }
      }
    }
    const float Ab = warp_sum(a8), Wb = warp_sum(w8), Ub = warp_sum(u8);
    if (lane == 0) {
      S.ba[wp + 8 * i] = Ab;
      S.bw[wp + 8 * i] = Wb;
      S.bu[wp + 8 * i] = Ub;
    }
  }
  __syncthreads();
  // warp 0: alpha over the chunk's blocks (fixed order) and the level-1 race
  Race race;
  race_init(race);
  float alpha_c = 0.f;
  if (wp == 0) {
    alpha_c = warp_sum(S.ba[lane]);
    const float W = S.bw[lane];
    if (need_race && W > 0.f) {
      const uint32_t b = (uint32_t)(c * (kChunk / kRaceBlock) + lane);
      race_consider(race, W, S.bu[lane] - W, b, block_word(A, row, pos, b));
    }
    warp_race_merge(race);
  }
  if (threadIdx.x == 0) {
    BRec br;
    br.alpha = alpha_c;
    br.s1 = race.s1;
    br.t1 = race.t1;
    br.s2 = race.s2;
    br.t2 = race.t2;
    br.v1 = race.v1;
    br.pad[0] = br.pad[1] = 0;
    A.brec[(size_t)u * A.NC + c] = br;
    const uint32_t t = atomic_add_acq_rel(&A.b_ticket[u], 1u);
    S.bci[1] = (t == (uint32_t)A.NC - 1u) ? 1 : 0;
  }
  __syncthreads();
  const bool last = S.bci[1] != 0;
  __syncthreads();
  if (!last) return;
  if (invalid) {   // the A finaliser wrote the record already
    if (threadIdx.x == 0) {
      A.b_ticket[u] = 0;
      A.ready[u] = 0;
    }
    __syncthreads();
    return;
  }
  // last chunk: merge in chunk order and settle the unit
  const BRec* R = A.brec + (size_t)u * A.NC;
  Race a;
  race_init(a);
  float alpha_v = 0.f;
  for (int cc = 0; cc < A.NC; ++cc) {
    alpha_v += __ldcg(&R[cc].alpha);
    if (need_race) {
      Race rb;
      rb.s1 = __ldcg(&R[cc].s1);
      rb.t1 = __ldcg(&R[cc].t1);
      rb.s2 = __ldcg(&R[cc].s2);
      rb.t2 = __ldcg(&R[cc].t2);
      rb.v1 = __ldcg(&R[cc].v1);
      rb.s1lo = 0.f;
      race_merge(a, rb);
    }
  }
  uint32_t draw_flags = 0;
  uint32_t y = 0xffffffffu;
  if (need_race) {
    if (a.s1 >= 0.f) {
      if (threadIdx.x < 32) {
        const Race l2 = race_in_block<kBF16>(A, row, pos, a.v1, m, cfg.c, invZ, RW_RESIDUAL, nullptr);
        if (threadIdx.x == 0) {
          S.bci[8] = (int)l2.v1;
          S.bci[9] = (draw_margin(a) || draw_margin(l2)) ? 1 : 0;
        }
      }
      __syncthreads();
      y = (uint32_t)S.bci[8];
      if (S.bci[9]) draw_flags |= SPEC_F_MARGIN_DRAW;
      __syncthreads();
    } else {
      // empty residual: draw from p over the whole row
      draw_flags |= SPEC_F_RESIDUAL_EMPTY;
      bool mg = false;
      y = draw_row<kBF16>(A, S, row, pos, m, cfg.c, invZ, RW_P, nullptr, &mg);
      if (mg) draw_flags |= SPEC_F_MARGIN_DRAW;
    }
  }
  if (threadIdx.x == 0) {
    UnitRecord rec = empty_record(__ldcg(&sp->flags));
    rec.accept = accept ? 1 : 0;
    rec.lp_x = __ldcg(&sp->lp_x);
    rec.alpha = alpha_v;
    if (need_race) {
      const uint32_t yy = y < (uint32_t)A.V ? y : (uint32_t)am;
      rec.y = (int32_t)yy;
      rec.lp_y = (load_logit(A, kBF16, lrow + yy) - m) * cfg.invT - __ldcg(&sp->lnZ);
      rec.draw_flags = draw_flags;
    }
    A.b_ticket[u] = 0;
    A.ready[u] = 0;
    commit_record(A, u, row, rec);
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// The persistent kernel.
// ---------------------------------------------------------------------------
template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const Args A) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Shm& S = *reinterpret_cast<Shm*>(smem_raw);
  // A items, claimed kClaim at a time; the next batch is fetched one batch ahead
  int next = 0;
  if (threadIdx.x == 0) next = (int)atomicAdd(&A.ws->a_next, (uint32_t)kClaim);
  while (true) {
    if (threadIdx.x == 0) S.bci[15] = next;
    __syncthreads();
    const int first = S.bci[15];
    __syncthreads();
    if (first >= A.NA) break;
    if (threadIdx.x == 0) next = (int)atomicAdd(&A.ws->a_next, (uint32_t)kClaim);
    for (int item = first; item < first + kClaim && item < A.NA; ++item) item_A<kBF16>(A, S, item);
  }
  if (A.NB > 0) {
    if (threadIdx.x == 0) next = (int)atomicAdd(&A.ws->b_next, (uint32_t)kClaim);
    while (true) {
      if (threadIdx.x == 0) S.bci[15] = next;
      __syncthreads();
      const int first = S.bci[15];
      __syncthreads();
      if (first >= A.NB) break;
      if (threadIdx.x == 0) next = (int)atomicAdd(&A.ws->b_next, (uint32_t)kClaim);
      for (int item = first; item < first + kClaim && item < A.NB; ++item) item_B<kBF16>(A, S, item);
    }
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t d = atomicAdd(&A.ws->ctas_done, 1u);
    if (d == (uint32_t)A.n_ctas - 1u) {
      A.ws->a_next = 0u;
      A.ws->b_next = 0u;
      A.ws->ctas_done = 0u;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
template <bool kBF16>
static int plan(int device, int* n_ctas) {
  static std::mutex mu;
  static int cached[64][2];
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return SPEC_E_CUDA;
  if (cached[device][kBF16] > 0) {
    *n_ctas = cached[device][kBF16];
    return SPEC_OK;
  }
  auto kern = verify_kernel<kBF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Shm)) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, sizeof(Shm)) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || per_sm <= 0) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  cached[device][kBF16] = per_sm * sms;
  *n_ctas = per_sm * sms;
  return SPEC_OK;
}

template <bool kBF16>
static int launch(Args A, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  int n = 0;
  const int rc = plan<kBF16>(dev, &n);
  if (rc != SPEC_OK) return rc;
  const long long work = (long long)A.NA + A.NB;
  A.n_ctas = (int)(n < work ? n : work);
  verify_kernel<kBF16><<<A.n_ctas, kThreads, sizeof(Shm), stream>>>(A);
  if (cudaGetLastError() != cudaSuccess) return SPEC_E_CUDA;
  return SPEC_OK;
}

}  // namespace specv

extern "C" size_t spec_verify_workspace_size(int B, int k, int V) {
  if (B < 0 || k < 0 || V < 1) return 0;
  return specv::ws_layout(B, k, V).total;
}

static inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

extern "C" int spec_verify(const void* logits, int logits_dtype, const float* draft_probs,
                           const int32_t* draft_tokens, const spec_params_t* params, uint64_t seed,
                           int B, int k, int V, int32_t* tokens, int32_t* accept_len,
                           float* logprobs, float* alpha, uint32_t* flags, void* workspace,
                           size_t workspace_bytes, void* cuda_stream) {
  if (B < 0 || k < 0 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return SPEC_E_DIM;
  if ((long long)B * (k + 1) > (1ll << 24)) return SPEC_E_DIM;
  if (logits_dtype != SPEC_F32 && logits_dtype != SPEC_BF16) return SPEC_E_DTYPE;
  if (B == 0) return SPEC_OK;
  if (!logits || !params || !tokens || !accept_len || !logprobs || !flags || !workspace)
    return SPEC_E_NULL;
  if (k > 0 && (!draft_probs || !draft_tokens || !alpha)) return SPEC_E_NULL;
  const size_t es = logits_dtype == SPEC_BF16 ? 2 : 4;
  if (!aligned(logits, es) || !aligned(params, 4) || !aligned(tokens, 4) || !aligned(accept_len, 4) ||
      !aligned(logprobs, 4) || !aligned(flags, 4) || !aligned(workspace, 16))
    return SPEC_E_ALIGN;
  if (k > 0 && (!aligned(draft_probs, 4) || !aligned(draft_tokens, 4) || !aligned(alpha, 4)))
    return SPEC_E_ALIGN;
  const specv::Layout L = specv::ws_layout(B, k, V);
  if (workspace_bytes < L.total) return SPEC_E_WORKSPACE;
  const long long items = (long long)B * (k + 1) * ((V + specv::kChunk - 1) / specv::kChunk);
  if (items > 0x7fffffffLL) return SPEC_E_DIM;
  const int arc = specv::check_arch();
  if (arc != SPEC_OK) return arc;

  specv::Args A;
  memset(&A, 0, sizeof(A));
  A.logits = logits;
  A.q = draft_probs;
  A.drafts = draft_tokens;
  A.params = params;
  A.tokens = tokens;
  A.accept_len = accept_len;
  A.logprobs = logprobs;
  A.alpha = alpha;
  A.flags = flags;
  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  A.ws = reinterpret_cast<specv::WsHeader*>(ws);
  A.row_ticket = reinterpret_cast<uint32_t*>(ws + L.row_ticket);
  A.a_ticket = reinterpret_cast<uint32_t*>(ws + L.a_ticket);
  A.b_ticket = reinterpret_cast<uint32_t*>(ws + L.b_ticket);
  A.ready = reinterpret_cast<uint32_t*>(ws + L.ready);
  A.crec = reinterpret_cast<specv::ChunkRec*>(ws + L.crec);
  A.ust = reinterpret_cast<specv::UnitState*>(ws + L.ust);
  A.brec = reinterpret_cast<specv::BRec*>(ws + L.brec);
  A.urec = reinterpret_cast<specv::UnitRecord*>(ws + L.urec);
  A.smax = reinterpret_cast<float*>(ws + L.smax);
  A.key0 = (uint32_t)(seed & 0xffffffffull);
  A.key1 = (uint32_t)(seed >> 32);
  A.B = B;
  A.k = k;
  A.V = V;
  A.NC = (V + specv::kChunk - 1) / specv::kChunk;
  A.U = B * (k + 1);
  A.NA = A.U * A.NC;
  A.NB = B * k * A.NC;
  A.vec_logits = aligned(logits, 16) && ((size_t)V * es) % 16 == 0;
  A.vec_q = k > 0 && aligned(draft_probs, 16) && (V % 4) == 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
  return logits_dtype == SPEC_BF16 ? specv::launch<true>(A, st) : specv::launch<false>(A, st);
}
