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
// Execution model.  One (row, position) pair is a "unit".  A persistent grid
// of thread-block clusters (C CTAs each, C chosen from V) pulls units from a
// queue in the workspace.  The C CTAs of a cluster split the unit's
// vocabulary into C slices and stage their slice of the logits in shared
// memory with 128-bit loads; every later pass over the logits reads shared
// memory, and cross-CTA reductions go through distributed shared memory
// (DSMEM) with a fixed combination order, so results are bit-reproducible.
// Each unit decides its own draft's acceptance and, when its draft is
// rejected (or it is the bonus position), runs the exponential race that
// draws the token at that position.  The last unit of a row to finish (an
// atomic ticket, no waiting) resolves the accept chain and writes the row's
// outputs.  Nothing waits on another CTA except through cluster barriers.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/spec_verify.h"
#include "spec_device.cuh"
#include "spec_host.h"

namespace specv {

constexpr int kCandCap = 1024;       // candidate buffer of the small top-k path
constexpr int kTopkSmall = 128;      // top_k <= this uses the candidate path
constexpr int kMaxC = 16;
constexpr int kQD = 3;               // depth of the per-thread q prefetch ring

struct WsHeader {
  uint32_t queue_next;
  uint32_t clusters_done;
  uint32_t pad[62];
};

struct UnitRecord {       // 32 bytes, one per (row, position)
  uint32_t flags;         // F_NAN | F_BAD_PARAM | F_BAD_TOKEN | F_MARGIN_TOPP | F_MARGIN_ACCEPT
  int32_t accept;         // 1 if this position's draft was accepted
  float lp_x;             // logprob of the draft token (j < k)
  float alpha;            // alpha_j (j < k)
  int32_t y;              // token drawn at this position, -1 if not drawn
  float lp_y;             // logprob of y
  uint32_t draw_flags;    // F_MARGIN_DRAW | F_RESIDUAL_EMPTY of this position's draw
  uint32_t pad;
};

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
  uint32_t* tickets;
  UnitRecord* recs;
  uint32_t key0, key1;
  int B, k, V;
  int C;
  int groups_total;   // ceil(V / 8)
  int slice_groups;   // groups per CTA (last CTA may have fewer)
  int n_units;
  int n_clusters;
  int vec_logits;     // 16-byte vector loads allowed on logit rows
  int vec_q;          // 16-byte vector loads allowed on q rows
};

// Shared-memory control block (the staged slice and the arrays follow it).
struct alignas(16) Ctl {
  unsigned long long xch[2][8];          // cluster exchange (published per CTA)
  uint32_t hist[2][256];                 // counts (double buffered)
  uint32_t mlo[2][256];                  // fixed-point mass, low words (double buffered)
  uint32_t mhi[2][256];                  // fixed-point mass, high words
  unsigned long long total[256];         // block- or cluster-reduced histogram
  unsigned long long bc64[8];            // block broadcast
  float wred[kWarps * 8];                // warp partials
  float bcf[8];
  int bci[8];
  int unit;                              // next unit (written by the cluster leader)
  uint32_t cand_count;                   // leader: candidates appended by the cluster
};

struct Smem {
  Ctl* ctl;
  unsigned char* slice;       // staged logits (raw dtype), slice_groups * 8 elements
  float* gmax;                // per-group maximum
  unsigned long long* cand;   // candidate keys (leader)
  float* list_e;              // leader: e of the kept candidates
  float* list_cum;            // leader: prefix sums
  float* qring;               // kQD x kThreads x 8 floats: per-thread q prefetch ring
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <bool kBF16>
__host__ __device__ inline size_t smem_bytes(int slice_groups) {
  size_t off = align_up(sizeof(Ctl), 128);
  off += align_up((size_t)slice_groups * 8 * (kBF16 ? 2 : 4), 128);
  size_t gm = (size_t)slice_groups * 4;
  size_t lists = (size_t)2 * kTopkSmall * 4;
  off += align_up(gm > lists ? gm : lists, 128);
  off += (size_t)kCandCap * 8;
  off += (size_t)kQD * kThreads * 8 * 4;
  return off;
}

template <bool kBF16>
__device__ inline Smem carve(unsigned char* base, int slice_groups) {
  Smem s;
  size_t off = 0;
  s.ctl = reinterpret_cast<Ctl*>(base);
  off = align_up(sizeof(Ctl), 128);
  s.slice = base + off;
  off += align_up((size_t)slice_groups * 8 * (kBF16 ? 2 : 4), 128);
  s.gmax = reinterpret_cast<float*>(base + off);
  s.list_e = s.gmax;                  // the leader reuses its group maxima area
  s.list_cum = s.gmax + kTopkSmall;
  size_t gm = (size_t)slice_groups * 4;
  size_t lists = (size_t)2 * kTopkSmall * 4;
  off += align_up(gm > lists ? gm : lists, 128);
  s.cand = reinterpret_cast<unsigned long long*>(base + off);
  off += (size_t)kCandCap * 8;
  s.qring = reinterpret_cast<float*>(base + off);
  return s;
}

// ---------------------------------------------------------------------------
// Per-CTA view of the current unit.
// ---------------------------------------------------------------------------
struct Unit {
  int row, pos;
  int rank, C;
  int g0, ng;            // first global group of this CTA's slice, number of groups
  bool greedy;
  bool bad_param;
  int K;                 // active top-k (0 = off)
  float P;               // active top-p (1 = off)
  float T, c, invT;      // temperature, log2(e)/T, 1/T
  size_t lrow;           // element offset of this unit's logit row
  size_t qrow;           // element offset of this unit's q row (pos < k)
};

template <bool kBF16>
__device__ __forceinline__ void load_group_values(const Smem& S, int gl, float v[8]) {
  if (kBF16) {
    const uint4 w = reinterpret_cast<const uint4*>(S.slice)[gl];
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
    v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
    v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
  } else {
    const float4 a = reinterpret_cast<const float4*>(S.slice)[2 * gl];
    const float4 b = reinterpret_cast<const float4*>(S.slice)[2 * gl + 1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

__device__ __forceinline__ float load_logit_global(const Args& A, bool bf16, size_t off) {
  if (bf16) {
    const uint16_t h = reinterpret_cast<const uint16_t*>(A.logits)[off];
    return __uint_as_float((uint32_t)h << 16);
  }
  return reinterpret_cast<const float*>(A.logits)[off];
}

// ---------------------------------------------------------------------------
// Cluster helpers.  Each reduction publishes one value per CTA into xch[slot]
// (slots alternate, and every reduction is followed by another cluster
// barrier before its slot is reused), then warp 0 gathers the C values in
// rank order and combines them with a fixed xor tree.
// ---------------------------------------------------------------------------
struct Cluster {
  cg::cluster_group cl;
  int C, rank;
  int step;
};

template <typename T>
__device__ __forceinline__ T* remote(Cluster& K, T* p, int r) {
  return K.cl.map_shared_rank(p, r);
}

// Publish v (thread 0's value) and return the cluster maximum (u64).
__device__ unsigned long long cl_max_u64(Cluster& K, Smem& S, unsigned long long v) {
  const int slot = K.step++ & 1;
  if (threadIdx.x == 0) S.ctl->xch[slot][0] = v;
  K.cl.sync();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    unsigned long long x = 0;
    if (lane < K.C) x = *remote(K, &S.ctl->xch[slot][0], lane);
    x = warp_max_u64(x);
    if (lane == 0) S.ctl->bc64[0] = x;
  }
  __syncthreads();
  return S.ctl->bc64[0];
}

__device__ unsigned long long cl_sum_u64(Cluster& K, Smem& S, unsigned long long v) {
  const int slot = K.step++ & 1;
  if (threadIdx.x == 0) S.ctl->xch[slot][0] = v;
  K.cl.sync();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    unsigned long long x = 0;
    if (lane < K.C) x = *remote(K, &S.ctl->xch[slot][0], lane);
    x = warp_sum_u64(x);
    if (lane == 0) S.ctl->bc64[0] = x;
  }
  __syncthreads();
  return S.ctl->bc64[0];
}

// Sums two floats across the cluster (fixed order).
__device__ float2 cl_sum_f2(Cluster& K, Smem& S, float a, float b) {
  const int slot = K.step++ & 1;
  if (threadIdx.x == 0) {
    S.ctl->xch[slot][0] = __float_as_uint(a);
    S.ctl->xch[slot][1] = __float_as_uint(b);
  }
  K.cl.sync();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float x = 0.f, y = 0.f;
    if (lane < K.C) {
      x = __uint_as_float((uint32_t)*remote(K, &S.ctl->xch[slot][0], lane));
      y = __uint_as_float((uint32_t)*remote(K, &S.ctl->xch[slot][1], lane));
    }
    x = warp_sum(x);
    y = warp_sum(y);
    if (lane == 0) {
      S.ctl->bcf[0] = x;
      S.ctl->bcf[1] = y;
    }
  }
  __syncthreads();
  return make_float2(S.ctl->bcf[0], S.ctl->bcf[1]);
}

// Cluster min and max of two u32 values published by thread 0.
__device__ uint2 cl_minmax_u32(Cluster& K, Smem& S, uint32_t mn, uint32_t mx) {
  const int slot = K.step++ & 1;
  if (threadIdx.x == 0) S.ctl->xch[slot][0] = ((unsigned long long)(~mn) << 32) | mx;
  K.cl.sync();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t a = 0, b = 0;
    if (lane < K.C) {
      const unsigned long long x = *remote(K, &S.ctl->xch[slot][0], lane);
      a = (uint32_t)(x >> 32);
      b = (uint32_t)x;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
      b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    if (lane == 0) {
      S.ctl->bci[0] = (int)~a;
      S.ctl->bci[1] = (int)b;
    }
  }
  __syncthreads();
  return make_uint2((uint32_t)S.ctl->bci[0], (uint32_t)S.ctl->bci[1]);
}

// Race state merged over the cluster.
__device__ Race cl_race(Cluster& K, Smem& S, const Race& mine) {
  const int slot = K.step++ & 1;
  if (threadIdx.x == 0) {
    S.ctl->xch[slot][0] = __float_as_uint(mine.s1);
    S.ctl->xch[slot][1] = __float_as_uint(mine.t1);
    S.ctl->xch[slot][2] = __float_as_uint(mine.s2);
    S.ctl->xch[slot][3] = __float_as_uint(mine.t2);
    S.ctl->xch[slot][4] = mine.v1;
  }
  K.cl.sync();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    Race r;
    race_init(r);
    if (lane < K.C) {
      r.s1 = __uint_as_float((uint32_t)*remote(K, &S.ctl->xch[slot][0], lane));
      r.t1 = __uint_as_float((uint32_t)*remote(K, &S.ctl->xch[slot][1], lane));
      r.s2 = __uint_as_float((uint32_t)*remote(K, &S.ctl->xch[slot][2], lane));
      r.t2 = __uint_as_float((uint32_t)*remote(K, &S.ctl->xch[slot][3], lane));
      r.v1 = (uint32_t)*remote(K, &S.ctl->xch[slot][4], lane);
    }
    warp_race_merge(r);
    if (lane == 0) {
      S.ctl->bcf[0] = r.s1;
      S.ctl->bcf[1] = r.t1;
      S.ctl->bcf[2] = r.s2;
      S.ctl->bcf[3] = r.t2;
      S.ctl->bci[0] = (int)r.v1;
    }
  }
  __syncthreads();
  Race o;
  o.s1 = S.ctl->bcf[0];
  o.t1 = S.ctl->bcf[1];
  o.s2 = S.ctl->bcf[2];
  o.t2 = S.ctl->bcf[3];
  o.v1 = (uint32_t)S.ctl->bci[0];
  o.s1lo = 0.f;
  return o;
}

// Sum a 256-bin histogram over the cluster into S.ctl->total (every CTA gets
// the same totals).  The caller must have filled hist[slot] and synced the block.
__device__ void cl_hist(Cluster& K, Smem& S, int slot, bool mass = false) {
  K.cl.sync();
  const int t = threadIdx.x;
  unsigned long long s = 0;
  for (int r = 0; r < K.C; ++r) {
    if (mass) {
      const unsigned long long lo = *remote(K, &S.ctl->mlo[slot][t], r);
      const unsigned long long hi = *remote(K, &S.ctl->mhi[slot][t], r);
      s += (hi << 32) + lo;
    } else {
      s += *remote(K, &S.ctl->hist[slot][t], r);
    }
  }
  S.ctl->total[t] = s;
  __syncthreads();
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
// Block reductions (fixed order).
// ---------------------------------------------------------------------------
__device__ float2 block_sum_f2(Smem& S, float a, float b) {
  a = warp_sum(a);
  b = warp_sum(b);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    S.ctl->wred[w] = a;
    S.ctl->wred[kWarps + w] = b;
  }
  __syncthreads();
  float x = 0.f, y = 0.f;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kWarps; ++i) {
      x += S.ctl->wred[i];
      y += S.ctl->wred[kWarps + i];
    }
  }
  __syncthreads();
  return make_float2(x, y);   // valid in thread 0
}

__device__ unsigned long long block_max_u64(Smem& S, unsigned long long v) {
  v = warp_max_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  unsigned long long* buf = reinterpret_cast<unsigned long long*>(S.ctl->wred);
  if (l == 0) buf[w] = v;
  __syncthreads();
  unsigned long long x = 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kWarps; ++i) x = buf[i] > x ? buf[i] : x;
  __syncthreads();
  return x;
}

__device__ unsigned long long block_sum_u64(Smem& S, unsigned long long v) {
  v = warp_sum_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  unsigned long long* buf = reinterpret_cast<unsigned long long*>(S.ctl->wred);
  if (l == 0) buf[w] = v;
  __syncthreads();
  unsigned long long x = 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kWarps; ++i) x += buf[i];
  __syncthreads();
  return x;
}

__device__ void block_race(Smem& S, Race& r) {
  warp_race_merge(r);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  float* f = S.ctl->wred;   // 8 warps x 5 floats fits in wred (64 floats)
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
    r = a;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Histogram selection helpers.
// Given totals[256] (bins ordered so that larger bin index = larger key),
// find the bin b where the cumulative count from the top reaches `need`;
// returns b and the mass strictly above it.  Run by warp 0; result broadcast.
// ---------------------------------------------------------------------------
__device__ void select_from_top(Smem& S, unsigned long long need, int* out_bin,
                                unsigned long long* out_above, const unsigned long long* bins = nullptr) {
  const unsigned long long* tot = bins ? bins : S.ctl->total;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    // lane l owns bins 255-8l .. 248-8l (descending)
    unsigned long long own = 0;
    for (int i = 0; i < 8; ++i) own += tot[255 - 8 * lane - i];
    // inclusive scan over lanes (lane 0 = top bins)
    unsigned long long inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const unsigned long long exc = inc - own;
    const unsigned ball = __ballot_sync(0xffffffffu, inc >= need);
    int src = ball ? (__ffs(ball) - 1) : 31;
    if (lane == src) {
      unsigned long long above = exc;
      int b = 255 - 8 * lane;
      int chosen = 248 - 8 * lane;   // fallback: lowest bin of the lane
      for (int i = 0; i < 8; ++i) {
        const unsigned long long t = tot[b - i];
        if (above + t >= need) { chosen = b - i; break; }
        if (i == 7) { chosen = b - i; break; }
        above += t;
      }
      S.ctl->bci[2] = chosen;
      S.ctl->bc64[1] = above;
    }
  }
  __syncthreads();
  *out_bin = S.ctl->bci[2];
  *out_above = S.ctl->bc64[1];
  __syncthreads();
}

// Same, with bins ordered so that bin 0 is the top (largest values first).
__device__ void select_from_bin0(Smem& S, unsigned long long need, int* out_bin,
                                 unsigned long long* out_above) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    unsigned long long own = 0;
    for (int i = 0; i < 8; ++i) own += S.ctl->total[8 * lane + i];
    unsigned long long inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const unsigned long long exc = inc - own;
    const unsigned ball = __ballot_sync(0xffffffffu, inc >= need);
    int src = ball ? (__ffs(ball) - 1) : 31;
    if (lane == src) {
      unsigned long long above = exc;
      int chosen = 8 * lane + 7;
      for (int i = 0; i < 8; ++i) {
        const unsigned long long t = S.ctl->total[8 * lane + i];
        if (above + t >= need || i == 7) { chosen = 8 * lane + i; break; }
        above += t;
      }
      S.ctl->bci[2] = chosen;
      S.ctl->bc64[1] = above;
    }
  }
  __syncthreads();
  *out_bin = S.ctl->bci[2];
  *out_above = S.ctl->bc64[1];
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Rank select on distances from the maximum.  Values are described by their
// distance d = key(max) - key(v) >= 0 in the order-key space (key = the 16-bit
// bf16 pattern order or the 32-bit float order), so the largest values have
// the smallest distances.  kth_distance finds the distance of the value of
// 1-based rank `need` (counting multiplicity) among the values that `each`
// enumerates (per CTA, or over the whole cluster when kCluster).  The first
// histogram gives every distance below 255 << s0 a bin and lumps the tail
// without touching it, so only values near the top cost an atomic; the
// selected bin is refined 8 bits at a time.  If the rank lies in the tail, a
// plain top-down radix over all bits takes over.  On return `need` is the
// rank inside the group of values at exactly that distance.
// ---------------------------------------------------------------------------
template <bool kCluster, typename Each>
__device__ uint32_t kth_distance(Cluster& K, Smem& S, Each each, unsigned long long& need, int s0,
                                 int dbits, int& hs) {
  auto reduce = [&](int slot) {
    if (kCluster) {
      cl_hist(K, S, slot);
    } else {
      S.ctl->total[threadIdx.x] = S.ctl->hist[slot][threadIdx.x];
      __syncthreads();
    }
  };
  // level 1: exact near-top bins, tail lumped
  {
    const int slot = hs++ & 1;
    S.ctl->hist[slot][threadIdx.x] = 0;
    __syncthreads();
    const uint32_t lim = 255u << s0;
    each([&](uint32_t d) {
      if (d < lim) atomicAdd(&S.ctl->hist[slot][d >> s0], 1u);
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
        S.ctl->hist[sl][threadIdx.x] = 0;
        __syncthreads();
        const uint32_t span = 1u << (s + 8);
        each([&](uint32_t d) {
          if (d >= base && d - base < span) atomicAdd(&S.ctl->hist[sl][(d - base) >> s], 1u);
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
  // tail: top-down radix over all distance bits
  uint32_t prefix = 0u, mask = 0u;
  for (int shift = dbits - 8; shift >= 0; shift -= 8) {
    const int slot = hs++ & 1;
    S.ctl->hist[slot][threadIdx.x] = 0;
    __syncthreads();
    each([&](uint32_t d) {
      if ((d & mask) == prefix) atomicAdd(&S.ctl->hist[slot][(d >> shift) & 255u], 1u);
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
// Full 32-bit order key of the value whose kf() is k.
template <bool kBF16>
__device__ __forceinline__ uint32_t full_key(uint32_t k) {
  if (!kBF16) return k;
  return (k << 16) | ((k & 0x8000u) ? 0u : 0xffffu);
}

// ---------------------------------------------------------------------------
// Kept-set description.  v is kept iff key(v) > tkey, or key(v) == tkey and
// v <= tidx.  tkey = 0 keeps every non-NaN value.
// ---------------------------------------------------------------------------
struct Thresh {
  uint32_t tkey;
  uint32_t tidx;
};
__device__ __forceinline__ bool kept(const Thresh& t, uint32_t key, uint32_t v) {
  return key > t.tkey || (key == t.tkey && v <= t.tidx);
}

// Index of the n-th (1-based) element in index order with key == tkey among
// the elements kept by `outer`.  Cluster-wide; every CTA runs the same
// barriers.  Returns 0xffffffff when n exceeds the number of such elements.
template <bool kBF16>
__device__ uint32_t nth_tie_index(Cluster& K, Smem& S, const Unit& U, const Args& A,
                                  uint32_t tkey, unsigned long long n) {
  // 1. count ties in this CTA
  unsigned long long cnt = 0;
  for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) {
    float v[8];
    load_group_values<kBF16>(S, gl, v);
    const int e0 = (U.g0 + gl) * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (e0 + i < A.V && okey(v[i]) == tkey) ++cnt;
  }
  cnt = block_sum_u64(S, cnt);
  // 2. exchange counts: every CTA learns the counts of lower ranks
  const int slot = K.step++ & 1;
  if (threadIdx.x == 0) S.ctl->xch[slot][0] = cnt;
  K.cl.sync();
  unsigned long long before = 0;
  for (int r = 0; r < K.rank; ++r) before += *remote(K, &S.ctl->xch[slot][0], r);
  cnt = *remote(K, &S.ctl->xch[slot][0], K.rank);
  uint32_t found = 0xffffffffu;
  if (n > before && n <= before + cnt) {
    // 3. ordered scan of this CTA's groups, one row of kThreads groups at a time
    unsigned long long need = n - before;
    for (int base = 0; base < U.ng; base += kThreads) {
      const int gl = base + threadIdx.x;
      int c = 0;
      float v[8];
      if (gl < U.ng) {
        load_group_values<kBF16>(S, gl, v);
        const int e0 = (U.g0 + gl) * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (e0 + i < A.V && okey(v[i]) == tkey) ++c;
      }
      // block exclusive scan of c (thread order = index order)
      int inc = c;
      const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      int* wsum = reinterpret_cast<int*>(S.ctl->wred);
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
        const int e0 = (U.g0 + gl) * 8;
        for (int i = 0; i < 8; ++i) {
          if (e0 + i < A.V && okey(v[i]) == tkey) {
            if (--want == 0) {
              S.ctl->bci[3] = e0 + i;
              break;
            }
          }
        }
      }
      __syncthreads();
      if (need <= (unsigned long long)rowtot) {
        found = (uint32_t)S.ctl->bci[3];
        break;
      }
      need -= rowtot;
      __syncthreads();
    }
  }
  // 4. cluster min of the found index
  __syncthreads();
  const uint2 mm = cl_minmax_u32(K, S, found, 0u);
  return mm.x;
}

// The first `need` elements of the total order (top-k over the whole unit):
// the exact value by kth_distance over the cluster, then the index cut inside
// that value's ties.
template <bool kBF16>
__device__ Thresh select_count(Cluster& K, Smem& S, const Unit& U, const Args& A, float m,
                               unsigned long long need) {
  const uint32_t km = kf<kBF16>(m);
  auto each = [&](auto fn) {
    for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) {
      float v[8];
      load_group_values<kBF16>(S, gl, v);
      const int e0 = (U.g0 + gl) * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (e0 + i < A.V) fn(km - kf<kBF16>(v[i]));
    }
  };
  int hs = 0;
  const uint32_t d = kth_distance<true>(K, S, each, need, kBF16 ? 0 : 16, kBF16 ? 16 : 32, hs);
  Thresh t;
  t.tkey = full_key<kBF16>(km - d);
  t.tidx = nth_tie_index<kBF16>(K, S, U, A, t.tkey, need);
  return t;
}

// ---------------------------------------------------------------------------
// Unit bookkeeping: records and the per-row finalize.
// ---------------------------------------------------------------------------
__device__ void finalize_row(const Args& A, int row) {
  const int k = A.k;
  const UnitRecord* R = A.recs + (size_t)row * (k + 1);
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
    const uint32_t f = __ldcg(&R[j].flags);
    uflags |= f & SPEC_F_MARGIN_ACCEPT;
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

// Thread 0 of the cluster leader: publish the record and finalize the row if
// this was its last unit.
__device__ void commit_record(const Args& A, const Unit& U, const UnitRecord& rec) {
  UnitRecord* dst = A.recs + (size_t)U.row * (A.k + 1) + U.pos;
  *dst = rec;
  __threadfence();
  const uint32_t old = atomicAdd(&A.tickets[U.row], 1u);
  if (old == (uint32_t)A.k) {
    __threadfence();
    finalize_row(A, U.row);
    A.tickets[U.row] = 0;   // leave the workspace clean for the next call
  }
}

// Accept test of draft x at this unit (identical in every CTA of the cluster).
struct AcceptInfo {
  bool valid;
  int x;
  float px, qx;
  bool accept;
  bool margin;
  float lx;     // logit of x
};

__device__ AcceptInfo accept_test(const Args& A, const Unit& U, bool bf16, float m, float px_num,
                                  bool x_kept, float Zs, bool greedy, int am) {
  AcceptInfo ai;
  ai.x = A.drafts[(size_t)U.row * A.k + U.pos];
  ai.valid = ai.x >= 0 && ai.x < A.V;
  ai.lx = 0.f;
  ai.px = 0.f;
  ai.qx = 0.f;
  if (ai.valid) {
    ai.lx = load_logit_global(A, bf16, U.lrow + ai.x);
    ai.qx = A.q[U.qrow + ai.x];
    if (greedy) ai.px = (ai.x == am) ? 1.0f : 0.0f;
    else ai.px = x_kept ? px_num / Zs : 0.0f;
  }
  const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)U.pos, (uint32_t)U.row, 0u), A.key0, A.key1);
  const float u = uniform_of(w.x);
  const float d = fmaf(u, ai.qx, -ai.px);   // exact sign of u*q - p
  ai.accept = d < 0.0f;
  ai.margin = (ai.px > 0.0f && ai.px < 1.0f && fabsf(d) < kMargin);
  (void)m;
  return ai;
}

// ---------------------------------------------------------------------------
// The small top-k path, per CTA: every top-K element of the slice lies in a
// group whose maximum is among the K largest group maxima of the slice, so
// the K-th largest local group maximum tau bounds the local candidates
// (elements >= tau, at most 8 per qualifying group).  They are sorted exactly
// in the total order; the first K form the CTA's list.  Returns the list
// length; *overflow is set when the candidates do not fit the buffer.
// ---------------------------------------------------------------------------
__device__ void bitonic_desc(unsigned long long* s, int n);

template <bool kBF16>
__device__ int local_topk(Cluster& K, Smem& S, const Unit& U, const Args& A, float m, int Ktop,
                          bool* overflow) {
  // tau: kf() of the K-th largest group maximum of this CTA (all groups when fewer)
  uint32_t tau = 0u;
  const uint32_t km = kf<kBF16>(m);
  if (Ktop < U.ng) {
    unsigned long long need = (unsigned long long)Ktop;
    auto each = [&](auto fn) {
      for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) fn(km - kf<kBF16>(S.gmax[gl]));
    };
    int hs = 0;
    const uint32_t d = kth_distance<false>(K, S, each, need, kBF16 ? 0 : 16, kBF16 ? 16 : 32, hs);
    tau = km - d;
  }
  if (threadIdx.x == 0) S.ctl->cand_count = 0;
  __syncthreads();
  for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) {
    if (kf<kBF16>(S.gmax[gl]) < tau) continue;
    float v[8];
    load_group_values<kBF16>(S, gl, v);
    const int e0 = (U.g0 + gl) * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t key = okey(v[i]);
      if (e0 + i < A.V && kf<kBF16>(v[i]) >= tau) {
        const uint32_t slot = atomicAdd(&S.ctl->cand_count, 1u);
        if (slot < (uint32_t)kCandCap) S.cand[slot] = key64(key, (uint32_t)(e0 + i));
      }
    }
  }
  __syncthreads();
  const uint32_t count = S.ctl->cand_count;
  *overflow = count > (uint32_t)kCandCap;
  if (*overflow || count == 0) return 0;
  int n = 1;
  while (n < (int)count) n <<= 1;
  for (int i = (int)count + threadIdx.x; i < n; i += kThreads) S.cand[i] = 0ull;
  __syncthreads();
  bitonic_desc(S.cand, n);
  return min((int)count, Ktop);
}

// Number of entries of a descending list greater than key.
__device__ __forceinline__ int count_greater(const unsigned long long* l, int n, unsigned long long key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (l[mid] > key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Leader: merge the C sorted per-CTA lists into the first Ktop entries of
// S.cand (ranks by binary search; keys are unique).  Returns the list length.
__device__ int merge_lists(Cluster& K, Smem& S, const int* counts, int Ktop) {
  unsigned long long* mb = reinterpret_cast<unsigned long long*>(S.slice);
  int off[kMaxC + 1];
  off[0] = 0;
  for (int c = 0; c < K.C; ++c) off[c + 1] = off[c] + counts[c];
  const int total = off[K.C];
  for (int c = 0; c < K.C; ++c) {
    const unsigned long long* src = remote(K, S.cand, c);
    for (int i = threadIdx.x; i < counts[c]; i += kThreads) mb[off[c] + i] = src[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < total; e += kThreads) {
    int c = 0;
    while (e >= off[c + 1]) ++c;
    const unsigned long long key = mb[e];
    int rank = e - off[c];
    for (int d = 0; d < K.C && rank < Ktop; ++d)
      if (d != c) rank += count_greater(mb + off[d], counts[d], key);
    if (rank < Ktop) S.cand[rank] = key;
  }
  __syncthreads();
  return min(total, Ktop);
}

// Bitonic sort of cand[0..n) descending (n a power of two), one CTA.
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

// Leader-only processing of the sorted candidate list (warp 0).
template <bool kBF16>
__device__ void list_unit(Smem& S, const Unit& U, const Args& A, float m, int am, int n_k,
                          uint32_t base_flags) {
  const int lane = threadIdx.x & 31;
  const bool has_q = U.pos < A.k;
  // e_i and prefix sums in the total order
  float running = 0.f;
  for (int base = 0; base < n_k; base += 32) {
    const int i = base + lane;
    float e = 0.f;
    if (i < n_k) {
      const float val = from_okey((uint32_t)(S.cand[i] >> 32));
      e = ex2((val - m) * U.c);
      S.list_e[i] = e;
    }
    float inc = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (i < n_k) S.list_cum[i] = running + inc;
    running += __shfl_sync(0xffffffffu, inc, 31);
  }
  __syncwarp();
  const float Zk = running;
  int n_s = n_k;
  uint32_t flags = base_flags;
  if (U.P < 1.0f) {
    const float target = U.P * Zk;
    int first = n_k - 1;
    for (int base = 0; base < n_k; base += 32) {
      const int i = base + lane;
      const unsigned ball = __ballot_sync(0xffffffffu, i < n_k && S.list_cum[i] >= target);
      if (ball) {
        first = base + __ffs(ball) - 1;
        break;
      }
    }
    n_s = first + 1;
    const float at = S.list_cum[n_s - 1] / Zk;
    const float before = n_s >= 2 ? S.list_cum[n_s - 2] / Zk : 0.f;
    if (fabsf(at - U.P) < kMargin || fabsf(U.P - before) < kMargin) flags |= SPEC_F_MARGIN_TOPP;
  }
  const float Zs = S.list_cum[n_s - 1];
  const float invZ = 1.0f / Zs;
  const float lnZ = logf(Zs);

  // membership of the draft token and alpha
  UnitRecord rec;
  rec.flags = flags;
  rec.accept = 0;
  rec.lp_x = 0.f;
  rec.alpha = 0.f;
  rec.y = -1;
  rec.lp_y = 0.f;
  rec.draw_flags = 0;
  rec.pad = 0;
  bool need_draw = !has_q;
  AcceptInfo ai;
  if (has_q) {
    const int x = A.drafts[(size_t)U.row * A.k + U.pos];
    int xi = -1;
    for (int base = 0; base < n_s; base += 32) {
      const int i = base + lane;
      const unsigned ball =
          __ballot_sync(0xffffffffu, i < n_s && key64_idx(S.cand[i]) == (uint32_t)x);
      if (ball) {
        xi = base + __ffs(ball) - 1;
        break;
      }
    }
    const float ex = xi >= 0 ? S.list_e[xi] : 0.f;
    ai = accept_test(A, U, kBF16, m, ex, xi >= 0, Zs, false, am);
    if (ai.valid == false) rec.flags |= SPEC_F_BAD_TOKEN;
    rec.accept = ai.accept ? 1 : 0;
    if (ai.margin) rec.flags |= SPEC_F_MARGIN_ACCEPT;
    rec.lp_x = ai.valid ? (ai.lx - m) * U.invT - lnZ : 0.f;
    float al = 0.f;
    for (int i = lane; i < n_s; i += 32) {
      const float p = S.list_e[i] * invZ;
      const float qv = A.q[U.qrow + key64_idx(S.cand[i])];
      al += fminf(p, qv);
    }
    rec.alpha = warp_sum(al);
    need_draw = !ai.accept;
  }
  if (need_draw) {
    Race r;
    race_init(r);
    bool any = false;
    for (int i = lane; i < n_s; i += 32) {
      const uint32_t v = key64_idx(S.cand[i]);
      const float p = S.list_e[i] * invZ;
      const float qv = has_q ? A.q[U.qrow + v] : 0.f;
      const float w = has_q ? fmaxf(p - qv, 0.f) : p;
      if (w > 0.f) {
        any = true;
        const uint4 ww = philox4x32_10(make_uint4(v >> 2, (uint32_t)U.pos, (uint32_t)U.row, 1u), A.key0, A.key1);
        race_consider(r, w, 2.0f * qv, v, word_of(ww, v & 3));
      }
    }
    any = __any_sync(0xffffffffu, any);
    if (!any) {
      rec.draw_flags |= SPEC_F_RESIDUAL_EMPTY;
      for (int i = lane; i < n_s; i += 32) {
        const uint32_t v = key64_idx(S.cand[i]);
        const float p = S.list_e[i] * invZ;
        const uint4 ww = philox4x32_10(make_uint4(v >> 2, (uint32_t)U.pos, (uint32_t)U.row, 1u), A.key0, A.key1);
        race_consider(r, p, 0.f, v, word_of(ww, v & 3));
      }
    }
    warp_race_merge(r);
    const uint32_t y = r.v1 < (uint32_t)A.V ? r.v1 : (uint32_t)am;
    rec.y = (int32_t)y;
    if (r.s2 >= 0.f && (r.s1 - r.s2) < kMargin * (r.t1 + r.t2)) rec.draw_flags |= SPEC_F_MARGIN_DRAW;
    const float ly = load_logit_global(A, kBF16, U.lrow + y);
    rec.lp_y = (ly - m) * U.invT - lnZ;
  }
  if (lane == 0) commit_record(A, U, rec);
}

// ---------------------------------------------------------------------------
// One unit, all CTAs of the cluster.
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ void process_unit(Cluster& K, Smem& S, const Args& A, int unit) {
  Unit U;
  U.pos = A.k - unit / A.B;
  U.row = unit % A.B;
  U.rank = K.rank;
  U.C = K.C;
  U.g0 = K.rank * A.slice_groups;
  U.ng = min(A.slice_groups, A.groups_total - U.g0);
  if (U.ng < 0) U.ng = 0;
  U.lrow = ((size_t)U.row * (A.k + 1) + U.pos) * (size_t)A.V;
  U.qrow = ((size_t)U.row * A.k + U.pos) * (size_t)A.V;

  const spec_params_t prm = A.params[U.row];
  const float T = prm.temperature;
  const float Pp = prm.top_p;
  const bool T_ok = (T == 0.0f) || (isfinite(T) && T >= 1.17549435e-38f);
  const bool P_ok = isfinite(Pp) && Pp > 0.0f && Pp <= 1.0f;
  U.bad_param = !(T_ok && P_ok);
  U.greedy = U.bad_param || T == 0.0f;
  U.K = (prm.top_k > 0 && prm.top_k < A.V) ? prm.top_k : 0;
  U.P = (U.greedy || Pp >= 1.0f) ? 1.0f : Pp;
  U.T = U.greedy ? 0.f : T;
  U.c = U.greedy ? kLog2e : kLog2e / T;
  U.invT = U.greedy ? 1.0f : 1.0f / T;
  const bool has_q = U.pos < A.k;
  const bool small_topk = !U.greedy && U.K > 0 && U.K <= kTopkSmall;

  // ---- stage: global -> shared, group maxima, max / argmax, NaN ----
  // Every thread copies its own groups (cp.async, the whole slice in flight at
  // once) and later passes read back exactly the groups the thread copied, so
  // no block barrier is needed between staging and use.
  unsigned long long best = 0;   // key64 of (value, index)
  bool nan_seen = false;
  {
    constexpr int ES = kBF16 ? 2 : 4;
    const unsigned char* gbase = reinterpret_cast<const unsigned char*>(A.logits) + U.lrow * ES;
    for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) {
      const int e0 = (U.g0 + gl) * 8;
      unsigned char* dst = S.slice + (size_t)gl * 8 * ES;
      if (A.vec_logits && e0 + 8 <= A.V) {
        cp_async16(dst, gbase + (size_t)e0 * ES);
        if (!kBF16) cp_async16(dst + 16, gbase + (size_t)e0 * ES + 16);
      } else if (kBF16) {
        const uint16_t* p16 = reinterpret_cast<const uint16_t*>(gbase);
        uint32_t h[8];
        for (int i = 0; i < 8; ++i) h[i] = (e0 + i < A.V) ? p16[e0 + i] : 0xff80u;
        *reinterpret_cast<uint4*>(dst) = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16),
                                                   h[4] | (h[5] << 16), h[6] | (h[7] << 16));
      } else {
        const float* p32 = reinterpret_cast<const float*>(gbase);
        float t[8];
        for (int i = 0; i < 8; ++i) t[i] = (e0 + i < A.V) ? p32[e0 + i] : -INFINITY;
        reinterpret_cast<float4*>(dst)[0] = make_float4(t[0], t[1], t[2], t[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(t[4], t[5], t[6], t[7]);
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
    for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) {
      const int e0 = (U.g0 + gl) * 8;
      float gm;
      if (kBF16) {
        const uint4 w = reinterpret_cast<const uint4*>(S.slice)[gl];
        const uint32_t m2 = max_nan_bf16x2(max_nan_bf16x2(w.x, w.y), max_nan_bf16x2(w.z, w.w));
        gm = max_nan(bf16_lo(m2), bf16_hi(m2));
      } else {
        const float4 a = reinterpret_cast<const float4*>(S.slice)[2 * gl];
        const float4 b = reinterpret_cast<const float4*>(S.slice)[2 * gl + 1];
        gm = max_nan(max_nan(max_nan(a.x, a.y), max_nan(a.z, a.w)),
                     max_nan(max_nan(b.x, b.y), max_nan(b.z, b.w)));
      }
      S.gmax[gl] = gm;
      if (gm != gm) {
        nan_seen = true;
      } else if (best == 0 || gm > from_okey((uint32_t)(best >> 32))) {
        float v[8];
        load_group_values<kBF16>(S, gl, v);
        int first = 0;
#pragma unroll
        for (int i = 7; i >= 0; --i)
          if (v[i] == gm) first = i;
        best = key64(okey(gm), (uint32_t)(e0 + first));
      }
    }
  }
  // A NaN anywhere makes the maximum key all ones, which decodes to NaN.
  if (nan_seen) best = ~0ull;
  best = block_max_u64(S, best);
  const unsigned long long gbest = cl_max_u64(K, S, best);
  const float m = from_okey((uint32_t)(gbest >> 32));
  const int am = (int)key64_idx(gbest);
  const bool invalid = gbest == 0 || !(m > -INFINITY) || !(m < INFINITY);

  if (invalid) {
    if (K.rank == 0 && threadIdx.x == 0) {
      UnitRecord rec;
      memset(&rec, 0, sizeof(rec));
      rec.flags = SPEC_F_NAN;
      rec.y = -1;
      commit_record(A, U, rec);
    }
    return;
  }
  const uint32_t base_flags = U.bad_param ? SPEC_F_BAD_PARAM : 0u;

  // ---------------- greedy ----------------
  if (U.greedy) {
    float z0 = 0.f, z1 = 0.f;
    for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) {
      float v[8];
      load_group_values<kBF16>(S, gl, v);
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        z0 += ex2((v[i] - m) * kLog2e);
        z1 += ex2((v[i + 1] - m) * kLog2e);
      }
    }
    const float2 zb = block_sum_f2(S, z0 + z1, 0.f);
    const float2 Z = cl_sum_f2(K, S, zb.x, 0.f);
    if (K.rank == 0 && threadIdx.x == 0) {
      const float lnZ = logf(Z.x);
      UnitRecord rec;
      memset(&rec, 0, sizeof(rec));
      rec.flags = base_flags;
      rec.y = -1;
      bool need_draw = !has_q;
      float q_am = 0.f;
      if (has_q) {
        AcceptInfo ai = accept_test(A, U, kBF16, m, 0.f, false, 1.f, true, am);
        if (!ai.valid) rec.flags |= SPEC_F_BAD_TOKEN;
        rec.accept = ai.accept ? 1 : 0;
        rec.lp_x = ai.valid ? (ai.lx - m) - lnZ : 0.f;
        q_am = A.q[U.qrow + am];
        rec.alpha = fminf(1.0f, q_am);
        need_draw = !ai.accept;
      }
      if (need_draw) {
        rec.y = am;
        rec.lp_y = -lnZ;
        if (has_q && !(1.0f - q_am > 0.0f)) rec.draw_flags |= SPEC_F_RESIDUAL_EMPTY;
      }
      commit_record(A, U, rec);
    }
    return;
  }

  // ---------------- small top-k: candidate list ----------------
  if (small_topk) {
    bool ovf = false;
    const int nloc = local_topk<kBF16>(K, S, U, A, m, U.K, &ovf);
    const int slot = K.step++ & 1;
    if (threadIdx.x == 0) S.ctl->xch[slot][0] = (unsigned long long)nloc | (ovf ? (1ull << 40) : 0ull);
    K.cl.sync();
    int counts[kMaxC];
    bool any_ovf = false;
    for (int c = 0; c < K.C; ++c) {
      const unsigned long long w = *remote(K, &S.ctl->xch[slot][0], c);
      counts[c] = (int)(w & 0xffffffffull);
      any_ovf |= (w >> 40) != 0;
    }
    if (!any_ovf) {
      if (K.rank == 0) {
        const int n_k = K.C > 1 ? merge_lists(K, S, counts, U.K) : counts[0];
        if (threadIdx.x < 32) list_unit<kBF16>(S, U, A, m, am, n_k, base_flags);
      }
      return;
    }
    // overflow: fall through to the general threshold path
  }

  // ---------------- general path: threshold-described kept set ----------------
  Thresh th;
  th.tkey = 0u;
  th.tidx = 0xffffffffu;
  if (U.K > 0) th = select_count<kBF16>(K, S, U, A, m, (unsigned long long)U.K);
  const bool filtered = U.K > 0 || U.P < 1.0f;
  const bool fused_bonus = !has_q && !filtered;

  // Z pass (+ fixed-point mass histogram for top-p) (+ bonus race when unfiltered)
  Race race;
  race_init(race);
  if (fused_bonus) {
    // probe: the argmax entry bounds the race from below
    const uint4 pw = philox4x32_10(make_uint4((uint32_t)am >> 2, (uint32_t)U.pos, (uint32_t)U.row, 1u), A.key0, A.key1);
    race_consider(race, 1.0f, 0.f, (uint32_t)am, word_of(pw, am & 3));
  }
  const bool topp = U.P < 1.0f;
  const int hslot = 0;
  if (topp) {
    S.ctl->mlo[hslot][threadIdx.x] = 0;
    S.ctl->mhi[hslot][threadIdx.x] = 0;
    __syncthreads();
  }
  unsigned long long tail = 0;   // mass of the lumped last bin, kept in registers
  float z0 = 0.f, z1 = 0.f;
  for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) {
    float v[8];
    load_group_values<kBF16>(S, gl, v);
    const int e0 = (U.g0 + gl) * 8;
    float e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float x = (v[i] - m) * U.c;
      bool in = true;
      if (U.K > 0) in = kept(th, okey(v[i]), (uint32_t)(e0 + i)) && (e0 + i < A.V);
      e[i] = in ? ex2(x) : 0.f;
      if (i & 1) z1 += e[i]; else z0 += e[i];
      if (topp && e[i] > 0.f) {
        const int bin = __float2int_rz(fminf(-x * 8.0f, 255.0f));
        const unsigned long long fx = mass_fixed(e[i]);
        if (bin < 255) mass_add(&S.ctl->mlo[hslot][bin], &S.ctl->mhi[hslot][bin], fx);
        else tail += fx;
      }
    }
    if (fused_bonus) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float* eh = e + 4 * h;
        if (eh[0] > 0.f || eh[1] > 0.f || eh[2] > 0.f || eh[3] > 0.f) {
          const uint32_t blk = (uint32_t)((e0 >> 2) + h);
          const uint4 w = philox4x32_10(make_uint4(blk, (uint32_t)U.pos, (uint32_t)U.row, 1u), A.key0, A.key1);
          if (eh[0] > 0.f) race_consider(race, eh[0], 0.f, blk * 4 + 0, w.x);
          if (eh[1] > 0.f) race_consider(race, eh[1], 0.f, blk * 4 + 1, w.y);
          if (eh[2] > 0.f) race_consider(race, eh[2], 0.f, blk * 4 + 2, w.z);
          if (eh[3] > 0.f) race_consider(race, eh[3], 0.f, blk * 4 + 3, w.w);
        }
      }
    }
  }
  float Zs;
  uint32_t flags = base_flags;
  if (topp) {
    __syncthreads();
    tail = block_sum_u64(S, tail);
    if (threadIdx.x == 0) {
      S.ctl->mlo[hslot][255] = (uint32_t)tail;
      S.ctl->mhi[hslot][255] = (uint32_t)(tail >> 32);
    }
    __syncthreads();
    cl_hist(K, S, hslot, true);
    unsigned long long zk = 0;
    {
      // total mass: sum of the reduced histogram (every thread holds one bin)
      zk = block_sum_u64(S, S.ctl->total[threadIdx.x]);
      if (threadIdx.x == 0) S.ctl->bc64[2] = zk;
      __syncthreads();
      zk = S.ctl->bc64[2];
      __syncthreads();
    }
    const double target_d = ceil((double)U.P * (double)zk);
    const unsigned long long target = (unsigned long long)target_d;
    int b;
    unsigned long long above;
    select_from_bin0(S, target, &b, &above);
    // range of keys in bin b
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) {
      float v[8];
      load_group_values<kBF16>(S, gl, v);
      const int e0 = (U.g0 + gl) * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (e0 + i >= A.V) continue;
        const uint32_t key = okey(v[i]);
        if (U.K > 0 && !kept(th, key, (uint32_t)(e0 + i))) continue;
        const float x = (v[i] - m) * U.c;
        const float e = ex2(x);
        if (!(e > 0.f)) continue;
        const int bin = __float2int_rz(fminf(-x * 8.0f, 255.0f));
        if (bin == b) {
          kmin = min(kmin, key);
          kmax = max(kmax, key);
        }
      }
    }
    // block min/max then cluster
    {
      uint32_t a = ~kmin, c = kmax;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
        c = max(c, __shfl_xor_sync(0xffffffffu, c, o));
      }
      uint32_t* wb = reinterpret_cast<uint32_t*>(S.ctl->wred);
      if ((threadIdx.x & 31) == 0) {
        wb[2 * (threadIdx.x >> 5)] = a;
        wb[2 * (threadIdx.x >> 5) + 1] = c;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        uint32_t aa = 0, cc = 0;
        for (int i = 0; i < kWarps; ++i) {
          aa = max(aa, wb[2 * i]);
          cc = max(cc, wb[2 * i + 1]);
        }
        kmin = ~aa;
        kmax = cc;
      }
      __syncthreads();
    }
    const uint2 mm = cl_minmax_u32(K, S, kmin, kmax);
    uint32_t lo = mm.x, hi = mm.y;
    unsigned long long rem = target - above;   // mass still needed inside bin b
    int hs = 1;
    while (hi > lo) {
      const uint32_t span = hi - lo;
      const int nbits = 32 - __clz(span);
      const int shift = nbits > 8 ? nbits - 8 : 0;
      const int slot = hs++ & 1;
      S.ctl->mlo[slot][threadIdx.x] = 0;
      S.ctl->mhi[slot][threadIdx.x] = 0;
      __syncthreads();
      for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) {
        float v[8];
        load_group_values<kBF16>(S, gl, v);
        const int e0 = (U.g0 + gl) * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (e0 + i >= A.V) continue;
          const uint32_t key = okey(v[i]);
          if (key < lo || key > hi) continue;
          if (U.K > 0 && !kept(th, key, (uint32_t)(e0 + i))) continue;
          const float e = ex2((v[i] - m) * U.c);
          const uint32_t bin = (hi - key) >> shift;
          mass_add(&S.ctl->mlo[slot][bin], &S.ctl->mhi[slot][bin], mass_fixed(e));
        }
      }
      __syncthreads();
      cl_hist(K, S, slot, true);
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
    const float tv = from_okey(tkey);
    const float et = ex2((tv - m) * U.c);
    const unsigned long long efx = mass_fixed(et);
    unsigned long long n_need = efx ? (rem + efx - 1) / efx : 1ull;
    if (n_need == 0) n_need = 1;
    // the n-th tie among kept elements; with a top-k threshold at the same key,
    // the ties kept by top-k are a prefix of the ties, so the rank carries over
    th.tidx = nth_tie_index<kBF16>(K, S, U, A, tkey, n_need);
    th.tkey = tkey;
    const unsigned long long zs_fx = above + n_need * efx;
    Zs = (float)((double)zs_fx * (1.0 / 1099511627776.0));
    const double at = (double)zs_fx / (double)zk;
    const double bef = (double)(zs_fx - efx) / (double)zk;
    if (fabs(at - (double)U.P) < 1e-6 || fabs((double)U.P - bef) < 1e-6) flags |= SPEC_F_MARGIN_TOPP;
  } else {
    const float2 zb = block_sum_f2(S, z0 + z1, 0.f);
    const float2 Z = cl_sum_f2(K, S, zb.x, 0.f);
    Zs = Z.x;
  }
  const bool filt = U.K > 0 || topp;
  const float invZ = 1.0f / Zs;
  const float lnZ = logf(Zs);

  // accept decision (every CTA computes the same)
  AcceptInfo ai;
  ai.accept = false;
  ai.valid = true;
  ai.margin = false;
  ai.lx = 0.f;
  bool need_race = !has_q;
  if (has_q) {
    const int x = A.drafts[(size_t)U.row * A.k + U.pos];
    bool xin = false;
    float ex = 0.f;
    if (x >= 0 && x < A.V) {
      const float lx = load_logit_global(A, kBF16, U.lrow + x);
      xin = !filt || kept(th, okey(lx), (uint32_t)x);
      ex = ex2((lx - m) * U.c);
    }
    ai = accept_test(A, U, kBF16, m, ex, xin, Zs, false, am);
    need_race = !ai.accept;
  }

  // alpha / race pass (or the race for a filtered bonus position)
  float al0 = 0.f, al1 = 0.f;
  if (has_q || (need_race && !fused_bonus)) {
    if (need_race && has_q) {
      // probe: the argmax entry (always kept)
      const float p_am = invZ;
      const float q_am = A.q[U.qrow + am];
      const float w = fmaxf(p_am - q_am, 0.f);
      if (w > 0.f) {
        const uint4 pw = philox4x32_10(make_uint4((uint32_t)am >> 2, (uint32_t)U.pos, (uint32_t)U.row, 1u), A.key0, A.key1);
        race_consider(race, w, 2.0f * q_am, (uint32_t)am, word_of(pw, am & 3));
      }
    } else if (need_race) {
      const uint4 pw = philox4x32_10(make_uint4((uint32_t)am >> 2, (uint32_t)U.pos, (uint32_t)U.row, 1u), A.key0, A.key1);
      race_consider(race, 1.0f, 0.f, (uint32_t)am, word_of(pw, am & 3));
    }
    const float* qbase = A.q + U.qrow;
    // q streams through a per-thread ring of kQD slots: group i of this thread
    // is copied kQD-1 iterations before it is consumed (empty commits keep the
    // group count uniform), so each thread keeps 64+ bytes of q in flight.
    const bool qpipe = has_q && A.vec_q;
    float* ring = S.qring + (size_t)threadIdx.x * 8;
    auto q_issue = [&](int i) {
      const int gl = threadIdx.x + i * kThreads;
      if (gl < U.ng) {
        const int e0 = (U.g0 + gl) * 8;
        if (e0 + 8 <= A.V) {
          float* d = ring + (size_t)(i % kQD) * kThreads * 8;
          cp_async16(d, qbase + e0);
          cp_async16(d + 4, qbase + e0 + 4);
        }
      }
      cp_async_commit();
    };
    if (qpipe)
      for (int i = 0; i < kQD - 1; ++i) q_issue(i);
    int it = 0;
    for (int gl = threadIdx.x; gl < U.ng; gl += kThreads, ++it) {
      float v[8];
      load_group_values<kBF16>(S, gl, v);
      const int e0 = (U.g0 + gl) * 8;
      float qv[8];
      if (has_q) {
        if (qpipe && e0 + 8 <= A.V) {
          q_issue(it + kQD - 1);
          cp_async_wait<kQD - 1>();
          const float* d = ring + (size_t)(it % kQD) * kThreads * 8;
          const float4 qa = *reinterpret_cast<const float4*>(d);
          const float4 qb = *reinterpret_cast<const float4*>(d + 4);
          qv[0] = qa.x; qv[1] = qa.y; qv[2] = qa.z; qv[3] = qa.w;
          qv[4] = qb.x; qv[5] = qb.y; qv[6] = qb.z; qv[7] = qb.w;
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) qv[i] = (e0 + i < A.V) ? qbase[e0 + i] : 0.f;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) qv[i] = 0.f;
      }
      float w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        bool in = e0 + i < A.V;
        if (filt) in = in && kept(th, okey(v[i]), (uint32_t)(e0 + i));
        const float e = in ? ex2((v[i] - m) * U.c) : 0.f;
        const float p = has_q ? e * invZ : e;
        if (has_q) {
          if (i & 1) al1 += fminf(p, qv[i]); else al0 += fminf(p, qv[i]);
        }
        w[i] = has_q ? fmaxf(p - qv[i], 0.f) : p;
      }
      if (need_race) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float* wh = w + 4 * h;
          if (wh[0] > 0.f || wh[1] > 0.f || wh[2] > 0.f || wh[3] > 0.f) {
            const uint32_t blk = (uint32_t)((e0 >> 2) + h);
            const uint4 ww = philox4x32_10(make_uint4(blk, (uint32_t)U.pos, (uint32_t)U.row, 1u), A.key0, A.key1);
            if (wh[0] > 0.f) race_consider(race, wh[0], 2.0f * qv[4 * h + 0], blk * 4 + 0, ww.x);
            if (wh[1] > 0.f) race_consider(race, wh[1], 2.0f * qv[4 * h + 1], blk * 4 + 1, ww.y);
            if (wh[2] > 0.f) race_consider(race, wh[2], 2.0f * qv[4 * h + 2], blk * 4 + 2, ww.z);
            if (wh[3] > 0.f) race_consider(race, wh[3], 2.0f * qv[4 * h + 3], blk * 4 + 3, ww.w);
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  float alpha_v = 0.f;
  if (has_q) {
    const float2 ab = block_sum_f2(S, al0 + al1, 0.f);
    alpha_v = cl_sum_f2(K, S, ab.x, 0.f).x;
  }
  uint32_t draw_flags = 0;
  Race gr;
  race_init(gr);
  if (need_race) {
    block_race(S, race);
    if (threadIdx.x != 0) race_init(race);
    gr = cl_race(K, S, race);
    if (gr.s1 < 0.f) {
      // empty residual: draw from p instead
      draw_flags |= SPEC_F_RESIDUAL_EMPTY;
      race_init(race);
      for (int gl = threadIdx.x; gl < U.ng; gl += kThreads) {
        float v[8];
        load_group_values<kBF16>(S, gl, v);
        const int e0 = (U.g0 + gl) * 8;
        for (int i = 0; i < 8; ++i) {
          bool in = e0 + i < A.V;
          if (filt) in = in && kept(th, okey(v[i]), (uint32_t)(e0 + i));
          const float e = in ? ex2((v[i] - m) * U.c) : 0.f;
          if (e > 0.f) {
            const uint32_t vv = (uint32_t)(e0 + i);
            const uint4 ww = philox4x32_10(make_uint4(vv >> 2, (uint32_t)U.pos, (uint32_t)U.row, 1u), A.key0, A.key1);
            race_consider(race, e, 0.f, vv, word_of(ww, vv & 3));
          }
        }
      }
      block_race(S, race);
      if (threadIdx.x != 0) race_init(race);
      gr = cl_race(K, S, race);
    }
    if (gr.s2 >= 0.f && (gr.s1 - gr.s2) < kMargin * (gr.t1 + gr.t2)) draw_flags |= SPEC_F_MARGIN_DRAW;
  }

  if (K.rank == 0 && threadIdx.x == 0) {
    UnitRecord rec;
    memset(&rec, 0, sizeof(rec));
    rec.flags = flags;
    rec.y = -1;
    if (has_q) {
      if (!ai.valid) rec.flags |= SPEC_F_BAD_TOKEN;
      if (ai.margin) rec.flags |= SPEC_F_MARGIN_ACCEPT;
      rec.accept = ai.accept ? 1 : 0;
      rec.lp_x = ai.valid ? (ai.lx - m) * U.invT - lnZ : 0.f;
      rec.alpha = alpha_v;
    }
    if (need_race) {
      const uint32_t y = gr.v1 < (uint32_t)A.V ? gr.v1 : (uint32_t)am;   // am always competes
      rec.y = (int32_t)y;
      const float ly = load_logit_global(A, kBF16, U.lrow + y);
      rec.lp_y = (ly - m) * U.invT - lnZ;
      rec.draw_flags = draw_flags;
    }
    commit_record(A, U, rec);
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const Args A) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem S = carve<kBF16>(smem_raw, A.slice_groups);
  Cluster K{cg::this_cluster(), A.C, 0, 0};
  K.rank = (int)K.cl.block_rank();
  const bool leader = K.rank == 0;
  while (true) {
    if (leader && threadIdx.x == 0) {
      S.ctl->unit = (int)atomicAdd(&A.ws->queue_next, 1u);
      S.ctl->cand_count = 0;
    }
    K.cl.sync();
    if (threadIdx.x == 0) S.ctl->bci[7] = *remote(K, &S.ctl->unit, 0);
    __syncthreads();
    const int unit = S.ctl->bci[7];
    if (unit >= A.n_units) break;
    process_unit<kBF16>(K, S, A, unit);
  }
  K.cl.sync();   // keep shared memory alive until every CTA is done with DSMEM
  if (leader && threadIdx.x == 0) {
    __threadfence();
    const uint32_t d = atomicAdd(&A.ws->clusters_done, 1u);
    if (d == (uint32_t)A.n_clusters - 1u) {
      A.ws->queue_next = 0u;
      A.ws->clusters_done = 0u;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
struct LaunchCfg {
  int C;
  int slice_groups;
  size_t smem;
  int max_clusters;
};

static size_t ws_bytes(int B, int k) {
  size_t s = sizeof(WsHeader);
  s += align_up((size_t)B * 4, 256);
  s += (size_t)B * (k + 1) * sizeof(UnitRecord);
  return s;
}

template <bool kBF16>
static int plan(int V, int device, LaunchCfg* cfg) {
  const int groups = (V + 7) / 8;
  const size_t es = kBF16 ? 2 : 4;
  const size_t budget = 40 * 1024;
  int C = 1;
  while (C < kMaxC && (size_t)((groups + C - 1) / C) * 8 * es > budget) C <<= 1;
  const int sg = (groups + C - 1) / C;
  cfg->C = C;
  cfg->slice_groups = sg;
  cfg->smem = smem_bytes<kBF16>(sg);

  static std::mutex mu;
  static int cache_key[64][4];
  static int cache_val[64];
  static int cache_n = 0;
  // The dynamic shared memory limit is a property of the kernel (per device),
  // not of one launch: keep it at the largest size any launch has needed.
  static int smem_set[64][2];
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return SPEC_E_CUDA;
  auto kern = verify_kernel<kBF16>;
  if (smem_set[device][kBF16] < (int)cfg->smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg->smem) != cudaSuccess) {
      cudaGetLastError();
      return SPEC_E_CUDA;
    }
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
      cudaGetLastError();
      return SPEC_E_CUDA;
    }
    smem_set[device][kBF16] = (int)cfg->smem;
  }
  for (int i = 0; i < cache_n; ++i)
    if (cache_key[i][0] == device && cache_key[i][1] == C && cache_key[i][2] == (int)cfg->smem &&
        cache_key[i][3] == (int)kBF16) {
      cfg->max_clusters = cache_val[i];
      return SPEC_OK;
    }
  cudaLaunchConfig_t lc;
  memset(&lc, 0, sizeof(lc));
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(C, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = cfg->smem;
  lc.attrs = at;
  lc.numAttrs = 1;
  int nc = 0;
  if (cudaOccupancyMaxActiveClusters(&nc, kern, &lc) != cudaSuccess || nc <= 0) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  cfg->max_clusters = nc;
  if (cache_n < 64) {
    cache_key[cache_n][0] = device;
    cache_key[cache_n][1] = C;
    cache_key[cache_n][2] = (int)cfg->smem;
    cache_key[cache_n][3] = (int)kBF16;
    cache_val[cache_n] = nc;
    ++cache_n;
  }
  return SPEC_OK;
}

template <bool kBF16>
static int launch(const Args& base, int V, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_E_CUDA;
  LaunchCfg cfg;
  const int rc = plan<kBF16>(V, dev, &cfg);
  if (rc != SPEC_OK) return rc;
  Args A = base;
  A.C = cfg.C;
  A.groups_total = (V + 7) / 8;
  A.slice_groups = cfg.slice_groups;
  A.n_clusters = min(A.n_units, cfg.max_clusters);
  cudaLaunchConfig_t lc;
  memset(&lc, 0, sizeof(lc));
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cfg.C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(A.n_clusters * cfg.C, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = stream;
  lc.attrs = at;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, verify_kernel<kBF16>, A) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  return SPEC_OK;
}

}  // namespace specv

extern "C" size_t spec_verify_workspace_size(int B, int k, int V) {
  (void)V;
  if (B < 0 || k < 0) return 0;
  return specv::ws_bytes(B, k);
}

static inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

extern "C" int spec_verify(const void* logits, int logits_dtype, const float* draft_probs,
                           const int32_t* draft_tokens, const spec_params_t* params, uint64_t seed,
                           int B, int k, int V, int32_t* tokens, int32_t* accept_len,
                           float* logprobs, float* alpha, uint32_t* flags, void* workspace,
                           size_t workspace_bytes, void* cuda_stream) {
  if (B < 0 || k < 0 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return SPEC_E_DIM;
  if ((long long)B * (k + 1) > (1ll << 26)) return SPEC_E_DIM;
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
  if (workspace_bytes < specv::ws_bytes(B, k)) return SPEC_E_WORKSPACE;
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
  A.tickets = reinterpret_cast<uint32_t*>(ws + sizeof(specv::WsHeader));
  A.recs = reinterpret_cast<specv::UnitRecord*>(ws + sizeof(specv::WsHeader) +
                                                specv::align_up((size_t)B * 4, 256));
  A.key0 = (uint32_t)(seed & 0xffffffffull);
  A.key1 = (uint32_t)(seed >> 32);
  A.B = B;
  A.k = k;
  A.V = V;
  A.n_units = B * (k + 1);
  A.vec_logits = aligned(logits, 16) && ((size_t)V * es) % 16 == 0;
  A.vec_q = k > 0 && aligned(draft_probs, 16) && (V % 4) == 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
  return logits_dtype == SPEC_BF16 ? specv::launch<true>(A, V, st) : specv::launch<false>(A, V, st);
}
