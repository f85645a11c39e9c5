// spec_verify: the verify kernel (sm_103a).
//
// One persistent CTA of 16 warps per SM, launched cooperatively (all CTAs
// resident, so warps may wait on one another).  Nothing in it waits on a
// barrier across CTAs and nothing stores with a fence: results pass between
// warps as 64-bit words tagged with the call's epoch, which a reader polls.
//   * Stream warps.  Each owns two 6 KB shared-memory buffers and has the
//     copy engine stream its next item into one (cp.async.bulk completed on
//     an mbarrier) while it reduces the other with warp collectives.  The
//     items of all units form one sequence, which the stream warps of all
//     SMs take in order from one counter:
//       A items of drafted unfiltered units, of small top-k units, of
//       unfiltered bonus positions, of greedy units; B items of drafted
//       unfiltered units.
//     An A item is a chunk of one unit's logits (3072 bf16 / 1536 fp32):
//     max, the softmax sum relative to the chunk max, for greedy units the
//     first argmax, at a bonus position the level-1 race of the chunk's
//     256-entry blocks, for a small top-k the chunk's 8 largest entries in
//     the total order (the smallest last).  A B item (1024 bf16 / 768 fp32 logits, read again from
//     L2, plus q) takes the unit state from its tagged words and computes
//     alpha = sum min(p, q) and the level-1 race of the residual.
//   * Settle warps (the first scheduler's warps, four per SM, on as many SMs
//     as the tasks need).  Each takes its units in
//     the same class order, waits for their records and settles them
//     (spec_settle.cuh); a drafted unfiltered unit publishes its state for
//     the B items and is finished after them.
//   * Rows that need a global threshold search (spec_general.cuh) are taken
//     last by half-CTA groups.
// The last settled unit of a row resolves the accept chain and writes the
// row's outputs.  Every wait is bounded and ends with an error bit;
// reductions have a fixed order and no floating-point atomics are used, so
// results are bit-reproducible.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "spec_general.cuh"
#include "spec_host.h"
#include "spec_settle.cuh"
#include "spec_verify_common.cuh"

namespace specv {

constexpr int kSW = 16;                // warps per CTA
constexpr int kAllThreads = kSW * 32;
constexpr int kOrderSmem = 512;        // batches up to this many rows keep order and configs in shared memory
constexpr int kStage = 64;             // per-warp staging of a top-k item's candidates
constexpr unsigned kFull = 0xffffffffu;
static_assert(kAllThreads == 2 * kThreads, "two general-path groups per CTA");

struct OrderScratch {
  int n_class[4];
  int run[4];
  int scan[kSW][4];
};

struct alignas(128) VShm {
  union {
    unsigned char buf[kSW][2][kSlot];  // stream buffers; a settle warp's pair is its top-k scratch
    GenShm gen[2];                     // general-path groups, at the end
  };
  unsigned long long bar[kSW][2];
  u64 stage[kSW][kStage];
  uint32_t order[kOrderSmem];
  RowPack cfg[kOrderSmem];
  OrderScratch ord;
  int gtask[2];
  uint32_t tag;
};
static_assert(sizeof(GenShm) * 2 <= sizeof(unsigned char) * kSW * 2 * kSlot, "general scratch");

// ---------------------------------------------------------------------------
// Row order: rows of each class, stably, as [unfiltered][small top-k][greedy]
// [general].
// ---------------------------------------------------------------------------
__device__ __forceinline__ int class_base(const OrderScratch& O, int cl) {
  const int nD = O.n_class[UT_DENSE], nT = O.n_class[UT_TOPK], nG = O.n_class[UT_GREEDY];
  return cl == UT_DENSE ? 0 : (cl == UT_TOPK ? nD : (cl == UT_GREEDY ? nD + nT : nD + nT + nG));
}

// Stable placement of one round of kAllThreads rows (cl < 0: no row).
__device__ __forceinline__ void place_round(uint32_t* order, OrderScratch& O, int r, int cl) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  unsigned mine = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const unsigned b = __ballot_sync(kFull, cl == t);
    if (lane == 0) O.scan[w][t] = __popc(b);
    if (cl == t) mine = b;
  }
  __syncthreads();
  if (cl >= 0) {
    int off = class_base(O, cl) + O.run[cl];
    for (int ww = 0; ww < w; ++ww) off += O.scan[ww][cl];
    off += __popc(mine & ((1u << lane) - 1u));
    order[off] = (uint32_t)r;
  }
  __syncthreads();
  if (tid < 4) {
    int s = 0;
    for (int ww = 0; ww < kSW; ++ww) s += O.scan[ww][tid];
    O.run[tid] += s;
  }
  __syncthreads();
}

static_assert(kOrderSmem == kAllThreads, "one placement round for a shared-memory order");

// Batches of up to kOrderSmem rows: every CTA classifies the rows into
// shared memory (one parameter load per row).
__device__ __noinline__ void build_order_smem(const Args& A, uint32_t* order, RowPack* cfgs, OrderScratch& O) {
  const int tid = threadIdx.x;
  if (tid < 4) {
    O.n_class[tid] = 0;
    O.run[tid] = 0;
  }
  __syncthreads();
  int cl = -1;
  if (tid < A.B) {
    const RowCfg c = classify(A.params[tid], A.V);
    cfgs[tid] = pack_cfg(c);
    cl = c.type;
    atomicAdd(&O.n_class[cl], 1);
  }
  __syncthreads();
  place_round(order, O, tid, cl);
}

// Larger batches: CTA 0 writes the order and the class counts into the
// workspace and publishes them with the call's tag; the other CTAs wait for it.
__device__ __noinline__ void build_order_global(const Args& A, OrderScratch& O, uint32_t tag) {
  const int tid = threadIdx.x;
  if (tid < 4) {
    O.n_class[tid] = 0;
    O.run[tid] = 0;
  }
  __syncthreads();
  for (int r = tid; r < A.B; r += kAllThreads) atomicAdd(&O.n_class[classify(A.params[r], A.V).type], 1);
  __syncthreads();
  for (int base = 0; base < A.B; base += kAllThreads) {
    const int r = base + tid;
    place_round(A.order, O, r, r < A.B ? classify(A.params[r], A.V).type : -1);
  }
  if (tid < 4) A.ws->n_class[tid] = (uint32_t)O.n_class[tid];
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    store_release(&A.ws->order_tag, tag);
  }
}

// ---------------------------------------------------------------------------
// Work items.
// ---------------------------------------------------------------------------
struct Plan {
  const uint32_t* order;
  const RowPack* cfg;       // per-row configs in shared memory (null: classify from the parameters)
  int nD, nT, nG, nX;       // rows: unfiltered, small top-k, greedy, general
  int NCA, NCB;
  uint32_t sDD, sTK, sDB, sB, sGR;   // segments of the item sequence
};

// A work item.  kind: 0 none, 1 A item, 2 B item.
struct Item {
  int kind;
  int reread;               // the logits are read again later (default L2 policy)
  int row, pos, u, c, n;    // unit, chunk, valid entries in the item
};

__device__ __forceinline__ RowCfg plan_cfg(const Args& A, const Plan& P, int row) {
  return P.cfg ? unpack_cfg(P.cfg[row]) : classify(A.params[row], A.V);
}


// Item t of the sequence [A: drafted unfiltered][A: small top-k][A: bonus
// positions][A: greedy][B: drafted unfiltered]: the states that the B items
// need are published early, the top-k units, whose settle takes longest,
// follow, and the greedy items run before the B items.
template <bool kBF16>
__device__ __forceinline__ Item map_item(const Args& A, const Plan& P, uint32_t t) {
  using G = Geo<kBF16>;
  Item it;
  it.kind = 0;
  const int k = A.k, k1 = A.k + 1;
  int row, pos, j;
  uint32_t s = t;
  it.reread = 0;
  if (s < P.sDD) {
    j = (int)(s / (uint32_t)P.NCA);
    it.c = (int)s - j * P.NCA;
    row = (int)P.order[j / k];
    pos = j % k;
    it.reread = 1;
    it.kind = 1;
  } else if ((s -= P.sDD) < P.sTK) {
    j = (int)(s / (uint32_t)P.NCA);
    it.c = (int)s - j * P.NCA;
    row = (int)P.order[P.nD + j / k1];
    pos = j % k1;
    it.kind = 1;
  } else if ((s -= P.sTK) < P.sDB) {
    j = (int)(s / (uint32_t)P.NCA);
    it.c = (int)s - j * P.NCA;
    row = (int)P.order[j];
    pos = k;
    it.kind = 1;
  } else if ((s -= P.sDB) < P.sGR) {
    j = (int)(s / (uint32_t)P.NCA);
    it.c = (int)s - j * P.NCA;
    row = (int)P.order[P.nD + P.nT + j / k1];
    pos = j % k1;
    it.kind = 1;
  } else if ((s -= P.sGR) < P.sB) {
    j = (int)(s / (uint32_t)P.NCB);
    it.c = (int)s - j * P.NCB;
    row = (int)P.order[j / k];
    pos = j % k;
    it.kind = 2;
  } else {
    return it;
  }
  it.row = row;
  it.pos = pos;
  it.u = row * k1 + pos;
  it.n = it.kind == 1 ? min(G::EA, A.V - it.c * G::EA) : min(G::EB, A.V - it.c * G::EB);
  return it;
}

// Lane 0: post the copies of an item into buffer `buf`, completing on `bar`.
template <bool kBF16>
__device__ __forceinline__ void issue(const Args& A, const Item& it, unsigned char* buf, unsigned long long* bar) {
  using G = Geo<kBF16>;
  if (it.kind == 0) return;
  const unsigned char* lg = reinterpret_cast<const unsigned char*>(A.logits);
  fence_proxy_async();
  // inputs read once are marked evict-first in L2, so they do not push out the
  // records, the kernels' code and the logits the B pass reads again
  const uint64_t once = l2_policy_evict_first();
  if (it.kind == 1) {
    const uint32_t bl = A.vec_logits ? ((uint32_t)(it.n * G::es) & ~15u) : 0u;
    mbar_arrive_expect_tx(bar, bl);
    if (bl) {
      const unsigned char* src = lg + ((size_t)it.u * A.V + (size_t)it.c * G::EA) * G::es;
      if (it.reread) bulk_g2s(buf, src, bl, bar);
      else bulk_g2s_hint(buf, src, bl, bar, once);
    }
  } else {
    const uint32_t bl = A.vec_logits ? ((uint32_t)(it.n * G::es) & ~15u) : 0u;
    const uint32_t bq = A.vec_q ? ((uint32_t)(it.n * 4) & ~15u) : 0u;
    mbar_arrive_expect_tx(bar, bl + bq);
    if (bl) bulk_g2s_hint(buf, lg + ((size_t)it.u * A.V + (size_t)it.c * G::EB) * G::es, bl, bar, once);
    if (bq)
      bulk_g2s_hint(buf + G::EB * G::es,
                    A.q + ((size_t)it.row * A.k + it.pos) * (size_t)A.V + (size_t)it.c * G::EB, bq, bar, once);
  }
}

// Wait for a buffer's copies (bounded).  False if the wait gave up.
__device__ __forceinline__ bool wait_buffer(const Args& A, unsigned long long* bar, uint32_t parity) {
  long long spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if (++spins == kSpinLimit) {
      if ((threadIdx.x & 31) == 0) atomicOr(&A.ws->error, 2u);
    }
    if (spins > 2 * kSpinLimit) return false;
  }
  return true;
}

// The part of an item the bulk copy did not cover: the ragged tail (read
// with plain loads), and padding up to the end of the last block (-inf
// logits, zero q).  With rows that are not 16-byte aligned, everything.
template <bool kBF16>
__device__ __noinline__ void fill_tail(const Args& A, const Item& it, unsigned char* buf) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int E = it.kind == 1 ? G::EA : G::EB;
  const int end = ceil_div(it.n, kRaceBlock) * kRaceBlock;
  const int done = A.vec_logits ? (int)(((uint32_t)(it.n * G::es) & ~15u) / G::es) : 0;
  const size_t lrow = (size_t)it.u * A.V + (size_t)it.c * E;
  for (int e = done + lane; e < end; e += 32) {
    if (kBF16) {
      const uint16_t h = e < it.n ? reinterpret_cast<const uint16_t*>(A.logits)[lrow + e] : (uint16_t)0xff80u;
      reinterpret_cast<uint16_t*>(buf)[e] = h;
    } else {
      reinterpret_cast<float*>(buf)[e] = e < it.n ? reinterpret_cast<const float*>(A.logits)[lrow + e] : -INFINITY;
    }
  }
  if (it.kind == 2) {
    float* qb = reinterpret_cast<float*>(buf + G::EB * G::es);
    const int dq = A.vec_q ? (int)(((uint32_t)(it.n * 4) & ~15u) / 4) : 0;
    const size_t qrow = ((size_t)it.row * A.k + it.pos) * (size_t)A.V + (size_t)it.c * G::EB;
    for (int e = dq + lane; e < end; e += 32) qb[e] = e < it.n ? A.q[qrow + e] : 0.f;
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Lane layout inside a block of 256 entries: lane l holds entries 4l..4l+3
// and 128+4l..128+4l+3 (slots 0..7), so every shared load of a warp reads one
// contiguous span and no bank is hit twice.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int slot_entry(int b, int l, int j) {
  return b * kRaceBlock + (j < 4 ? 4 * l + j : 128 + 4 * l + (j - 4));
}

template <bool kBF16>
__device__ __forceinline__ void sload(const unsigned char* buf, int b, int l, float v[8]) {
  if (kBF16) {
    const uint2 a = *reinterpret_cast<const uint2*>(buf + (b * kRaceBlock + 4 * l) * 2);
    const uint2 c = *reinterpret_cast<const uint2*>(buf + (b * kRaceBlock + 128 + 4 * l) * 2);
    v[0] = bf16_lo(a.x); v[1] = bf16_hi(a.x); v[2] = bf16_lo(a.y); v[3] = bf16_hi(a.y);
    v[4] = bf16_lo(c.x); v[5] = bf16_hi(c.x); v[6] = bf16_lo(c.y); v[7] = bf16_hi(c.y);
  } else {
    const float4 a = *reinterpret_cast<const float4*>(buf + (b * kRaceBlock + 4 * l) * 4);
    const float4 c = *reinterpret_cast<const float4*>(buf + (b * kRaceBlock + 128 + 4 * l) * 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
  }
}

__device__ __forceinline__ void sload_q(const float* qb, int b, int l, float q[8]) {
  const float4 a = *reinterpret_cast<const float4*>(qb + b * kRaceBlock + 4 * l);
  const float4 c = *reinterpret_cast<const float4*>(qb + b * kRaceBlock + 128 + 4 * l);
  q[0] = a.x; q[1] = a.y; q[2] = a.z; q[3] = a.w;
  q[4] = c.x; q[5] = c.y; q[6] = c.z; q[7] = c.w;
}


// Packed f32x2 arithmetic (two lanes of work per instruction).
__device__ __forceinline__ u64 pack2(float a, float b) {
  u64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(u64 r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ u64 sub2(u64 a, u64 b) {
  u64 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
  u64 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ u64 add2(u64 a, u64 b) {
  u64 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// exp2((a - m) c) of a pair, rounded like the scalar (a - m) * c.
__device__ __forceinline__ u64 exp_pair(float a0, float a1, u64 m2, u64 c2) {
  float x0, x1;
  unpack2(mul2(sub2(pack2(a0, a1), m2), c2), x0, x1);
  return pack2(ex2(x0), ex2(x1));
}

// ---------------------------------------------------------------------------
// A items.  Lane layout: bf16 lane l reads entries 8l..8l+7 of every block of
// 256 (one 16-byte shared load); fp32 lane l reads 4l..4l+3 and
// 128+4l..128+4l+3 (two).
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ __forceinline__ int a_entry(int b, int lane, int j) {
  return kBF16 ? b * kRaceBlock + 8 * lane + j : slot_entry(b, lane, j);
}
template <bool kBF16>
__device__ __forceinline__ void a_vals(const unsigned char* buf, int b, int lane, float v[8]) {
  if (kBF16) {
    const uint4 w = *reinterpret_cast<const uint4*>(buf + (b * kRaceBlock + 8 * lane) * 2);
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
  } else {
    sload<false>(buf, b, lane, v);
  }
}

// Max (NaN-propagating) of the lane's 8 entries of block b.
template <bool kBF16>
__device__ __forceinline__ float a_block_max(const unsigned char* buf, int b, int lane) {
  if (kBF16) {
    const uint4 w = *reinterpret_cast<const uint4*>(buf + (b * kRaceBlock + 8 * lane) * 2);
    const uint32_t t = max_nan_bf16x2(max_nan_bf16x2(w.x, w.y), max_nan_bf16x2(w.z, w.w));
    return max_nan(bf16_lo(t), bf16_hi(t));
  } else {
    float v[8];
    sload<false>(buf, b, lane, v);
    return max_nan(max_nan(max_nan(v[0], v[1]), max_nan(v[2], v[3])), max_nan(max_nan(v[4], v[5]), max_nan(v[6], v[7])));
  }
}

// Greedy and unfiltered A item: the tagged record words (lanes 0..7).  The
// max first (the lane's max and the first block reaching it, for the
// argmax), then the softmax sum relative to it -- at a bonus position per
// block of 256, for the level-1 race.
template <bool kBF16>
__device__ __noinline__ void a_stats(const Args& A, uint32_t tag, const Item& it, const RowCfg& cfg,
                                     const unsigned char* buf) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int nb = ceil_div(it.n, kRaceBlock);
  const int e0 = it.c * G::EA;
  const float c = cfg.c;
  const bool greedy = cfg.type == UT_GREEDY;
  const bool bonus = !greedy && it.pos == A.k;
  // max pass: the lane's max and the first of its blocks reaching it
  float lm = -INFINITY;
  int lb = 0;
#pragma unroll 2
  for (int b = 0; b < nb; ++b) {
    const float bm = a_block_max<kBF16>(buf, b, lane);
    lb = bm > lm ? b : lb;
    lm = max_nan(lm, bm);
  }
  const bool nanl = lm != lm;
  const float mc = warp_max_f(lm);
  float z = 0.f;
  Race r;
  race_init(r);
  if (mc > -INFINITY && mc < INFINITY) {
    if (!bonus) {
      // the softmax sum relative to the chunk max
      float z0 = 0.f, z1 = 0.f;
#pragma unroll 2
      for (int b = 0; b < nb; ++b) {
        float v[8];
        a_vals<kBF16>(buf, b, lane, v);
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          z0 += ex2((v[j] - mc) * c);
          z1 += ex2((v[j + 1] - mc) * c);
        }
      }
      z = warp_sum(z0 + z1);
    } else {
      // block weights (one warp sum per block), then the level-1 race
      float myW = 0.f;
#pragma unroll 1
      for (int b = 0; b < nb; ++b) {
        float v[8];
        a_vals<kBF16>(buf, b, lane, v);
        float s8 = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) s8 += ex2((v[j] - mc) * c);
        const float W = warp_sum(s8);
        z += W;
        if (lane == b) myW = W;
      }
      if (myW > 0.f) {
        const uint32_t blk = (uint32_t)(e0 / kRaceBlock + lane);
        race_consider(r, myW, 0.f, blk, block_word(A, it.row, it.pos, blk));
      }
      warp_race_merge(r);
    }
  }
  const bool nan = __any_sync(kFull, nanl);
  uint32_t idx = 0xffffffffu;
  if (greedy && !nan) {
    // first index of the chunk max: in the lane's first block reaching it
    if (lm == mc) {
      float v[8];
      a_vals<kBF16>(buf, lb, lane, v);
#pragma unroll
      for (int j = 7; j >= 0; --j)
        if (v[j] == lm) idx = (uint32_t)(e0 + a_entry<kBF16>(lb, lane, j));
    }
    idx = warp_min_u32(idx);
  }
  u64* rec = A.rec + ((size_t)it.u * A.NCA + it.c) * kRecWords;
  const uint32_t v = lane_word8(lane, nan ? 0x7fc00000u : __float_as_uint(mc), idx, __float_as_uint(z),
                                __float_as_uint(r.s1), __float_as_uint(r.t1), __float_as_uint(r.s2),
                                __float_as_uint(r.t2), r.v1);
  if (lane < (bonus ? 8 : 3)) __stcg(rec + lane, tagw(tag, v));
  __syncwarp();
}

// Stages every finite entry >= t8 of the item (up to kStage; returns the
// count of all), block by block.
template <bool kBF16>
__device__ __noinline__ uint32_t stage_all(const unsigned char* buf, int nb, int lane, float t8, u64* stage) {
  uint32_t n = 0;
#pragma unroll 1
  for (int b = 0; b < nb; ++b) {
    float v[8];
    a_vals<kBF16>(buf, b, lane, v);
    uint32_t keep = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) keep |= (v[j] >= t8 && v[j] > -INFINITY) ? (1u << j) : 0u;
    uint32_t tot = 0;
    uint32_t p = n + warp_excl_scan((uint32_t)__popc(keep), &tot);
    n += tot;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if ((keep >> j) & 1u) {
        if (p < (uint32_t)kStage) stage[p] = key64(okey(v[j]), (uint32_t)a_entry<kBF16>(b, lane, j));
        ++p;
      }
  }
  return n;
}

// Bitonic network over lanes 0..S-1, fully unrolled: groups of S/2 sorted
// (alternating directions), then of the last merge the half-cleaners down to
// stride kList, which leave the kList largest keys in lanes 0..kList-1.
template <int S>
__device__ __forceinline__ u64 top8_network(u64 a, int lane) {
#pragma unroll
  for (int size = 2; size <= S; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (size == S && stride < kList) break;
      const u64 o = __shfl_xor_sync(kFull, a, stride);
      const bool keep_max = ((lane & size) == 0) == ((lane & stride) == 0);
      a = keep_max ? (o > a ? o : a) : (o < a ? o : a);
    }
  }
  return a;
}

// Small top-k A item: the chunk's kList largest entries in the total order,
// the smallest of them last when there are kList (key, chunk-local index),
// tagged words in lanes 0..15.  Every such entry is
// at least the 8th largest lane maximum t8; a lane keeps up to kLaneCand of
// its entries >= t8 (blocks whose maximum is below t8 are skipped), and a
// lane holding more marks the list partial.
constexpr int kLaneCand = 4;
template <bool kBF16>
__device__ __noinline__ void a_list(const Args& A, uint32_t tag, const Item& it, const unsigned char* buf,
                                    u64* stage) {
  constexpr int NB = Geo<kBF16>::NBA;
  const int lane = threadIdx.x & 31;
  const int nb = ceil_div(it.n, kRaceBlock);
  float bm[NB];
  float lm = -INFINITY;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    bm[b] = b < nb ? a_block_max<kBF16>(buf, b, lane) : -INFINITY;
    lm = max_nan(lm, bm[b]);
  }
  const bool nan = __any_sync(kFull, lm != lm);
  uint32_t flags = nan ? kListNaN : 0u;
  uint32_t nn = 0;
  if (!nan) {
    // t8: take the largest lane maxima (with their multiplicity) until 8
    uint32_t key = okey(lm), need = (uint32_t)kList, t8k = 0u;
    bool found = false;   // warp-uniform
#pragma unroll
    for (int i = 0; i < kList; ++i) {
      if (!found) {
        const uint32_t mx = __reduce_max_sync(kFull, key);
        const uint32_t c = (uint32_t)__popc(__ballot_sync(kFull, key == mx));
        t8k = mx;
        found = c >= need;
        need -= found ? 0u : c;
        key = key == mx ? 0u : key;
      }
    }
    const float t8 = from_okey(t8k);
    // the lane's blocks holding finite entries >= t8, then those entries
    uint32_t hit = 0;
#pragma unroll
    for (int b = 0; b < NB; ++b) hit |= (bm[b] >= t8 && bm[b] > -INFINITY) ? (1u << b) : 0u;
    uint32_t cnt = 0;
    u64 k0 = 0ull, k1 = 0ull, k2 = 0ull, k3 = 0ull;
#pragma unroll 1
    while (hit) {
      const int b = __ffs(hit) - 1;
      hit &= hit - 1u;
      float v[8];
      a_vals<kBF16>(buf, b, lane, v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (v[j] >= t8 && v[j] > -INFINITY) {
          k3 = k2;
          k2 = k1;
          k1 = k0;
          k0 = key64(okey(v[j]), (uint32_t)a_entry<kBF16>(b, lane, j));
          ++cnt;
        }
    }
    uint32_t n = 0;
    if (!__any_sync(kFull, cnt > (uint32_t)kLaneCand)) {
      const uint32_t p = warp_excl_scan(cnt, &n);
      if (cnt > 0 && p < (uint32_t)kStage) stage[p] = k0;
      if (cnt > 1 && p + 1 < (uint32_t)kStage) stage[p + 1] = k1;
      if (cnt > 2 && p + 2 < (uint32_t)kStage) stage[p + 2] = k2;
      if (cnt > 3 && p + 3 < (uint32_t)kStage) stage[p + 3] = k3;
    } else {
      n = stage_all<kBF16>(buf, nb, lane, t8, stage);   // a lane holds more: every entry >= t8
    }
    __syncwarp();
    if (n > (uint32_t)kStage) flags |= kListPartial;
    nn = min(n, (uint32_t)kStage);
    if (nn > (uint32_t)kList && nn <= 32) {
      // one candidate per lane: a bitonic network in registers over lanes
      // 0..S-1 (S the power of two >= nn; lanes from nn on hold 0) that sorts
      // groups of S/2, then of the last merge only the half-cleaners down to
      // stride 8: lanes 0..7 then hold the 8 largest (in no particular order)
      u64 a = (uint32_t)lane < nn ? stage[lane] : 0ull;
      a = nn <= 16u ? top8_network<16>(a, lane) : top8_network<32>(a, lane);
      __syncwarp();
      stage[lane] = a;
      __syncwarp();
    } else if (nn > 32) {
      warp_sort_desc(stage, (int)nn);
    }
    // nn <= 8: the staged candidates are the list.  A full list keeps its
    // smallest entry in slot 7 (the keys are distinct: one lane matches).
    if (nn >= (uint32_t)kList) {
      const u64 mine = lane < kList ? stage[lane] : ~0ull;
      const uint32_t mh = __reduce_min_sync(kFull, (uint32_t)(mine >> 32));
      const uint32_t ml = __reduce_min_sync(kFull, (uint32_t)(mine >> 32) == mh ? (uint32_t)mine : 0xffffffffu);
      const int at = __ffs(__ballot_sync(kFull, lane < kList && mine == (((u64)mh << 32) | ml))) - 1;
      const u64 last = stage[kList - 1];
      __syncwarp();
      if (lane == at && at != kList - 1) {
        stage[at] = last;
        stage[kList - 1] = mine;
      }
      __syncwarp();
    }
  }
  // word 2j: key of entry j (0 = none); word 2j + 1: its chunk-local index
  const int j = lane >> 1;
  uint32_t v = 0;
  if (lane < 2 * kList) {
    const bool has = (uint32_t)j < nn;
    const u64 k = has ? stage[j] : 0ull;
    if ((lane & 1) == 0) v = has ? (uint32_t)(k >> 32) : 0u;
    else v = (has ? key64_idx(k) : kListIdx) | (j == 0 ? flags : 0u);
    __stcg(A.rec + ((size_t)it.u * A.NCA + it.c) * kRecWords + lane, tagw(tag, v));
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// B items.
// ---------------------------------------------------------------------------
// The unit state words of a drafted unfiltered unit (loads in flight; checked
// by state_ready).
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

template <bool kBF16>
__device__ __noinline__ void b_item(const Args& A, uint32_t tag, const Item& it, const RowCfg& cfg, const UnitState& st,
                                    const unsigned char* buf) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int nb = ceil_div(it.n, kRaceBlock);
  const int e0 = it.c * G::EB;
  const bool need_race = !st.accept;
  const float* qb = reinterpret_cast<const float*>(buf + G::EB * G::es);
  float alpha_c = 0.f, myW = 0.f, myU = 0.f;
  const float m = st.m, invZ = st.invZ, c = cfg.c;
  if (!need_race) {
    // accepted draft: alpha only
    const u64 m2 = pack2(m, m), c2 = pack2(c, c), z2 = pack2(invZ, invZ);
    float a0 = 0.f, a1 = 0.f;
    for (int b = 0; b < nb; ++b) {
      float v[8], q[8];
      sload<kBF16>(buf, b, lane, v);
      sload_q(qb, b, lane, q);
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        float p0, p1;
        unpack2(mul2(exp_pair(v[j], v[j + 1], m2, c2), z2), p0, p1);
        a0 += fminf(p0, q[j]);
        a1 += fminf(p1, q[j + 1]);
      }
    }
    alpha_c = warp_sum(a0 + a1);
  }
  if (need_race) {
    const u64 m2 = pack2(m, m), c2 = pack2(c, c), z2 = pack2(invZ, invZ);
    float a8 = 0.f;
    for (int b = 0; b < nb; ++b) {
      float v[8], q[8];
      sload<kBF16>(buf, b, lane, v);
      sload_q(qb, b, lane, q);
      float w8 = 0.f, u8 = 0.f;
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        float p0, p1;
        unpack2(mul2(exp_pair(v[j], v[j + 1], m2, c2), z2), p0, p1);   // padding: -inf -> 0
        a8 += fminf(p0, q[j]) + fminf(p1, q[j + 1]);
        const float w0 = p0 - q[j], w1 = p1 - q[j + 1];
        w8 += fmaxf(w0, 0.f) + fmaxf(w1, 0.f);
        u8 += (w0 > 0.f ? p0 + q[j] : 0.f) + (w1 > 0.f ? p1 + q[j + 1] : 0.f);
      }
      const float Wb = warp_sum(w8), Ub = warp_sum(u8);
      if (lane == b) {
        myW = Wb;
        myU = Ub;
      }
    }
    alpha_c = warp_sum(a8);
  }
  Race r;
  race_init(r);
  if (need_race && myW > 0.f) {
    const uint32_t blk = (uint32_t)(e0 / kRaceBlock + lane);
    race_consider(r, myW, myU - myW, blk, block_word(A, it.row, it.pos, blk));
  }
  if (need_race) warp_race_merge(r);   // accepted: the empty race as it is
  u64* rec = A.brec + ((size_t)it.u * A.NCB + it.c) * kBRecWords;
  const uint32_t v = lane_word8(lane, __float_as_uint(alpha_c), __float_as_uint(r.s1), __float_as_uint(r.t1),
                                __float_as_uint(r.s2), __float_as_uint(r.t2), r.v1, 0u, 0u);
  if (lane < 6) __stcg(rec + lane, tagw(tag, v));
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Warps.
// ---------------------------------------------------------------------------
struct Bufs {
  unsigned char* a;
  unsigned char* b;
  unsigned long long* ba;
  unsigned long long* bb;
  uint32_t pa, pb;
  __device__ __forceinline__ void rotate() {
    unsigned char* tb = a;
    a = b;
    b = tb;
    unsigned long long* tr = ba;
    ba = bb;
    bb = tr;
    const uint32_t tp = pa;
    pa = pb;
    pb = tp;
  }
};


// A stream warp: items of the sequence, taken in order from a shared counter.
template <bool kBF16>
__device__ __noinline__ void stream(const Args& A, const Plan& P0, VShm& S, uint32_t tag, int w, uint32_t gs,
                                    uint32_t nws) {
  const int lane = threadIdx.x & 31;
  const Plan P = P0;
  Bufs B;
  B.a = S.buf[w][0];
  B.b = S.buf[w][1];
  B.ba = &S.bar[w][0];
  B.bb = &S.bar[w][1];
  B.pa = 0u;
  B.pb = 0u;
  if (lane == 0) {
    mbar_init(B.ba, 1);    // issue() orders the inits before the copies (fence.proxy.async)
    mbar_init(B.bb, 1);
  }
  __syncwarp();
  // stream warp gs starts on items gs and nws + gs; later items are taken in
  // order from one counter, one per item processed (the ticket is in flight
  // while the item is reduced)
  Item ia = map_item<kBF16>(A, P, gs);
  Item ib = map_item<kBF16>(A, P, nws + gs);
  if (lane == 0) {
    issue<kBF16>(A, ia, B.a, B.ba);
    issue<kBF16>(A, ib, B.b, B.bb);
  }
  while (ia.kind != 0) {
    uint32_t tn = 0;
    if (lane == 0 && ib.kind != 0) tn = 2u * nws + atomicAdd(&A.ws->next_item, 1u);
    const RowCfg cfg = plan_cfg(A, P, ia.row);
    u64 sw[kStateWords];
    if (ia.kind == 2) state_load(A, ia.u, sw);     // in flight during the copy wait
    if (!wait_buffer(A, B.ba, B.pa)) return;
    B.pa ^= 1u;
    if (!A.vec_logits || (ia.kind == 2 && !A.vec_q) || (ia.n & (kRaceBlock - 1)) != 0) fill_tail<kBF16>(A, ia, B.a);
    if (ia.kind == 1) {
      if (cfg.type == UT_TOPK) a_list<kBF16>(A, tag, ia, B.a, S.stage[w]);
      else a_stats<kBF16>(A, tag, ia, cfg, B.a);
    } else {
      // the unit state (bounded wait: a settle warp publishes it)
      long long spins = 0;
      while (!__all_sync(kFull, state_ok(sw, tag))) {
        if (++spins > kSpinLimit) {
          if (lane == 0) atomicOr(&A.ws->error, 1u);
          break;
        }
        __nanosleep(128);
        state_load(A, ia.u, sw);
      }
      const UnitState st = state_of(sw);
      if (!st.invalid) b_item<kBF16>(A, tag, ia, cfg, st, B.a);
    }
    __syncwarp();
    tn = __shfl_sync(kFull, tn, 0);
    Item in;
    in.kind = 0;
    if (ib.kind != 0) in = map_item<kBF16>(A, P, tn);
    if (lane == 0) issue<kBF16>(A, in, B.a, B.ba);
    ia = ib;
    ib = in;
    B.rotate();
  }
}

// A settle warp: tasks s0, s0 + nsw, ... in the order [small top-k]
// [drafted unfiltered: state][bonus positions][greedy][drafted unfiltered: B
// records].  Every task before the last group waits only for A records, so
// every state the B items wait for is published whatever the task spread.
template <bool kBF16>
__device__ __noinline__ void settle(const Args& A, const Plan& P, VShm& S, uint32_t tag, int w, uint32_t s0,
                                    uint32_t nsw, uint32_t nS) {
  const int k = A.k, k1 = A.k + 1;
  for (uint32_t t = s0; t < nS; t += nsw) {
    int s = (int)t, row, pos;
    bool finish = false;
    if (s < P.nT * k1) {
      row = (int)P.order[P.nD + s / k1];
      pos = s % k1;
    } else if ((s -= P.nT * k1) < P.nD * k) {
      row = (int)P.order[s / k];
      pos = s % k;
    } else if ((s -= P.nD * k) < P.nD) {
      row = (int)P.order[s];
      pos = k;
    } else if ((s -= P.nD) < P.nG * k1) {
      row = (int)P.order[P.nD + P.nT + s / k1];
      pos = s % k1;
    } else {
      s -= P.nG * k1;
      row = (int)P.order[s / k];
      pos = s % k;
      finish = true;
    }
    const int u = row * k1 + pos;
    const RowCfg cfg = plan_cfg(A, P, row);
    if (finish) {
      // the published state (bounded wait), then the B records
      u64 sw[kStateWords];
      state_load(A, u, sw);
      long long spins = 0;
      while (!__all_sync(kFull, state_ok(sw, tag))) {
        if (++spins > kSpinLimit) {
          if ((threadIdx.x & 31) == 0) atomicOr(&A.ws->error, 1u);
          break;
        }
        __nanosleep(256);
        state_load(A, u, sw);
      }
      const UnitState st = state_of(sw);
      if (!st.invalid) fin_b<kBF16>(A, tag, u, row, pos, cfg, st);
    } else if (cfg.type == UT_TOPK) {
      topk_settle<kBF16>(A, tag, *reinterpret_cast<TopkScratch*>(S.buf[w][0]), u, row, pos, cfg);
    } else {
      UnitState st;
      fin_stats<kBF16>(A, tag, u, row, pos, cfg, st);
    }
  }
}

// General-path units, taken by the two half-CTA groups.
template <bool kBF16>
__device__ __noinline__ void general_phase(const Args& A, const Plan& P, VShm& S) {
  const int k1 = A.k + 1;
  const int nGU = P.nX * k1;
  const int gbase = P.nD + P.nT + P.nG;
  const int grp = threadIdx.x >> 8;
  while (true) {
    if (ctid() == 0) S.gtask[grp] = (int)atomicAdd(&A.ws->gnext, 1u);
    csync();
    const int g = S.gtask[grp];
    csync();
    if (g >= nGU) break;
    const int row = (int)P.order[gbase + g / k1], pos = g % k1;
    unit_general<kBF16>(A, S.gen[grp], S.tag, row * k1 + pos, row, pos, plan_cfg(A, P, row));
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kAllThreads, 1) verify_kernel(const Args A) {
  using G = Geo<kBF16>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  VShm& S = *reinterpret_cast<VShm*>(smem_raw);
  const int w = threadIdx.x >> 5;
  if (threadIdx.x == 0) S.tag = __ldcg(&A.ws->epoch) + 1u;
  Plan P;
  if (!A.global_order) {
    build_order_smem(A, S.order, S.cfg, S.ord);     // synchronises the CTA
    P.order = S.order;
    P.cfg = S.cfg;
    P.nD = S.ord.n_class[UT_DENSE];
    P.nT = S.ord.n_class[UT_TOPK];
    P.nG = S.ord.n_class[UT_GREEDY];
    P.nX = S.ord.n_class[UT_GENERAL];
  } else {
    __syncthreads();
    if (blockIdx.x == 0) build_order_global(A, S.ord, S.tag);
    if (threadIdx.x == 0) {
      long long spins = 0;
      while (load_acquire(&A.ws->order_tag) != S.tag) {
        if (++spins > kSpinLimit) {
          atomicOr(&A.ws->error, 8u);
          break;
        }
        __nanosleep(128);
      }
    }
    __syncthreads();
    P.order = A.order;
    P.cfg = nullptr;
    P.nD = (int)__ldcg(&A.ws->n_class[UT_DENSE]);
    P.nT = (int)__ldcg(&A.ws->n_class[UT_TOPK]);
    P.nG = (int)__ldcg(&A.ws->n_class[UT_GREEDY]);
    P.nX = (int)__ldcg(&A.ws->n_class[UT_GENERAL]);
  }
  const uint32_t tag = S.tag;
  P.NCA = ceil_div(A.V, G::EA);
  P.NCB = ceil_div(A.V, G::EB);
  P.sDD = (uint32_t)(P.nD * A.k * P.NCA);
  P.sTK = (uint32_t)(P.nT * (A.k + 1) * P.NCA);
  P.sDB = (uint32_t)(P.nD * P.NCA);
  P.sB = (uint32_t)(P.nD * A.k * P.NCB);
  P.sGR = (uint32_t)(P.nG * (A.k + 1) * P.NCA);
  const uint32_t nw = (uint32_t)A.n_ctas * kSW;
  // settle warps are the warps on the SMs' first schedulers (w % 4 == 0),
  // four per SM: consecutive tasks (one class, neighbouring rows) settle on
  // one SM, whose first scheduler then runs no stream warp, and the other
  // schedulers run stream code only
  const uint32_t g = (w & 3) == 0 ? blockIdx.x * 4u + (uint32_t)(w >> 2)
                                   : 4u * (uint32_t)A.n_ctas + (uint32_t)((w & 3) - 1) * (4u * (uint32_t)A.n_ctas) +
                                         (uint32_t)(w >> 2) * (uint32_t)A.n_ctas + blockIdx.x;
  const uint32_t nS = (uint32_t)(2 * P.nD * A.k + P.nT * (A.k + 1) + P.nD + P.nG * (A.k + 1));
  const uint32_t nsw = min(nS, nw / 4u);
  if (g < nsw) {
    settle<kBF16>(A, P, S, tag, w, g, nsw, nS);
  } else {
    stream<kBF16>(A, P, S, tag, w, g - nsw, nw - nsw);
  }
  if (P.nX > 0) {
    __syncthreads();
    general_phase<kBF16>(A, P, S);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t d = atomicAdd(&A.ws->ctas_done, 1u);
    if (d == (uint32_t)A.n_ctas - 1u) {
      A.ws->gnext = 0u;
      A.ws->next_item = 0u;
      A.ws->ctas_done = 0u;
      A.ws->epoch = tag;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
template <bool kBF16>
int launch_verify(const Args& A0, cudaStream_t stream) {
  static std::mutex mu;
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  int n = 0;
  auto kern = verify_kernel<kBF16>;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
      int per_sm = 0, sms = 0;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(VShm)) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kAllThreads, sizeof(VShm)) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || per_sm <= 0) {
        cudaGetLastError();
        return SPEC_E_CUDA;
      }
      cached[dev] = per_sm * sms;
    }
    n = cached[dev];
  }
  Args A = A0;
  A.n_ctas = n;
  A.global_order = A.B > kOrderSmem ? 1 : 0;
  // cooperative launch: every CTA is resident, so every wait between warps ends
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)A.n_ctas);
  cfg.blockDim = dim3(kAllThreads);
  cfg.dynamicSmemBytes = sizeof(VShm);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, A) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  return SPEC_OK;
}

template int launch_verify<true>(const Args&, cudaStream_t);
template int launch_verify<false>(const Args&, cudaStream_t);

}  // namespace specv
