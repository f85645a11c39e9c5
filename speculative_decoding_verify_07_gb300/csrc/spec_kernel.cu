// spec_verify: the verify kernel (sm_103a).
//
// One persistent CTA of 16 warps per SM, launched cooperatively (all CTAs
// resident), in two phases split by one grid barrier:
//   * Stream phase.  Every warp owns two 6 KB shared-memory buffers and has
//     the copy engine stream its next item into one (cp.async.bulk completed
//     on an mbarrier) while it reduces the other with warp collectives.  An A
//     item is a chunk of one unit's logits (3072 bf16 / 1536 fp32): max and
//     first argmax, the softmax sum relative to the chunk max, at an
//     unfiltered bonus position the level-1 race of the chunk's 256-entry
//     blocks, for a small top-k the maxima of its 64-entry super-groups.
//     Items are dealt round robin over the warps of all SMs; a warp stores
//     its records with plain stores and takes no ticket.
//   * Settle phase.  Each settle task is one unit, settled by one warp
//     (spec_settle.cuh): drafted unfiltered units first (they publish the
//     state the B items wait for), then small top-k units, bonus positions
//     and greedy units.  The other warps stream the B items of the drafted
//     unfiltered units (1024 bf16 / 768 fp32 logits, from L2, plus q):
//     alpha = sum min(p, q) and the level-1 race of the residual; each warp
//     takes a contiguous range, reads a unit's state once per run, and the
//     warp that completes a unit settles it.  Rows that need a global
//     threshold search (spec_general.cuh) are taken last by half-CTA groups.
// The last settled unit of a row resolves the accept chain and writes the
// row's outputs.  Every wait is bounded and ends with an error bit; reductions
// have a fixed order and no floating-point atomics are used, so results are
// bit-reproducible.
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
constexpr int kStage = 64;             // per-warp staging floats (super-group maxima of an item)
constexpr unsigned kFull = 0xffffffffu;
static_assert(Geo<true>::SPI <= kStage && Geo<false>::SPI <= kStage, "staging too small");
static_assert(kAllThreads == 2 * kThreads, "two general-path groups per CTA");

struct OrderScratch {
  int n_class[4];
  int run[4];
  int scan[kSW][4];
};

struct alignas(128) VShm {
  union {
    unsigned char buf[kSW][2][kSlot];  // stream buffers; a settle warp's pair is its top-k scratch
    GenShm gen[2];                     // general-path groups, after the settle phase
  };
  unsigned long long bar[kSW][2];
  float stage[kSW][kStage];
  uint32_t order[kOrderSmem];
  RowPack cfg[kOrderSmem];
  OrderScratch ord;
  int gtask[2];
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
// workspace before the grid barrier; the other CTAs read them after it.
__device__ __noinline__ void build_order_global(const Args& A, OrderScratch& O) {
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
}

// ---------------------------------------------------------------------------
// Work items.
// ---------------------------------------------------------------------------
struct Plan {
  const uint32_t* order;
  const RowPack* cfg;       // per-row configs in shared memory (null: classify from the parameters)
  int nD, nT, nG, nX;       // rows: unfiltered, small top-k, greedy, general
  int NCA, NCB;
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

// A item of ticket t in unit order (every unit, no configuration needed).
template <bool kBF16>
__device__ __forceinline__ Item map_a_raw(const Args& A, int NCA, uint32_t t) {
  using G = Geo<kBF16>;
  Item it;
  it.kind = 0;
  if (t >= (uint32_t)A.U * (uint32_t)NCA) return it;
  it.u = (int)(t / (uint32_t)NCA);
  it.c = (int)t - it.u * NCA;
  it.row = it.u / (A.k + 1);
  it.pos = it.u - it.row * (A.k + 1);
  it.n = min(G::EA, A.V - it.c * G::EA);
  it.reread = 1;
  it.kind = 1;
  return it;
}

// The next A item from ticket *t on (step nw), skipping rows of the general
// path; reread marks drafted unfiltered units, whose B items read the logits again.
template <bool kBF16>
__device__ __forceinline__ Item next_a(const Args& A, const Plan& P, uint32_t& t, uint32_t nw) {
  while (true) {
    Item it = map_a_raw<kBF16>(A, P.NCA, t);
    t += nw;
    if (it.kind == 0) return it;
    const RowCfg cfg = plan_cfg(A, P, it.row);
    if (cfg.type == UT_GENERAL) continue;
    it.reread = (cfg.type == UT_DENSE && it.pos < A.k) ? 1 : 0;
    return it;
  }
}

template <bool kBF16>
__device__ __forceinline__ Item map_b(const Args& A, const Plan& P, uint32_t t, uint32_t end) {
  using G = Geo<kBF16>;
  Item it;
  it.kind = 0;
  if (t >= end) return it;
  const int j = (int)(t / (uint32_t)P.NCB);
  it.c = (int)t - j * P.NCB;
  it.row = (int)P.order[j / A.k];
  it.pos = j % A.k;
  it.u = it.row * (A.k + 1) + it.pos;
  it.n = min(G::EB, A.V - it.c * G::EB);
  it.kind = 2;
  it.reread = 0;
  return it;
}

// The race helpers run once per item here: out of line, to keep the
// streaming loops' registers free.
static __device__ __noinline__ void race_consider_once(Race& r, float w, float tq, uint32_t v, uint32_t word) {
  race_consider(r, w, tq, v, word);
}
static __device__ __noinline__ void warp_race_merge_once(Race& r) { warp_race_merge(r); }

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

// Maximum (NaN-propagating) of a lane's two halves of block b: slots 0..3
// (entries 4l..4l+3) and slots 4..7 (entries 128+4l..128+4l+3).
template <bool kBF16>
__device__ __forceinline__ void shalf_max(const unsigned char* buf, int b, int l, float& h0, float& h1) {
  if (kBF16) {
    const uint2 a = *reinterpret_cast<const uint2*>(buf + (b * kRaceBlock + 4 * l) * 2);
    const uint2 c = *reinterpret_cast<const uint2*>(buf + (b * kRaceBlock + 128 + 4 * l) * 2);
    const uint32_t ma = max_nan_bf16x2(a.x, a.y), mc = max_nan_bf16x2(c.x, c.y);
    h0 = max_nan(bf16_lo(ma), bf16_hi(ma));
    h1 = max_nan(bf16_lo(mc), bf16_hi(mc));
  } else {
    float v[8];
    sload<false>(buf, b, l, v);
    h0 = max_nan(max_nan(v[0], v[1]), max_nan(v[2], v[3]));
    h1 = max_nan(max_nan(v[4], v[5]), max_nan(v[6], v[7]));
  }
}

// Reduce A item `it`; the record (valid in lane 0) or, for a small top-k, the
// super-group maxima (in `stage`) are stored by the caller.
template <bool kBF16>
__device__ void a_compute(const Args& A, const Item& it, const RowCfg& cfg, const unsigned char* buf, float* stage,
                          ChunkRec& rec) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int nb = ceil_div(it.n, kRaceBlock);
  const int e0 = it.c * G::EA;
  if (cfg.type == UT_TOPK) {
    // maxima of the 64-entry super-groups: super-group r of block b holds
    // entries [64r, 64r+64), i.e. the first (r < 2) or second half of lanes
    // 16(r%2)..16(r%2)+15
#pragma unroll 4
    for (int b = 0; b < nb; ++b) {
      float h0, h1;
      shalf_max<kBF16>(buf, b, lane, h0, h1);
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        h0 = max_nan(h0, __shfl_xor_sync(kFull, h0, o));
        h1 = max_nan(h1, __shfl_xor_sync(kFull, h1, o));
      }
      if ((lane & 15) == 0) {
        stage[b * 4 + (lane >> 4)] = h0;
        stage[b * 4 + 2 + (lane >> 4)] = h1;
      }
    }
    __syncwarp();
    for (int s = nb * 4 + lane; s < G::SPI; s += 32) stage[s] = -INFINITY;
    __syncwarp();
    return;
  }
  // greedy and unfiltered: max and first argmax, then the softmax sum
  // relative to the chunk max; at an unfiltered bonus position also the
  // block weights and the level-1 race of the chunk's blocks
  float lm = -INFINITY;
  int lb = 0;
  bool nan = false;
#pragma unroll 4
  for (int b = 0; b < nb; ++b) {
    float h0, h1;
    shalf_max<kBF16>(buf, b, lane, h0, h1);
    const float gm = max_nan(h0, h1);
    nan |= gm != gm;
    if (gm > lm) {
      lm = gm;
      lb = b;
    }
  }
  nan = __any_sync(kFull, nan);
  const float mc = warp_max_f(lm);
  uint32_t idx = 0xffffffffu;
  if (lm == mc) {
    float v[8];
    sload<kBF16>(buf, lb, lane, v);
#pragma unroll
    for (int j = 7; j >= 0; --j)
      if (v[j] == lm) idx = (uint32_t)(e0 + slot_entry(lb, lane, j));
  }
  idx = warp_min_u32(idx);
  float z = 0.f;
  Race r;
  race_init(r);
  const bool live = !nan && mc > -INFINITY && mc < INFINITY;
  const bool bonus = cfg.type == UT_DENSE && it.pos == A.k;
  if (live) {
    const float c = cfg.c;
    if (!bonus) {
      float z0 = 0.f, z1 = 0.f;
#pragma unroll 2
      for (int b = 0; b < nb; ++b) {
        float v[8];
        sload<kBF16>(buf, b, lane, v);
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          z0 += ex2((v[j] - mc) * c);
          z1 += ex2((v[j + 1] - mc) * c);
        }
      }
      z = warp_sum(z0 + z1);
    } else {
      float myW = 0.f;
      for (int b = 0; b < nb; ++b) {
        float v[8];
        sload<kBF16>(buf, b, lane, v);
        float s8 = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) s8 += ex2((v[j] - mc) * c);
        const float W = warp_sum(s8);
        z += W;
        if (lane == b) myW = W;
      }
      if (myW > 0.f) {
        const uint32_t blk = (uint32_t)(e0 / kRaceBlock + lane);
        race_consider_once(r, myW, 0.f, blk, block_word(A, it.row, it.pos, blk));
      }
      warp_race_merge_once(r);
    }
  }
  {
    rec.m = nan ? __uint_as_float(0x7fc00000u) : mc;
    rec.amax = idx;
    rec.z = z;
    rec.pad0 = 0;
    rec.s1 = r.s1;
    rec.t1 = r.t1;
    rec.s2 = r.s2;
    rec.t2 = r.t2;
    rec.v1 = r.v1;
    rec.pad[0] = rec.pad[1] = rec.pad[2] = 0;
  }
}

__device__ __forceinline__ UnitState load_state(const Args& A, int u) {
  UnitState st;
  st.m = __ldcg(&A.ust[u].m);
  st.invZ = __ldcg(&A.ust[u].invZ);
  st.lnZ = __ldcg(&A.ust[u].lnZ);
  st.lp_x = __ldcg(&A.ust[u].lp_x);
  st.accept = __ldcg(&A.ust[u].accept);
  st.flags = __ldcg(&A.ust[u].flags);
  st.invalid = __ldcg(&A.ust[u].invalid);
  st.am = __ldcg(&A.ust[u].am);
  return st;
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

template <bool kBF16>
__device__ __noinline__ void fin_b(const Args& A, const Item& it, const RowCfg& cfg, const UnitState& st) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int u = it.u, row = it.row, pos = it.pos;
  const int NC = ceil_div(A.V, G::EB);
  const BRec* R = A.brec + (size_t)u * A.NCB;
  const bool need_race = !st.accept;
  float al = 0.f;
  Race a;
  race_init(a);
  for (int c = lane; c < NC; c += 32) {
    al += __ldcg(&R[c].alpha);
    if (need_race) {
      Race rb;
      rb.s1 = __ldcg(&R[c].s1);
      rb.t1 = __ldcg(&R[c].t1);
      rb.s2 = __ldcg(&R[c].s2);
      rb.t2 = __ldcg(&R[c].t2);
      rb.v1 = __ldcg(&R[c].v1);
      rb.s1lo = 0.f;
      race_merge(a, rb);
    }
  }
  const float alpha_v = warp_sum(al);
  uint32_t draw_flags = 0;
  uint32_t y = 0xffffffffu;
  if (need_race) {
    warp_race_merge(a);
    if (a.s1 >= 0.f) {
      const Race l2 = race_in_block<kBF16>(A, row, pos, a.v1, st.m, cfg.c, st.invZ, RW_RESIDUAL, nullptr);
      y = l2.v1;
      if (draw_margin(a) || draw_margin(l2)) draw_flags |= SPEC_F_MARGIN_DRAW;
    } else {
      draw_flags |= SPEC_F_RESIDUAL_EMPTY;
      bool mg = false;
      y = warp_draw_p<kBF16>(A, row, pos, st.m, cfg.c, &mg);
      if (mg) draw_flags |= SPEC_F_MARGIN_DRAW;
    }
  }
  if (lane == 0) {
    UnitRecord rec = empty_record(st.flags);
    rec.accept = st.accept;
    rec.lp_x = st.lp_x;
    rec.alpha = alpha_v;
    if (need_race) {
      const uint32_t yy = y < (uint32_t)A.V ? y : (uint32_t)st.am;
      rec.y = (int32_t)yy;
      rec.lp_y = (load_logit(A, kBF16, (size_t)u * A.V + yy) - st.m) * cfg.invT - st.lnZ;
      rec.draw_flags = draw_flags;
    }
    A.b_ticket[u] = 0;
    A.ready[u] = 0;
    commit_record(A, u, row, rec);
  }
  __syncwarp();
}

template <bool kBF16>
__device__ void b_compute(const Args& A, const Item& it, const RowCfg& cfg, const UnitState& st, const unsigned char* buf,
                          BRec& br) {
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
    float a0 = 0.f, a1 = 0.f;
    for (int b = 0; b < nb; ++b) {
      float v[8], q[8];
      sload<kBF16>(buf, b, lane, v);
      sload_q(qb, b, lane, q);
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        a0 += fminf(ex2((v[j] - m) * c) * invZ, q[j]);
        a1 += fminf(ex2((v[j + 1] - m) * c) * invZ, q[j + 1]);
      }
    }
    alpha_c = warp_sum(a0 + a1);
  }
  for (int b = 0; need_race && b < nb; ++b) {
    float v[8], q[8];
    sload<kBF16>(buf, b, lane, v);
    sload_q(qb, b, lane, q);
    float a8 = 0.f, w8 = 0.f, u8 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float p = ex2((v[j] - m) * c) * invZ;   // padding: -inf -> 0
      a8 += fminf(p, q[j]);
      const float w = p - q[j];
      if (w > 0.f) {
        w8 += w;
        u8 += p + q[j];
      }
    }
    alpha_c += warp_sum(a8);
    const float Wb = warp_sum(w8), Ub = warp_sum(u8);
    if (lane == b) {
      myW = Wb;
      myU = Ub;
    }
  }
  Race r;
  race_init(r);
  if (need_race && myW > 0.f) {
    const uint32_t blk = (uint32_t)(e0 / kRaceBlock + lane);
    race_consider_once(r, myW, myU - myW, blk, block_word(A, it.row, it.pos, blk));
  }
  warp_race_merge_once(r);
  br.alpha = alpha_c;
  br.s1 = r.s1;
  br.t1 = r.t1;
  br.s2 = r.s2;
  br.t2 = r.t2;
  br.v1 = r.v1;
  br.pad[0] = br.pad[1] = 0;
}



// ---------------------------------------------------------------------------
// Phases.
// ---------------------------------------------------------------------------
// Results of A item `it` (plain stores; the grid barrier publishes them).
template <bool kBF16>
__device__ __forceinline__ void store_a(const Args& A, const Item& it, const RowCfg& cfg, const ChunkRec& rec,
                                        const float* stage) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  if (cfg.type == UT_TOPK) {
    float* dst = A.smax + (size_t)it.u * A.NSM + (size_t)it.c * G::SPI;
    for (int s = lane; s < G::SPI; s += 32) dst[s] = stage[s];
  } else if (lane == 0) {
    A.crec[(size_t)it.u * A.NCA + it.c] = rec;
  }
  __syncwarp();
}

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

// Stream phase of one warp: A items t0, t0 + nw, ... (the first two are
// already posted in ia, ib).
template <bool kBF16>
__device__ __noinline__ void stream_a(const Args& A, const Plan& P, VShm& S, int w, Bufs& B, Item ia, Item ib,
                                      uint32_t t, uint32_t nw) {
  while (ia.kind != 0) {
    if (!wait_buffer(A, B.ba, B.pa)) return;
    B.pa ^= 1u;
    const RowCfg cfg = plan_cfg(A, P, ia.row);
    if (cfg.type != UT_GENERAL) {
      if (!A.vec_logits || (ia.n & (kRaceBlock - 1)) != 0) fill_tail<kBF16>(A, ia, B.a);
      ChunkRec rec;
      a_compute<kBF16>(A, ia, cfg, B.a, S.stage[w], rec);
      store_a<kBF16>(A, ia, cfg, rec, S.stage[w]);
    }
    __syncwarp();
    Item in;
    in.kind = 0;
    if (ib.kind != 0) in = next_a<kBF16>(A, P, t, nw);
    if ((threadIdx.x & 31) == 0) issue<kBF16>(A, in, B.a, B.ba);
    ia = ib;
    ib = in;
    B.rotate();
  }
}

// One settle task: drafted unfiltered units, small top-k units, bonus
// positions, greedy units.
template <bool kBF16>
__device__ __noinline__ void settle_task(const Args& A, const Plan& P, VShm& S, int w, int s) {
  const int k = A.k, k1 = A.k + 1;
  int row, pos;
  if (s < P.nD * k) {
    row = (int)P.order[s / k];
    pos = s % k;
  } else if ((s -= P.nD * k) < P.nT * k1) {
    row = (int)P.order[P.nD + s / k1];
    pos = s % k1;
  } else if ((s -= P.nT * k1) < P.nD) {
    row = (int)P.order[s];
    pos = k;
  } else {
    s -= P.nD;
    row = (int)P.order[P.nD + P.nT + s / k1];
    pos = s % k1;
  }
  const int u = row * k1 + pos;
  const RowCfg cfg = plan_cfg(A, P, row);
  if (cfg.type == UT_TOPK) topk_settle<kBF16>(A, *reinterpret_cast<TopkScratch*>(S.buf[w][0]), u, row, pos, cfg);
  else fin_stats<kBF16>(A, u, row, pos, cfg);
}

// B items of one warp: the contiguous range [tb, end).
template <bool kBF16>
__device__ __noinline__ void stream_b(const Args& A, const Plan& P, Bufs& B, uint32_t tb, uint32_t end) {
  const int lane = threadIdx.x & 31;
  Item ia = map_b<kBF16>(A, P, tb, end);
  Item ib = map_b<kBF16>(A, P, tb + 1, end);
  tb += 2;
  if (lane == 0) {
    issue<kBF16>(A, ia, B.a, B.ba);
    issue<kBF16>(A, ib, B.b, B.bb);
  }
  Item run;                  // the unit whose chunks this warp is processing
  run.kind = 0;
  uint32_t run_n = 0;
  UnitState st;
  memset(&st, 0, sizeof(st));
  RowCfg cfg = classify(A.params[0], A.V);
  const uint32_t lastB = (uint32_t)P.NCB;
  auto close_run = [&]() {
    // add this warp's chunks of the finished run to the unit's ticket; the
    // warp that completes the unit settles it
    uint32_t old = 0;
    if (lane == 0) old = atomic_add_acq_rel(&A.b_ticket[run.u], run_n);
    old = __shfl_sync(kFull, old, 0);
    __syncwarp();
    if (old + run_n == lastB && !st.invalid) fin_b<kBF16>(A, run, cfg, st);
    else if (old + run_n == lastB && lane == 0) {
      A.b_ticket[run.u] = 0;
      A.ready[run.u] = 0;
    }
    run.kind = 0;
  };
  while (ia.kind != 0) {
    if (run.kind != 0 && run.u != ia.u) close_run();
    if (run.kind == 0) {
      // the unit state (bounded wait: a settle warp publishes it)
      if (lane == 0) {
        long long spins = 0;
        while (load_acquire(&A.ready[ia.u]) == 0u) {
          if (++spins > kSpinLimit) {
            atomicOr(&A.ws->error, 1u);
            break;
          }
          __nanosleep(64);
        }
      }
      __syncwarp();
      st = load_state(A, ia.u);
      cfg = plan_cfg(A, P, ia.row);
      run = ia;
      run_n = 0;
    }
    if (!wait_buffer(A, B.ba, B.pa)) return;
    B.pa ^= 1u;
    if (!A.vec_logits || !A.vec_q || (ia.n & (kRaceBlock - 1)) != 0) fill_tail<kBF16>(A, ia, B.a);
    if (!st.invalid) {
      BRec br;
      b_compute<kBF16>(A, ia, cfg, st, B.a, br);
      if (lane == 0) A.brec[(size_t)ia.u * A.NCB + ia.c] = br;
    }
    __syncwarp();
    ++run_n;
    Item in = map_b<kBF16>(A, P, tb, end);
    ++tb;
    if (lane == 0) issue<kBF16>(A, in, B.a, B.ba);
    ia = ib;
    ib = in;
    B.rotate();
  }
  if (run.kind != 0) close_run();
}

// Grid barrier (all CTAs are resident: cooperative launch).  Bounded.
__device__ __forceinline__ void grid_barrier(const Args& A) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&A.ws->arrived, 1u);
    long long spins = 0;
    while (load_acquire(&A.ws->arrived) < (uint32_t)A.n_ctas) {
      if (++spins > kSpinLimit) {
        atomicOr(&A.ws->error, 4u);
        break;
      }
      __nanosleep(64);
    }
  }
  __syncthreads();
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
    unit_general<kBF16>(A, S.gen[grp], row * k1 + pos, row, pos, plan_cfg(A, P, row));
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kAllThreads, 1) verify_kernel(const Args A) {
  using G = Geo<kBF16>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  VShm& S = *reinterpret_cast<VShm*>(smem_raw);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t nw = (uint32_t)A.n_ctas * kSW;
  const uint32_t g = (uint32_t)w * (uint32_t)A.n_ctas + blockIdx.x;   // warps of a round spread over the SMs
  Bufs B;
  B.a = S.buf[w][0];
  B.b = S.buf[w][1];
  B.ba = &S.bar[w][0];
  B.bb = &S.bar[w][1];
  B.pa = 0u;
  B.pb = 0u;
  const int NCA = ceil_div(A.V, G::EA);
  // the first two A items go out before anything else
  Item ia = map_a_raw<kBF16>(A, NCA, g);
  Item ib = map_a_raw<kBF16>(A, NCA, g + nw);
  if (lane == 0) {
    mbar_init(B.ba, 1);
    mbar_init(B.bb, 1);
    fence_mbar_init();
    issue<kBF16>(A, ia, B.a, B.ba);
    issue<kBF16>(A, ib, B.b, B.bb);
  }
  Plan P;
  P.NCA = NCA;
  P.NCB = ceil_div(A.V, G::EB);
  if (!A.global_order) {
    build_order_smem(A, S.order, S.cfg, S.ord);
    P.order = S.order;
    P.cfg = S.cfg;
  } else {
    if (blockIdx.x == 0) build_order_global(A, S.ord);
    P.order = A.order;
    P.cfg = nullptr;
  }
  __syncthreads();
  stream_a<kBF16>(A, P, S, w, B, ia, ib, g + 2 * nw, nw);
  grid_barrier(A);
  if (!A.global_order) {
    P.nD = S.ord.n_class[UT_DENSE];
    P.nT = S.ord.n_class[UT_TOPK];
    P.nG = S.ord.n_class[UT_GREEDY];
    P.nX = S.ord.n_class[UT_GENERAL];
  } else {
    P.nD = (int)__ldcg(&A.ws->n_class[UT_DENSE]);
    P.nT = (int)__ldcg(&A.ws->n_class[UT_TOPK]);
    P.nG = (int)__ldcg(&A.ws->n_class[UT_GREEDY]);
    P.nX = (int)__ldcg(&A.ws->n_class[UT_GENERAL]);
  }
  // settle tasks on the first warps of every SM, B items on the rest
  const uint32_t nS = (uint32_t)(P.nD * A.k + P.nT * (A.k + 1) + P.nD + P.nG * (A.k + 1));
  const uint32_t nSW = min(nS, nw / 2u);
  if (g < nSW) {
    for (uint32_t s = g; s < nS; s += nSW) settle_task<kBF16>(A, P, S, w, (int)s);
  } else {
    const uint32_t totalB = (uint32_t)(P.nD * A.k) * (uint32_t)P.NCB;
    const uint32_t nBW = nw - nSW;
    const uint32_t per = (totalB + nBW - 1) / nBW;
    const uint32_t tb = min(totalB, (g - nSW) * per);
    const uint32_t end = min(totalB, tb + per);
    if (tb < end) stream_b<kBF16>(A, P, B, tb, end);
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
      A.ws->arrived = 0u;
      A.ws->ctas_done = 0u;
      for (int i = 0; i < 4; ++i) A.ws->n_class[i] = 0u;
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
  // cooperative launch: every CTA is resident, so the grid barrier ends
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
