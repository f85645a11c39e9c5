// spec_verify: the verify kernel (sm_103a).
//
// One persistent CTA of 12 warps per SM, launched cooperatively (every CTA
// is resident, so warps may wait on one another; every such wait is
// bounded).  CTAs take one of two roles, so that each SM runs one kind of
// code and keeps it in its instruction cache:
//   * Stream CTAs (5 in 6).  Each of their 12 warps owns two 8 KB
//     shared-memory buffers and has the copy engine fill one (cp.async.bulk
//     completed on an mbarrier) while it reduces the other.  The tiles of
//     all units form one sequence of segments: A tiles of small top-k rows
//     (their settles are the longest, so they come first); unfiltered rows
//     in waves (each wave's drafted positions, then its bonus positions),
//     the B tiles of a wave placed a fixed number of items after its A
//     tiles; A tiles of greedy rows.  Item t belongs to stream CTA t mod
//     (stream CTAs), whose warps take its items in order from a
//     shared-memory counter; a unit's tiles are taken in a rotated order.
//     An A tile (4096 bf16 / 2048 fp32 logits of one unit) yields the tile
//     max, the softmax sum relative to it, the first argmax (greedy), the
//     level-1 race of its 256-entry blocks (bonus positions) or the 8
//     largest entries in the total order (small top-k).  A B tile (1280 /
//     1024 logits, read again from L2, plus q) computes alpha = sum min(p, q)
//     and the level-1 race of the residual from the unit's published state.
//     After a tile's record the warp adds one to the unit's tile count (a
//     reduction nobody waits for).
//   * Settle CTAs (1 in 6, every stride-th block).  Their warps take
//     the settle tasks -- one per unit after its A tiles, one per drafted
//     unfiltered unit after its B tiles -- in the order of the sequence,
//     task t to settle CTA t mod (settle CTAs); a warp waits for its task's tile
//     count, settles the unit (spec_settle.cuh) and clears the count.  Tasks
//     come in the order their tiles do, and a B tile only waits for a state
//     that an earlier task publishes, so every wait ends.  The last settled
//     unit of a row resolves its accept chain and writes the row's outputs.
// Rows with top-p and no top-k then run the grid-wide top-p passes
// (spec_topp.cuh, every warp of every CTA, grid barriers between passes);
// rows with a top-k above the candidate-list limit are taken next by the
// CTAs' first 256 threads (spec_general.cuh), and the fused commit
// (spec_fused.cuh) follows.  Each CTA numbers the call from a count of the
// CTAs that entered earlier calls; results pass between warps as 64-bit
// words tagged with the call's number, and the call counts in one of two
// counter sets by its parity (zeroing the other for the next call), so no
// CTA waits at the end to reset anything.  Reductions have a fixed order and
// no floating-point atomics are used, so results are bit-reproducible.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "spec_common.cuh"
#include "spec_fused.cuh"
#include "spec_general.cuh"
#include "spec_host.h"
#include "spec_settle.cuh"
#include "spec_topp.cuh"

namespace specv {

constexpr int kNW = kCtaWarps;         // warps per CTA (stream warps of a stream CTA, settle warps of a settle CTA)
constexpr int kAllThreads = kNW * 32;
constexpr int kOrderSmem = 256;        // batches up to this many rows keep order and configs in shared memory
constexpr int kStage = 64;             // per-warp staging of a top-k tile's candidates
constexpr int kMaxWaves = 40;
constexpr int kMaxSeg = 4 * kMaxWaves + 8;   // segments of the item sequence (2 A and at most 2 more per wave, 2 classes)
constexpr int kSettleEvery = 6;        // one settle CTA per this many CTAs
constexpr unsigned kFull = 0xffffffffu;
static_assert(kAllThreads >= kOrderSmem, "one placement round for a shared-memory order");
static_assert(kAllThreads >= kThreads, "the general phase uses the first kThreads threads");

// A segment of the item sequence: `nrows` rows from index `first` of the
// class order, each contributing the units at positions pos_lo ..
// pos_lo + upr - 1, each unit `tiles` tiles of one kind.
struct Seg {
  uint32_t start;     // first item of the segment
  uint32_t first;
  uint32_t nrows;
  uint32_t packed;    // tiles | pos_lo << 16 | upr << 21 | kind << 26 (0 A, 1 B)
};

constexpr int kOrderWarps = kOrderSmem / 32;   // warps that hold a row of a shared-memory order
static_assert(kOrderWarps == 8, "class counts are read as two uint4 per class");

struct OrderScratch {
  int n_class[kClasses];
  int run[kClasses];
  int scan[kNW][kClasses];
  alignas(16) uint32_t cnt[kClasses][kOrderWarps];   // shared-memory order: rows per class and warp
};

struct alignas(128) VShm {
  union {
    struct {
      unsigned char buf[kNW][2][kSlot];  // stream buffers
      u64 stage[kNW][kStage];            // top-k tile staging
    } s;
    TopkScratch tk[kNW];                 // settle scratch (settle CTAs)
    struct {
      GenShm gen;                        // general-path group, after the roles
      alignas(128) unsigned char ring[kGRing][kGSlot];   // its row chunks
      unsigned long long bar[kGRing];
    } g;
  };
  unsigned long long bar[kNW][2];
  unsigned long long cbar[kNW][2];       // fused commit: the warps' copy barriers
  uint32_t broken[kNW];                  // a copy wait of the warp gave up: its buffers are not used again
  uint32_t ticket;                       // the stream CTA's item counter
  Seg seg[kMaxSeg];
  uint32_t tstart[kMaxSeg];              // first settle task of each segment
  uint32_t bready[kMaxWaves];            // segment building: when each wave's B tiles fall due
  uint32_t order[kOrderSmem];
  RowPack cfg[kOrderSmem];
  OrderScratch ord;
  int nseg;
  uint32_t ntasks;
  int gtask;
  uint32_t tag;
};

static_assert(sizeof(VShm) <= 232448, "shared memory of a CTA exceeds 227 KB");

// ---------------------------------------------------------------------------
// Row order: rows of each class, stably, as [unfiltered][small top-k]
// [general][top-p][greedy].
// ---------------------------------------------------------------------------
__device__ __forceinline__ int class_base(const OrderScratch& O, int cl) {
  const int nD = O.n_class[UT_DENSE], nT = O.n_class[UT_TOPK], nX = O.n_class[UT_GENERAL],
            nP = O.n_class[UT_TOPP];
  return cl == UT_DENSE ? 0
       : cl == UT_TOPK ? nD
       : cl == UT_GENERAL ? nD + nT
       : cl == UT_TOPP ? nD + nT + nX
                       : nD + nT + nX + nP;
}

// Stable placement of one round of kAllThreads rows (cl < 0: no row).
__device__ __forceinline__ void place_round(uint32_t* order, OrderScratch& O, int r, int cl) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  unsigned mine = 0;
#pragma unroll
  for (int t = 0; t < kClasses; ++t) {
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
  if (tid < kClasses) {
    int s = 0;
    for (int ww = 0; ww < kNW; ++ww) s += O.scan[ww][tid];
    O.run[tid] += s;
  }
  __syncthreads();
}

// Batches of up to kOrderSmem rows: every CTA classifies the rows into
// shared memory (thread r loads row r's parameters) and places them by
// class with warp ballots; the warps' class counts meet behind one barrier.
// Returns with the counts of this thread's row class set up for placement;
// the caller places the row after the barrier (order_place_smem).
struct SmemPlace {
  int cl;          // the thread's row class (-1: no row)
  unsigned mine;   // the lanes of the thread's warp in that class
};
__device__ __forceinline__ SmemPlace order_classify_smem(const Args& A, RowPack* cfgs, OrderScratch& O) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  SmemPlace sp;
  sp.cl = -1;
  sp.mine = 0u;
  if (tid < A.B) {
    const RowCfg c = classify(A.params[tid], A.V);
    cfgs[tid] = pack_cfg(c);
    sp.cl = c.type;
  }
  if (w < kOrderWarps) {
#pragma unroll
    for (int t = 0; t < kClasses; ++t) {
      const unsigned b = __ballot_sync(kFull, sp.cl == t);
      if (lane == 0) O.cnt[t][w] = __popc(b);
      if (sp.cl == t) sp.mine = b;
    }
  }
  return sp;
}

// After the barrier: every thread with a row writes it into the order
// ([unfiltered][small top-k][general][top-p][greedy], stable), and thread 0
// also fills in the class totals.
__device__ __forceinline__ void order_place_smem(uint32_t* order, OrderScratch& O, const SmemPlace& sp) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (sp.cl < 0 && tid != 0) return;
  int n[kClasses];
#pragma unroll
  for (int t = 0; t < kClasses; ++t) {
    const uint4 a = *reinterpret_cast<const uint4*>(&O.cnt[t][0]);
    const uint4 b = *reinterpret_cast<const uint4*>(&O.cnt[t][4]);
    n[t] = (int)(a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w);
  }
  if (tid == 0) {
#pragma unroll
    for (int t = 0; t < kClasses; ++t) O.n_class[t] = n[t];
  }
  if (sp.cl < 0) return;
  const int cl = sp.cl;
  int off = cl == UT_DENSE ? 0
          : cl == UT_TOPK ? n[UT_DENSE]
          : cl == UT_GENERAL ? n[UT_DENSE] + n[UT_TOPK]
          : cl == UT_TOPP ? n[UT_DENSE] + n[UT_TOPK] + n[UT_GENERAL]
                          : n[UT_DENSE] + n[UT_TOPK] + n[UT_GENERAL] + n[UT_TOPP];
  for (int ww = 0; ww < w; ++ww) off += (int)O.cnt[cl][ww];
  off += __popc(sp.mine & ((1u << lane) - 1u));
  order[off] = (uint32_t)tid;
}

// Larger batches: CTA 0 writes the order and the class counts into the
// workspace and publishes them with the call's tag; the other CTAs wait for it.
__device__ __noinline__ void build_order_global(const Args& A, OrderScratch& O, uint32_t tag) {
  const int tid = threadIdx.x;
  if (tid < kClasses) {
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
  if (tid < kClasses) A.ws->n_class[tid] = (uint32_t)O.n_class[tid];
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    store_release(&A.ws->order_tag, tag);
  }
}

// ---------------------------------------------------------------------------
// The item sequence.
// ---------------------------------------------------------------------------
struct Plan {
  const uint32_t* order;
  const RowPack* cfg;       // per-row configs in shared memory (null: classify from the parameters)
  const Seg* seg;
  int nseg;
  int nD, nT, nG, nX, nP;   // rows: unfiltered, small top-k, greedy, general, top-p
  int NTA, NTB;             // tiles per unit of this call's dtype
};

// A work item.  kind: 0 none, 1 A tile, 2 B tile.
struct Item {
  int kind;
  uint32_t t;               // index in the sequence
  int reread;               // the logits are read again later (default L2 policy)
  int row, pos, u, c, n;    // unit, tile, valid entries in the tile
  int ntiles;               // tiles of this kind in the unit
};

// Classification from the parameters (batches whose configs are not kept in
// shared memory), out of line: it holds two divisions.
__device__ __noinline__ RowCfg classify_row(const Args& A, int row) { return classify(A.params[row], A.V); }
__device__ __forceinline__ RowCfg plan_cfg(const Args& A, Plan P, int row) {
  return P.cfg ? unpack_cfg(P.cfg[row]) : classify_row(A, row);
}

__device__ __forceinline__ Seg make_seg(uint32_t first, uint32_t nrows, int pos_lo, int upr, int tiles, int kind) {
  Seg s;
  s.start = 0;
  s.first = first;
  s.nrows = nrows;
  s.packed = (uint32_t)tiles | ((uint32_t)pos_lo << 16) | ((uint32_t)upr << 21) | ((uint32_t)kind << 26);
  return s;
}
__device__ __forceinline__ uint32_t seg_items(const Seg& s) {
  return s.nrows * ((s.packed >> 21) & 31u) * (s.packed & 0xffffu);
}

// The segment table (thread 0 of every CTA builds the same one).  The A
// tiles come class by class, the classes with the longest settles first:
// small top-k rows, unfiltered rows in waves (each wave's drafted positions,
// then its bonus positions), greedy rows.  The B tiles of a wave wait in
// a queue until `b_delay` items have been placed after the wave's A tiles
// (the wave's settles finish meanwhile) and are then inserted at the next
// row boundary; waves still waiting at the end come last.
// `rw0` = max(1, b_delay / (items of one row's A tiles)), from the host.
__device__ __forceinline__ void build_segments(const Args& A, VShm& S, int nD, int nT, int nX, int nG, int NTA,
                                               int NTB, uint32_t b_delay, int rw0) {
  const int k = A.k, k1 = A.k + 1;
  Seg* sg = S.seg;
  int n = 0;
  uint32_t pos = 0;     // items placed so far
  uint32_t tasks = 0;   // settle tasks placed so far
  int nw = 0, Rw = 1;
  if (nD > 0) {
    // a wave's A tiles are about b_delay items; waves of equal size
    Rw = max(rw0, ceil_div(nD, kMaxWaves));
    nw = ceil_div(nD, Rw);
    Rw = ceil_div(nD, nw);
    nw = ceil_div(nD, Rw);
  }
  uint32_t* ready = S.bready;   // waves [bh, bt) wait for their B tiles: the item count they wait for
  int bh = 0, bt = 0;
  auto place = [&](Seg sgm) {
    sgm.start = pos;
    pos += seg_items(sgm);
    S.tstart[n] = tasks;
    tasks += sgm.nrows * ((sgm.packed >> 21) & 31u);
    sg[n++] = sgm;
  };
  auto place_b = [&](int w) {
    place(make_seg((uint32_t)(w * Rw), (uint32_t)min(Rw, nD - w * Rw), 0, k, NTB, 1));
  };
  // rows [f, f + nr) of an A class, split where a B wave falls due
  auto place_rows = [&](uint32_t f, uint32_t nr, int pos_lo, int upr) {
    const uint32_t per_row = (uint32_t)upr * (uint32_t)NTA;
    while (nr > 0) {
      while (bh < bt && pos >= ready[bh]) place_b(bh++);
      uint32_t take = nr;
      if (bh < bt) take = min(nr, (ready[bh] - pos + per_row - 1u) / per_row);
      place(make_seg(f, take, pos_lo, upr, NTA, 0));
      f += take;
      nr -= take;
    }
  };
  // small top-k units first: their settles are the longest
  place_rows((uint32_t)nD, (uint32_t)nT, 0, k1);
  for (int i = 0; i < nw; ++i) {
    const uint32_t f = (uint32_t)(i * Rw), nr = (uint32_t)min(Rw, nD - i * Rw);
    if (k > 0) place_rows(f, nr, 0, k);
    place_rows(f, nr, k, 1);
    if (k > 0) ready[bt++] = pos + b_delay;
  }
  place_rows((uint32_t)(nD + nT + nX), (uint32_t)nG, 0, k1);
  while (bh < bt) place_b(bh++);
  S.nseg = n;
  S.ntasks = tasks;
}

// Item t of the sequence.
template <bool kBF16>
__device__ __noinline__ Item map_item(const Args& A, Plan P, uint32_t t) {
  using G = Geo<kBF16>;
  Item it;
  it.kind = 0;
  // the last segment whose start is <= t
  int lo = 0, hi = P.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.seg[mid].start <= t) lo = mid;
    else hi = mid - 1;
  }
  const Seg s = P.seg[lo];
  it.t = t;
  if (P.nseg == 0 || t < s.start || t - s.start >= seg_items(s)) return it;
  const uint32_t tiles = s.packed & 0xffffu, pos_lo = (s.packed >> 16) & 31u, upr = (s.packed >> 21) & 31u;
  const int kind = (int)((s.packed >> 26) & 1u);
  const uint32_t off = t - s.start;
  const uint32_t j = off / tiles;
  // a unit's tiles are taken in a rotated order (by the unit's index), so
  // that CTAs taking items at a fixed stride do not all get the same tile of
  // every unit (the last tile of a unit is the partial one)
  it.c = (int)((off - j * tiles + j) % tiles);
  const uint32_t ri = j / upr;
  it.row = (int)P.order[s.first + ri];
  it.pos = (int)(pos_lo + (j - ri * upr));
  it.u = it.row * (A.k + 1) + it.pos;
  it.kind = kind == 0 ? 1 : 2;
  it.ntiles = (int)tiles;
  // logits of an unfiltered unit are read again: by its B tiles (drafted
  // positions) or by its draw's level-2 race (bonus position)
  it.reread = (kind == 0 && plan_cfg(A, P, it.row).type == UT_DENSE) ? 1 : 0;
  it.n = it.kind == 1 ? min(G::EA, A.V - it.c * G::EA) : min(G::EB, A.V - it.c * G::EB);
  return it;
}

// Lane 0: post the copies of an item into buffer `buf`, completing on `bar`.
template <bool kBF16>
__device__ __forceinline__ void issue(const Args& A, Item it, unsigned char* buf, unsigned long long* bar) {
  using G = Geo<kBF16>;
  if (it.kind == 0) return;
  const unsigned char* lg = reinterpret_cast<const unsigned char*>(A.logits);
  fence_proxy_async();
  // inputs read once are marked evict-first in L2, so they do not push out the
  // records and the logits the B tiles read again
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
    if (++spins > kSpinLimit) {
      if ((threadIdx.x & 31) == 0) atomicOr(&cur(A).error, (uint32_t)ERR_COPY_WAIT);
      return false;
    }
    if (spins > 64) __nanosleep(32);
  }
  return true;
}

// The part of an item the bulk copy did not cover: the ragged tail (read
// with plain loads), and padding up to the end of the tile (-inf logits,
// zero q; 16-byte stores from the first 16-byte boundary), so that every
// tile is reduced over all its blocks.  With rows that are not 16-byte
// aligned, everything.
template <bool kBF16>
__device__ __noinline__ void fill_tail(const Args& A, Item it, unsigned char* buf) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int E = it.kind == 1 ? G::EA : G::EB;
  const int done = A.vec_logits ? (int)(((uint32_t)(it.n * G::es) & ~15u) / G::es) : 0;
  const size_t lrow = (size_t)it.u * A.V + (size_t)it.c * E;
  constexpr int per16 = 16 / G::es;   // entries per 16 bytes
  // entries [done, n), then -inf up to the next 16-byte boundary
  const int vb = min(E, (it.n + per16 - 1) / per16 * per16);
  for (int e = done + lane; e < vb; e += 32) {
    if (kBF16) {
      const uint16_t h = e < it.n ? reinterpret_cast<const uint16_t*>(A.logits)[lrow + e] : (uint16_t)0xff80u;
      reinterpret_cast<uint16_t*>(buf)[e] = h;
    } else {
      reinterpret_cast<float*>(buf)[e] = e < it.n ? reinterpret_cast<const float*>(A.logits)[lrow + e] : -INFINITY;
    }
  }
  const uint32_t ni = kBF16 ? 0xff80ff80u : 0xff800000u;
  const uint4 ninf = make_uint4(ni, ni, ni, ni);
  for (int v = vb / per16 + lane; v < E / per16; v += 32) reinterpret_cast<uint4*>(buf)[v] = ninf;
  if (it.kind == 2) {
    float* qb = reinterpret_cast<float*>(buf + G::EB * G::es);
    const int dq = A.vec_q ? (int)(((uint32_t)(it.n * 4) & ~15u) / 4) : 0;
    const size_t qrow = ((size_t)it.row * A.k + it.pos) * (size_t)A.V + (size_t)it.c * G::EB;
    const int vq = min(E, (it.n + 3) / 4 * 4);
    for (int e = dq + lane; e < vq; e += 32) qb[e] = e < it.n ? A.q[qrow + e] : 0.f;
    for (int v = vq / 4 + lane; v < E / 4; v += 32) reinterpret_cast<uint4*>(qb)[v] = make_uint4(0u, 0u, 0u, 0u);
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
// A tiles.  Lane layout: bf16 lane l reads entries 8l..8l+7 of every block of
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

// Greedy and unfiltered A tile: the tagged record words (lanes 0..7).  The
// lane's entries of every block are held in registers (tiles are padded to
// whole tiles): the max first (NaN-propagating; the first block reaching it
// for the argmax), then the softmax sum relative to it -- at a bonus
// position per block of 256, for the level-1 race.
template <bool kBF16>
__device__ __forceinline__ void a_block(const unsigned char* buf, int b, int lane, uint32_t (&w)[kBF16 ? 4 : 8]) {
  if (kBF16) {
    const uint4 x = *reinterpret_cast<const uint4*>(buf + (b * kRaceBlock + 8 * lane) * 2);
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
  } else {
    const uint4 x = *reinterpret_cast<const uint4*>(buf + (b * kRaceBlock + 4 * lane) * 4);
    const uint4 y = *reinterpret_cast<const uint4*>(buf + (b * kRaceBlock + 128 + 4 * lane) * 4);
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    w[4] = y.x; w[5] = y.y; w[6] = y.z; w[7] = y.w;
  }
}
// Entry j (0..7) of a lane's block words as a float.
template <bool kBF16>
__device__ __forceinline__ float a_val(const uint32_t* w, int j) {
  if (kBF16) return (j & 1) ? bf16_hi(w[j >> 1]) : bf16_lo(w[j >> 1]);
  return __uint_as_float(w[j]);
}
// Max (NaN-propagating) of a lane's block words.
template <bool kBF16>
__device__ __forceinline__ float a_wmax(const uint32_t* w) {
  if (kBF16) {
    const uint32_t t = max_nan_bf16x2(max_nan_bf16x2(w[0], w[1]), max_nan_bf16x2(w[2], w[3]));
    return max_nan(bf16_lo(t), bf16_hi(t));
  }
  return max_nan(max_nan(max_nan(__uint_as_float(w[0]), __uint_as_float(w[1])),
                         max_nan(__uint_as_float(w[2]), __uint_as_float(w[3]))),
                 max_nan(max_nan(__uint_as_float(w[4]), __uint_as_float(w[5])),
                         max_nan(__uint_as_float(w[6]), __uint_as_float(w[7]))));
}
// exp2((v - m) c) of the two bf16 entries of one word, as a packed pair:
// the two floats are built from the word's halves, (v - m) c is one packed
// subtract and one packed multiply (rounded like the scalar form).
__device__ __forceinline__ u64 exp_bf16x2(uint32_t w, u64 m2, u64 c2) {
  u64 r;
  asm("{\n"
      " .reg .b32 lo, hi;\n"
      " .reg .b64 p, d, x;\n"
      " shl.b32 lo, %1, 16;\n"
      " and.b32 hi, %1, 0xffff0000;\n"
      " mov.b64 p, {lo, hi};\n"
      " sub.rn.f32x2 d, p, %2;\n"
      " mul.rn.f32x2 x, d, %3;\n"
      " mov.b64 {lo, hi}, x;\n"
      " ex2.approx.ftz.f32 lo, lo;\n"
      " ex2.approx.ftz.f32 hi, hi;\n"
      " mov.b64 %0, {lo, hi};\n"
      "}"
      : "=l"(r)
      : "r"(w), "l"(m2), "l"(c2));
  return r;
}
// Sum of exp2((v - m) c) over a lane's 8 block entries, as two packed halves.
template <bool kBF16>
__device__ __forceinline__ u64 a_wexp(const uint32_t* w, u64 m2, u64 c2) {
  if (kBF16) {
    const u64 e0 = exp_bf16x2(w[0], m2, c2), e1 = exp_bf16x2(w[1], m2, c2);
    const u64 e2 = exp_bf16x2(w[2], m2, c2), e3 = exp_bf16x2(w[3], m2, c2);
    return add2(add2(e0, e1), add2(e2, e3));
  }
  const u64 e0 = exp_pair(a_val<kBF16>(w, 0), a_val<kBF16>(w, 1), m2, c2);
  const u64 e1 = exp_pair(a_val<kBF16>(w, 2), a_val<kBF16>(w, 3), m2, c2);
  const u64 e2 = exp_pair(a_val<kBF16>(w, 4), a_val<kBF16>(w, 5), m2, c2);
  const u64 e3 = exp_pair(a_val<kBF16>(w, 6), a_val<kBF16>(w, 7), m2, c2);
  return add2(add2(e0, e1), add2(e2, e3));
}
// Max (NaN-propagating) of a lane's entries over all blocks: for bf16 a
// packed running maximum, unpacked once.
template <bool kBF16, int NB, int NW>
__device__ __forceinline__ float a_lane_max(const uint32_t (&w)[NB][NW]) {
  if (kBF16) {
    uint32_t m = 0xff80ff80u;
#pragma unroll
    for (int b = 0; b < NB; ++b)
      m = max_nan_bf16x2(m, max_nan_bf16x2(max_nan_bf16x2(w[b][0], w[b][1]), max_nan_bf16x2(w[b][2], w[b][3])));
    return max_nan(bf16_lo(m), bf16_hi(m));
  }
  float m = -INFINITY;
#pragma unroll
  for (int b = 0; b < NB; ++b) m = max_nan(m, a_wmax<kBF16>(w[b]));
  return m;
}

template <bool kBF16>
__device__ __noinline__ void a_stats(const Args& A, uint32_t tag, Item it, RowCfg cfg,
                                     const unsigned char* buf) {
  using G = Geo<kBF16>;
  constexpr int NB = G::NBA;
  constexpr int NW = kBF16 ? 4 : 8;
  const int lane = threadIdx.x & 31;
  const int e0 = it.c * G::EA;
  const float c = cfg.c;
  const bool greedy = cfg.type == UT_GREEDY;
  const bool bonus = !greedy && it.pos == A.k;
  uint32_t w[NB][NW];
#pragma unroll
  for (int b = 0; b < NB; ++b) a_block<kBF16>(buf, b, lane, w[b]);
  // the lane max
  const float lm = a_lane_max<kBF16, NB, NW>(w);
  const float mc = warp_max_nan(lm);
  const bool nan = mc != mc;
  float z = 0.f;
  Race r;
  race_init(r);
  if (mc > -INFINITY && mc < INFINITY) {
    const u64 m2 = pack2(mc, mc), c2 = pack2(c, c);
    if (!bonus) {
      // the softmax sum relative to the tile max
      u64 za = pack2(0.f, 0.f), zb = pack2(0.f, 0.f);
#pragma unroll
      for (int b = 0; b < NB; b += 2) {
        za = add2(za, a_wexp<kBF16>(w[b], m2, c2));
        if (b + 1 < NB) zb = add2(zb, a_wexp<kBF16>(w[b + 1], m2, c2));
      }
      float a0, a1, b0, b1;
      unpack2(za, a0, a1);
      unpack2(zb, b0, b1);
      z = warp_sum((a0 + a1) + (b0 + b1));
    } else {
      // block weights by a transposed warp sum, then the level-1 race
      constexpr int NP = NB <= 8 ? 8 : (NB <= 16 ? 16 : 32);
      float ps[NP];
      float tot = 0.f;
#pragma unroll
      for (int b = 0; b < NP; ++b) {
        float s0 = 0.f, s1 = 0.f;
        if (b < NB) unpack2(a_wexp<kBF16>(w[b], m2, c2), s0, s1);
        ps[b] = s0 + s1;
        tot += ps[b];
      }
      z = warp_sum(tot);
      const float myW = warp_transpose_sum<NP>(ps);   // lane b: the weight of block b
      if (lane < NB && myW > 0.f) {
        const uint32_t blk = (uint32_t)(e0 / kRaceBlock + lane);
        race_consider(r, myW, 0.f, blk, block_word(A, it.row, it.pos, blk));
      }
      warp_race_merge(r);
    }
  }
  uint32_t idx = 0xffffffffu;
  if (greedy && !nan) {
    // first index of the tile max: in the first block of a lane holding it
    if (lm == mc) {
      int lb = NB - 1;
#pragma unroll
      for (int b = NB - 1; b >= 0; --b)
        if (a_wmax<kBF16>(w[b]) == lm) lb = b;
      float v[8];
      a_vals<kBF16>(buf, lb, lane, v);
#pragma unroll
      for (int j = 7; j >= 0; --j)
        if (v[j] == lm) idx = (uint32_t)(e0 + a_entry<kBF16>(lb, lane, j));
    }
    idx = __reduce_min_sync(kFull, idx);
    // the settle reads q at the unit's argmax, one of the tiles' argmaxes
    if (lane == 0 && it.pos < A.k && idx < (uint32_t)A.V)
      prefetch_l2(A.q + ((size_t)it.row * A.k + it.pos) * (size_t)A.V + idx);
  }
  u64* rec = A.rec + ((size_t)it.u * A.NTA + it.c) * kRecWords;
  const uint32_t v = lane_word8(lane, nan ? 0x7fc00000u : __float_as_uint(mc), idx, __float_as_uint(z),
                                __float_as_uint(r.s1), __float_as_uint(r.t1), __float_as_uint(r.s2),
                                __float_as_uint(r.t2), r.v1);
  if (lane < (bonus ? 8 : 3)) __stcg(rec + lane, tagw(tag, v));
  __syncwarp();
}

// Stages every finite entry >= t8 of the tile (up to kStage; returns the
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

// Small top-k A tile: the tile's kList largest entries in the total order,
// the smallest of them last when there are kList (key, tile-local index),
// tagged words in lanes 0..15.  Every such entry is at least the 8th largest
// lane maximum t8; a lane keeps up to kLaneCand of its entries >= t8 (blocks
// whose maximum is below t8 are skipped), and a lane holding more makes the
// warp stage every entry >= t8 (beyond kStage the list is marked partial).
constexpr int kLaneCand = 4;
template <bool kBF16>
__device__ __noinline__ void a_list(const Args& A, uint32_t tag, Item it, const unsigned char* buf,
                                    u64* stage) {
  constexpr int NB = Geo<kBF16>::NBA;
  const int lane = threadIdx.x & 31;
  const int nb = NB;   // tiles are padded to whole tiles
  float bm[NB];
  float lm = -INFINITY;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    bm[b] = a_block_max<kBF16>(buf, b, lane);
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
  // word 2j: key of entry j (0 = none); word 2j + 1: its tile-local index
  const int j = lane >> 1;
  uint32_t v = 0;
  if (lane < 2 * kList) {
    const bool has = (uint32_t)j < nn;
    const u64 k = has ? stage[j] : 0ull;
    if ((lane & 1) == 0) v = has ? (uint32_t)(k >> 32) : 0u;
    else v = (has ? key64_idx(k) : kListIdx) | (j == 0 ? flags : 0u);
    __stcg(A.rec + ((size_t)it.u * A.NTA + it.c) * kRecWords + lane, tagw(tag, v));
    // the settle reads q at the listed entries: bring those lines into L2 now
    const uint32_t gi = (uint32_t)(it.c * Geo<kBF16>::EA) + (has ? key64_idx(k) : 0u);
    if ((lane & 1) && has && it.pos < A.k && gi < (uint32_t)A.V)
      prefetch_l2(A.q + ((size_t)it.row * A.k + it.pos) * (size_t)A.V + gi);
  }
  __syncwarp();
}

// The record of a tile whose copy or wait gave up: its unit is settled as
// timed out.
__device__ __noinline__ void timeout_record(const Args& A, uint32_t tag, Item it, bool topk) {
  const int lane = threadIdx.x & 31;
  if (it.kind == 1) {
    u64* rec = A.rec + ((size_t)it.u * A.NTA + it.c) * kRecWords;
    uint32_t v = 0;
    if (topk) v = (lane & 1) ? (kListIdx | (lane == 1 ? kListTimeout : 0u)) : 0u;
    else v = lane == 0 ? kTimeoutNaN : 0u;
    if (lane < kRecWords) __stcg(rec + lane, tagw(tag, v));
  } else {
    u64* rec = A.brec + ((size_t)it.u * A.NTB + it.c) * kBRecWords;
    if (lane < 6) __stcg(rec + lane, tagw(tag, lane == 0 ? kTimeoutNaN : 0u));
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// B tiles.
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ __noinline__ void b_tile(const Args& A, uint32_t tag, Item it, RowCfg cfg, UnitState st,
                                    const unsigned char* buf) {
  using G = Geo<kBF16>;
  constexpr int NB = G::NBB;
  constexpr int NP = NB <= 4 ? 4 : 8;
  const int lane = threadIdx.x & 31;
  const int e0 = it.c * G::EB;
  const bool need_race = !st.accept;
  const float* qb = reinterpret_cast<const float*>(buf + G::EB * G::es);
  const float m = st.m, invZ = st.invZ, c = cfg.c;
  const u64 m2 = pack2(m, m), c2 = pack2(c, c), z2 = pack2(invZ, invZ);
  // the lane's entries of every block (logits and q), in registers
  float v[NB][8], q[NB][8];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    sload<kBF16>(buf, b, lane, v[b]);
    sload_q(qb, b, lane, q[b]);
  }
  float alpha_c, myW = 0.f, myQ = 0.f;
  if (!need_race) {
    // accepted draft: alpha only
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        float p0, p1;
        unpack2(mul2(exp_pair(v[b][j], v[b][j + 1], m2, c2), z2), p0, p1);
        a0 += fminf(p0, q[b][j]);
        a1 += fminf(p1, q[b][j + 1]);
      }
    }
    alpha_c = warp_sum(a0 + a1);
  } else {
    // alpha, and per block the residual weight W = sum max(p - q, 0) and
    // the q under it (the draw margin's weight is W + 2 sum q over w > 0)
    float a8 = 0.f;
    float wsum[NP], qsum[NP];
#pragma unroll
    for (int b = 0; b < NP; ++b) {
      float w8 = 0.f, q8 = 0.f;
      if (b < NB) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          float p0, p1;
          unpack2(mul2(exp_pair(v[b][j], v[b][j + 1], m2, c2), z2), p0, p1);   // padding: -inf -> 0
          a8 += fminf(p0, q[b][j]) + fminf(p1, q[b][j + 1]);
          const float d0 = p0 - q[b][j], d1 = p1 - q[b][j + 1];
          w8 += fmaxf(d0, 0.f) + fmaxf(d1, 0.f);
          q8 += (d0 > 0.f ? q[b][j] : 0.f) + (d1 > 0.f ? q[b][j + 1] : 0.f);
        }
      }
      wsum[b] = w8;
      qsum[b] = q8;
    }
    alpha_c = warp_sum(a8);
    myW = warp_transpose_sum<NP>(wsum);
    myQ = warp_transpose_sum<NP>(qsum);
  }
  Race r;
  race_init(r);
  if (need_race && lane < NB && myW > 0.f) {
    const uint32_t blk = (uint32_t)(e0 / kRaceBlock + lane);
    race_consider(r, myW, 2.0f * myQ, blk, block_word(A, it.row, it.pos, blk));
  }
  if (need_race) warp_race_merge(r);   // accepted: the empty race as it is
  u64* rec = A.brec + ((size_t)it.u * A.NTB + it.c) * kBRecWords;
  const uint32_t wv = lane_word8(lane, __float_as_uint(alpha_c), __float_as_uint(r.s1), __float_as_uint(r.t1),
                                 __float_as_uint(r.s2), __float_as_uint(r.t2), r.v1, 0u, 0u);
  if (lane < 6) __stcg(rec + lane, tagw(tag, wv));
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

// A stream warp: items of the sequence, the first two by its index, later
// ones from one counter (the next ticket is in flight while a tile is
// reduced).  After a tile's record, one is added to the unit's tile count.
template <bool kBF16>
__device__ __noinline__ void stream_loop(const Args& A, Plan P0, VShm& S, uint32_t tag, int sw, uint32_t srank,
                                         uint32_t n_stream) {
  const int lane = threadIdx.x & 31;
  const Plan P = P0;
  Bufs B;
  B.a = S.s.buf[sw][0];
  B.b = S.s.buf[sw][1];
  B.ba = &S.bar[sw][0];
  B.bb = &S.bar[sw][1];
  B.pa = 0u;
  B.pb = 0u;
  if (lane == 0) {
    mbar_init(B.ba, 1);    // issue() orders the inits before the copies (fence.proxy.async)
    mbar_init(B.bb, 1);
  }
  __syncwarp();
  const uint32_t gs = (uint32_t)sw * n_stream + srank;   // the warp's index over the stream warps
  Item ia = map_item<kBF16>(A, P, srank + n_stream * (uint32_t)sw);
  Item ib = map_item<kBF16>(A, P, srank + n_stream * (uint32_t)(kNW + sw));
  // the first buffer alone: the first data arrives behind half the bytes a
  // second copy per warp would put in flight; the second copy is posted as
  // soon as it has (below)
  if (lane == 0) issue<kBF16>(A, ia, B.a, B.ba);
  bool broken = false;
  bool first = true;
  while (ia.kind != 0) {
    uint32_t tn = 0;
    const bool take = ib.kind != 0 && !broken;   // warp-uniform
    if (lane == 0 && take) tn = srank + n_stream * (2u * kNW + atomicAdd(&S.ticket, 1u));
    const RowCfg cfg = plan_cfg(A, P, ia.row);
    u64 sw8[kStateWords];
    if (ia.kind == 2) state_load(A, ia.u, sw8);     // in flight during the copy wait
    const bool ok = !broken && wait_buffer(A, B.ba, B.pa);
    if (first) {
      if (lane == 0 && ok) TL(TL_FIRST_DATA, (int)gs, 2048);
      if (lane == 0 && ok) issue<kBF16>(A, ib, B.b, B.bb);
      first = false;
    }
#ifdef SPEC_TIMELINE
    if (lane == 0 && ia.t < 16384u) {
      TL(TL_ISTART, (int)ia.t, 16384);
      g_tl[TL_IWARP + ia.t] = gs + 1u + (ia.kind == 2 ? 0x10000u : 0u);
    }
#endif
    if (!ok) {
      // the buffer's copy never completed: mark this tile and stop taking new ones
      broken = true;
      timeout_record(A, tag, ia, cfg.type == UT_TOPK);
    } else {
      B.pa ^= 1u;
      if (!A.vec_logits || (ia.kind == 2 && !A.vec_q) || ia.n != (ia.kind == 1 ? Geo<kBF16>::EA : Geo<kBF16>::EB))
        fill_tail<kBF16>(A, ia, B.a);
      if (ia.kind == 1) {
        if (cfg.type == UT_TOPK) a_list<kBF16>(A, tag, ia, B.a, S.s.stage[sw]);
        else a_stats<kBF16>(A, tag, ia, cfg, B.a);
      } else {
        // the unit state (bounded wait: a settle warp publishes it)
        long long spins = 0;
        bool st_ok = true;
        while (!__all_sync(kFull, state_ok(sw8, tag))) {
          if (++spins > kSpinLimit) {
            if (lane == 0) atomicOr(&cur(A).error, (uint32_t)ERR_STATE_WAIT);
            st_ok = false;
            break;
          }
          __nanosleep(128);
          state_load(A, ia.u, sw8);
        }
        if (lane == 0 && ia.t < 16384u) TL(TL_ISTATE, (int)ia.t, 16384);
        if (!st_ok) {
          timeout_record(A, tag, ia, false);
        } else {
          const UnitState st = state_of(sw8);
          if (!st.invalid) b_tile<kBF16>(A, tag, ia, cfg, st, B.a);
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      TL(TL_ITEM, (int)ia.t, 16384);
      atomicAdd(&A.ucnt[(ia.kind == 2 ? A.U : 0) + ia.u], 1u);   // result unused: a reduction
    }
    tn = __shfl_sync(kFull, tn, 0);
    Item in;
    in.kind = 0;
    if (take) in = map_item<kBF16>(A, P, tn);   // after a failed copy: mapped, marked, not copied
    if (lane == 0 && !broken) issue<kBF16>(A, in, B.a, B.ba);
    ia = ib;
    ib = in;
    B.rotate();
  }
  if (lane == 0) {
    TL(TL_STREAM_END, (int)gs, 2048);
    S.broken[sw] = broken ? 1u : 0u;
  }
  __syncwarp();
}

// Settle task t: the unit and kind (settle-A after its A tiles, settle-B
// after its B tiles) and the tile count to wait for.
struct Task {
  int u, row, pos, ntiles, kind;   // kind 1: A, 2: B
};
__device__ __forceinline__ Task map_task(const Args& A, Plan P, const VShm& S, uint32_t t) {
  int lo = 0, hi = P.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.tstart[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const Seg s = P.seg[lo];
  const uint32_t upr = (s.packed >> 21) & 31u, pos_lo = (s.packed >> 16) & 31u;
  const uint32_t j = t - S.tstart[lo];
  const uint32_t ri = j / upr;
  Task k;
  k.row = (int)P.order[s.first + ri];
  k.pos = (int)(pos_lo + (j - ri * upr));
  k.u = k.row * (A.k + 1) + k.pos;
  k.ntiles = (int)(s.packed & 0xffffu);
  k.kind = ((s.packed >> 26) & 1u) ? 2 : 1;
  return k;
}

// A settle warp: tasks g, g + nst, ... in sequence order; each waits for its
// unit's tile count, settles the unit and clears the count.
template <bool kBF16>
__device__ __noinline__ void settle_loop(const Args& A, Plan P, VShm& S, uint32_t tag, int w, uint32_t g,
                                         uint32_t nst) {
  const int lane = threadIdx.x & 31;
  TopkScratch& TS = S.tk[w];
  for (uint32_t t = g; t < S.ntasks; t += nst) {
    const Task k = map_task(A, P, S, t);
    uint32_t* cnt = &A.ucnt[(k.kind == 2 ? A.U : 0) + k.u];
    // what the settle needs besides the records is loaded while the tiles
    // are still being reduced: the draft and its logit and q (settle-A), or
    // the unit's published state (settle-B)
    Pre pr;
    StateWords sw8;
    if (k.kind == 2) {
      state_load(A, k.u, sw8.w);
    } else {
      pr = load_pre<kBF16>(A, k.u, k.row, k.pos);
    }
    bool ready = true;
    if (lane == 0) {
      long long spins = 0;
      while (load_relaxed(cnt) != (uint32_t)k.ntiles) {
        if (++spins > 16ll * kSpinLimit) {
          atomicOr(&cur(A).error, (uint32_t)ERR_RECORD_WAIT);
          ready = false;
          break;
        }
        __nanosleep(spins > 64 ? 128 : 32);
      }
    }
    ready = __shfl_sync(kFull, ready ? 1 : 0, 0) != 0;
    const RowCfg cfg = plan_cfg(A, P, k.row);
    // the warp's last task: no settle follows it on this warp, and the SMs
    // are emptying, so its draw takes the inline race (lower latency alone)
    const bool late = t + nst >= S.ntasks;
    if (lane == 0) TL(k.kind == 2 ? TL_SB_START : TL_SA_START, k.u, 2048);
    if (!ready) {
      commit_record(A, tag, k.u, k.row, empty_record(SPEC_F_TIMEOUT));   // the records' polls would give up too
    } else if (k.kind == 2) {
      fin_b<kBF16>(A, tag, k.u, k.row, k.pos, cfg, sw8, late);
    } else if (cfg.type == UT_TOPK) {
      topk_settle<kBF16>(A, tag, TS, k.u, k.row, k.pos, cfg, pr);
    } else {
      fin_stats<kBF16>(A, tag, k.u, k.row, k.pos, cfg, pr, late);
    }
    if (lane == 0) {
      TL(k.kind == 2 ? TL_SB_END : TL_SA_END, k.u, 2048);
      *cnt = 0u;   // leave the workspace clean for the next call
    }
    __syncwarp();
  }
  if (lane == 0) TL(TL_SETTLE_END, (int)g, 256);
}

// General-path units, taken by the CTA's first kThreads threads.
template <bool kBF16>
__device__ __noinline__ void general_phase(const Args& A, Plan P, VShm& S, uint32_t tag) {
  const int k1 = A.k + 1;
  const int nGU = P.nX * k1;
  const int gbase = P.nD + P.nT;
  GenRing R;
  R.buf = &S.g.ring[0][0];
  R.bar = S.g.bar;
  R.fail = &S.g.gen.ring_fail;
  R.seq = 0u;
  R.ok = true;
  if (ctid() == 0) {
    for (int i = 0; i < kGRing; ++i) mbar_init(&R.bar[i], 1);   // the first copy's fence orders the inits
    S.g.gen.ring_fail = 0;
  }
  csync();
  while (true) {
    if (ctid() == 0) S.gtask = (int)atomicAdd(&cur(A).gnext, 1u);
    csync();
    const int g = S.gtask;
    csync();
    if (g >= nGU) break;
    const int row = (int)P.order[gbase + g / k1], pos = g % k1;
    if (ctid() == 0) TL(TL_SA_START, row * k1 + pos, 2048);
    unit_general<kBF16>(A, S.g.gen, R, tag, row * k1 + pos, row, pos, plan_cfg(A, P, row));
    if (ctid() == 0) TL(TL_SA_END, row * k1 + pos, 2048);
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kAllThreads, 1) verify_kernel(const __grid_constant__ Args A, uint32_t b_delay,
                                                                int rw0) {
  using G = Geo<kBF16>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  VShm& S = *reinterpret_cast<VShm*>(smem_raw);
  const int w = threadIdx.x >> 5;
  if (threadIdx.x == kAllThreads - 64 && A.l2_stage) {
    // Rows with top-p alone are read by every top-p pass, the first of which
    // starts only after the roles and a grid barrier: their logits go into
    // L2 now, in bulk prefetches of 64 KB, while the prologue and the roles
    // run.  A CTA classifies one row (a few when rows outnumber CTAs), so
    // the prologue does not wait on this thread; with more CTAs than rows, a
    // row's pieces are split over gridDim.x / B CTAs.
    const size_t row_bytes = (size_t)(A.k + 1) * (size_t)A.V * (size_t)G::es;
    const unsigned char* lg = reinterpret_cast<const unsigned char*>(A.logits);
    const int grid = (int)gridDim.x, cta = (int)blockIdx.x;
    const int per = grid >= A.B ? grid / A.B : 1;   // CTAs per row
    const int r0 = grid >= A.B ? (cta < per * A.B ? cta % A.B : A.B) : cta;
    const int rstep = grid >= A.B ? A.B : grid;
    const size_t o0 = grid >= A.B ? (size_t)(cta / A.B) * 65536 : 0;
    for (int r = r0; r < A.B; r += rstep) {
      if (classify(A.params[r], A.V).type != UT_TOPP) continue;
      for (size_t o = o0; o < row_bytes; o += (size_t)per * 65536) {
        const uint32_t n = (uint32_t)min((size_t)65536, row_bytes - o) & ~15u;
        if (n) bulk_prefetch_l2(lg + (size_t)r * row_bytes + o, n);
      }
    }
  }
  if (threadIdx.x == kAllThreads - 32) {
    // The call's number: the CTAs that entered earlier calls over the grid
    // size (calls on one workspace never overlap, and each launches the
    // same grid).  Its tag is that number plus one, wrapping past 0.
    const unsigned long long call = atomicAdd(&A.ws->arrivals, 1ull) / (unsigned long long)A.n_ctas;
    const uint32_t tag = (uint32_t)(call % 0xFFFFFFFFull) + 1u;
    const uint32_t par = (uint32_t)(call & 1ull);
    S.tag = tag;
    s_call_parity = par;
    if (blockIdx.x == 0) {
      // the next call's counters start at zero (the call before this one
      // used them, and it has ended)
      A.ws->epoch = tag;
      A.ws->last_set = par;
      uint4* nx = reinterpret_cast<uint4*>(&A.ws->call[par ^ 1u]);
      nx[0] = make_uint4(0u, 0u, 0u, 0u);
      nx[1] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (threadIdx.x == 0) {
    S.gtask = 0;
    S.ticket = 0u;
  }
  if ((threadIdx.x & 31) == 0) S.broken[threadIdx.x >> 5] = 0u;
  Plan P;
  bool order_ok = true;
  if (!A.global_order) {
    const SmemPlace sp = order_classify_smem(A, S.cfg, S.ord);
    __syncthreads();
    order_place_smem(S.order, S.ord, sp);
    if (threadIdx.x == 0)
      build_segments(A, S, S.ord.n_class[UT_DENSE], S.ord.n_class[UT_TOPK],
                     S.ord.n_class[UT_GENERAL] + S.ord.n_class[UT_TOPP], S.ord.n_class[UT_GREEDY],
                     ceil_div(A.V, G::EA), ceil_div(A.V, G::EB), b_delay, rw0);
    __syncthreads();
    P.order = S.order;
    P.cfg = S.cfg;
    P.nD = S.ord.n_class[UT_DENSE];
    P.nT = S.ord.n_class[UT_TOPK];
    P.nG = S.ord.n_class[UT_GREEDY];
    P.nX = S.ord.n_class[UT_GENERAL];
    P.nP = S.ord.n_class[UT_TOPP];
  } else {
    __syncthreads();
    if (blockIdx.x == 0) build_order_global(A, S.ord, S.tag);
    if (threadIdx.x == 0) {
      long long spins = 0;
      while (load_acquire(&A.ws->order_tag) != S.tag) {
        if (++spins > kSpinLimit) {
          atomicOr(&cur(A).error, (uint32_t)ERR_ORDER_WAIT);
          S.gtask = -1;
          break;
        }
        __nanosleep(128);
      }
    }
    __syncthreads();
    order_ok = S.gtask != -1;
    P.order = A.order;
    P.cfg = nullptr;
    P.nD = (int)__ldcg(&A.ws->n_class[UT_DENSE]);
    P.nT = (int)__ldcg(&A.ws->n_class[UT_TOPK]);
    P.nG = (int)__ldcg(&A.ws->n_class[UT_GREEDY]);
    P.nX = (int)__ldcg(&A.ws->n_class[UT_GENERAL]);
    P.nP = (int)__ldcg(&A.ws->n_class[UT_TOPP]);
    // (general and top-p rows have no stream tiles; greedy rows follow them)
    if (threadIdx.x == 0)
      build_segments(A, S, P.nD, P.nT, P.nX + P.nP, P.nG, ceil_div(A.V, G::EA), ceil_div(A.V, G::EB), b_delay, rw0);
    __syncthreads();
  }
  const uint32_t tag = S.tag;
  P.NTA = ceil_div(A.V, G::EA);
  P.NTB = ceil_div(A.V, G::EB);
  if (P.nP > 0 && order_ok) {
    // the top-p passes' scratch, zero before their first barrier
    const size_t n16 = (size_t)P.nP * (size_t)(A.k + 1) * (kTpStride / 2);
    uint4* z = reinterpret_cast<uint4*>(A.tp);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
      z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  P.seg = S.seg;
  P.nseg = S.nseg;
  if (threadIdx.x == 0) TL(TL_CTA_START, (int)blockIdx.x, 160);
  if (order_ok) {
    const int bx = (int)blockIdx.x;
    const bool settle_cta = (bx % A.settle_stride) == 0 && bx / A.settle_stride < A.n_settle;
    if (settle_cta) {
      const uint32_t nst = (uint32_t)A.n_settle * kNW;
      // task t to settle CTA t mod n_settle: consecutive tasks (one class,
      // neighbouring rows) go to different SMs
      settle_loop<kBF16>(A, P, S, tag, w, (uint32_t)w * (uint32_t)A.n_settle + (uint32_t)(bx / A.settle_stride), nst);
    } else {
      // stream CTA rank: blocks before this one, minus the settle CTAs among them
      const int srank = bx - min(A.n_settle, bx / A.settle_stride + 1);
      const int n_stream = A.n_ctas - A.n_settle;
      // item t belongs to stream CTA t mod n_stream (consecutive items on different SMs)
      stream_loop<kBF16>(A, P, S, tag, w, (uint32_t)srank, (uint32_t)n_stream);
    }
  }
  if (P.nP > 0 && order_ok) {
    // top-p rows: grid-wide passes (every thread of every CTA)
    __syncthreads();
    TpPlan T;
    T.order = P.order;
    T.cfg = P.cfg;
    T.base = P.nD + P.nT + P.nX;
    T.nU = P.nP * (A.k + 1);
    T.nlev = 0;
    topp_passes<kBF16>(A, T, tag, S.s.buf[w][0], S.broken[w] == 0u);
  }
  if (P.nX > 0 && order_ok) {
    __syncthreads();
    if (threadIdx.x < kThreads) general_phase<kBF16>(A, P, S, tag);
  }
  __syncthreads();
  if (A.fc.on && order_ok) {
    // the fused commit: every warp copies rows as they are finalized (not
    // after a copy wait that gave up: that copy may still land in a buffer)
    const bool copy_failed = (__shfl_sync(kFull, __ldcg(&cur(A).error), 0) & (uint32_t)ERR_COPY_WAIT) != 0u ||
                             S.broken[w] != 0u;
    if (!copy_failed) commit_phase(A, tag, S.s.buf[w][0], S.s.buf[w][1], S.cbar[w]);
    __syncthreads();
  }
  if (threadIdx.x == 0) TL(TL_CTA_END, (int)blockIdx.x, 160);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
// Items of A tiles between the end of an unfiltered wave's A tiles and its
// B tiles: the wave's settles (a few microseconds) finish meanwhile.
constexpr uint32_t kBDelayItems = 2800;

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
      cached[dev] = sms;   // one CTA per SM
    }
    n = cached[dev];
  }
  Args A = A0;
  A.n_ctas = n;
  A.n_settle = n >= 2 * kSettleEvery ? n / kSettleEvery : 1;
  A.settle_stride = n / A.n_settle;
  A.global_order = A.B > kOrderSmem ? 1 : 0;
  uint32_t b_delay = kBDelayItems;
  // rows of unfiltered units per wave, before the bound on the wave count
  const uint32_t row_items = (uint32_t)(A.k + 1) * (uint32_t)ceil_div(A.V, Geo<kBF16>::EA);
  const int rw0 = (int)std::max(1u, b_delay / std::max(1u, row_items));
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
  if (cudaLaunchKernelEx(&cfg, kern, A, b_delay, rw0) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  return SPEC_OK;
}

template int launch_verify<true>(const Args&, cudaStream_t);
template int launch_verify<false>(const Args&, cudaStream_t);

}  // namespace specv

#ifdef SPEC_TIMELINE
// Instrumented builds only: copy the timeline stamps to `out` (host,
// TL_SIZE words) after a synchronize, and clear them.
extern "C" int spec_timeline_read(unsigned long long* out) {
  if (cudaDeviceSynchronize() != cudaSuccess) return SPEC_E_CUDA;
  if (cudaMemcpyFromSymbol(out, specv::g_tl, sizeof(unsigned long long) * specv::TL_SIZE) != cudaSuccess)
    return SPEC_E_CUDA;
  static unsigned long long zero[specv::TL_SIZE];
  if (cudaMemcpyToSymbol(specv::g_tl, zero, sizeof(zero)) != cudaSuccess) return SPEC_E_CUDA;
  return SPEC_OK;
}
#endif
