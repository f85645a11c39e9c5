// spec_verify: the verify kernel (sm_103a).
//
// One persistent CTA of 12 warps per SM, launched cooperatively (every CTA
// is resident, so CTAs may wait on one another; every such wait is
// bounded).  The work runs in passes separated by grid barriers, so that
// each pass runs one kind of code on every SM and the latency-bound settles
// never queue behind the stream's copies:
//   1. A pass.  Every warp owns two 8 KB shared-memory buffers and has the
//      copy engine fill one (cp.async.bulk completed on an mbarrier) while
//      it reduces the other; the A tiles of all units (4096 bf16 / 2048
//      fp32 logits) are taken from one counter, class by class (small
//      top-k, greedy, unfiltered rows last, so that their logits are still
//      in L2 for the B pass).  A tile yields its max, the softmax sum
//      relative to it, the first argmax (greedy), the level-1 race of its
//      256-entry blocks (bonus positions) or its 8 largest entries in the
//      total order (small top-k), as tagged record words.
//   2. Settles.  One warp per unit (spec_settle.cuh): greedy and small
//      top-k units and bonus positions are settled; a drafted unfiltered
//      unit takes its accept test and publishes its state.  Warps without a
//      unit bring the q rows of the B pass into L2 meanwhile.
//   3. B pass (drafted positions of unfiltered rows only).  A B tile (1280
//      bf16 / 1024 fp32 logits, read again from L2, plus q) computes alpha =
//      sum min(p, q) and the level-1 race of the residual from the state.
//   4. Their settles: alpha and the residual draw.
// The last settled unit of a row resolves its accept chain and writes the
// row's outputs.  Rows that need a global threshold search
// (spec_general.cuh) are taken last by the CTAs' first 256 threads, and the
// fused commit (spec_fused.cuh) follows.  Results pass between warps as
// 64-bit words tagged with the call's epoch; reductions have a fixed order
// and no floating-point atomics are used, so results are bit-reproducible.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "spec_common.cuh"
#include "spec_fused.cuh"
#include "spec_general.cuh"
#include "spec_host.h"
#include "spec_settle.cuh"

namespace specv {

constexpr int kNW = kCtaWarps;         // warps per CTA
constexpr int kAllThreads = kNW * 32;
constexpr int kOrderSmem = 256;        // batches up to this many rows keep order and configs in shared memory
constexpr int kStage = 64;             // per-warp staging of a top-k tile's candidates
constexpr unsigned kFull = 0xffffffffu;
static_assert(kAllThreads >= kOrderSmem, "one placement round for a shared-memory order");
static_assert(kAllThreads >= kThreads, "the general phase uses the first kThreads threads");

struct OrderScratch {
  int n_class[4];
  int run[4];
  int scan[kNW][4];
};

struct alignas(128) VShm {
  union {
    struct {
      unsigned char buf[kNW][2][kSlot];  // stream buffers
      u64 stage[kNW][kStage];            // top-k tile staging
    } s;
    TopkCtaShm tkc;                      // settle scratch of a small top-k unit
    GenShm gen;                          // general-path group, after the roles
  };
  unsigned long long bar[kNW][2];        // the warps' stream-buffer barriers
  uint32_t par[kNW][2];                  // their phase parities (carried from the A pass to the B pass)
  uint32_t broken[kNW];                  // a copy wait of the warp gave up: its buffers are not used again
  uint32_t ticket[2];                    // the CTA's item counters of the A and B passes
  unsigned long long cbar[kNW][2];       // fused commit: the warps' copy barriers
  uint32_t order[kOrderSmem];
  RowPack cfg[kOrderSmem];
  OrderScratch ord;
  int gtask;
  uint32_t tag;
};

static_assert(sizeof(VShm) <= 232448, "shared memory of a CTA exceeds 227 KB");

// ---------------------------------------------------------------------------
// Row order: rows of each class, stably, as [unfiltered][small top-k]
// [general][greedy].
// ---------------------------------------------------------------------------
__device__ __forceinline__ int class_rank(int cl) {
  return cl == UT_DENSE ? 0 : (cl == UT_TOPK ? 1 : (cl == UT_GENERAL ? 2 : 3));
}
__device__ __forceinline__ int class_base(const OrderScratch& O, int cl) {
  const int nD = O.n_class[UT_DENSE], nT = O.n_class[UT_TOPK], nX = O.n_class[UT_GENERAL];
  const int r = class_rank(cl);
  return r == 0 ? 0 : (r == 1 ? nD : (r == 2 ? nD + nT : nD + nT + nX));
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
    for (int ww = 0; ww < kNW; ++ww) s += O.scan[ww][tid];
    O.run[tid] += s;
  }
  __syncthreads();
}

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
// Work of the phases.  Units are taken class by class: small top-k rows,
// greedy rows, then unfiltered rows (whose logits the B pass reads again, so
// they are the last to enter L2); each row contributes its k + 1 positions.
// ---------------------------------------------------------------------------
struct Plan {
  const uint32_t* order;    // rows by class: [unfiltered][small top-k][general][greedy]
  const RowPack* cfg;       // per-row configs in shared memory (null: classify from the parameters)
  int nD, nT, nG, nX;       // rows: unfiltered, small top-k, greedy, general
  int NTA, NTB;             // tiles per unit of this call's dtype
};

// A work item.  kind: 0 none, 1 A tile, 2 B tile.
struct Item {
  int kind;
  uint32_t t;               // index in its pass
  int reread;               // the logits are read again later (default L2 policy)
  int row, pos, u, c, n;    // unit, tile, valid entries in the tile
};

// Classification from the parameters (batches whose configs are not kept in
// shared memory), out of line: it holds two divisions.
__device__ __noinline__ RowCfg classify_row(const Args& A, int row) { return classify(A.params[row], A.V); }
__device__ __forceinline__ RowCfg plan_cfg(const Args& A, Plan P, int row) {
  return P.cfg ? unpack_cfg(P.cfg[row]) : classify_row(A, row);
}

// Row ri of the A pass order: small top-k, greedy, unfiltered.
__device__ __forceinline__ int a_row(const Plan& P, int ri) {
  if (ri < P.nT) return (int)P.order[P.nD + ri];
  ri -= P.nT;
  if (ri < P.nG) return (int)P.order[P.nD + P.nT + P.nX + ri];
  return (int)P.order[ri - P.nG];
}
__device__ __forceinline__ int a_units(const Args& A, const Plan& P) { return (P.nT + P.nG + P.nD) * (A.k + 1); }
__device__ __forceinline__ int b_units(const Args& A, const Plan& P) { return P.nD * A.k; }

// Item t of a pass: A tiles (pass 1) of every unit in the A pass order, or
// B tiles (pass 2) of the drafted positions of unfiltered rows.
template <bool kBF16>
__device__ __forceinline__ Item map_item(const Args& A, const Plan& P, int pass, uint32_t t, uint32_t n_items) {
  using G = Geo<kBF16>;
  Item it;
  it.kind = 0;
  it.t = t;
  if (t >= n_items) return it;
  // a unit's tiles are taken in a rotated order (by the unit's index), so
  // that the CTAs taking items at a fixed stride do not all get the same
  // tile of every unit (the last tile of a unit is the partial one)
  if (pass == 1) {
    const uint32_t j = t / (uint32_t)P.NTA;
    it.c = (int)((t - j * (uint32_t)P.NTA + j) % (uint32_t)P.NTA);
    const uint32_t ri = j / (uint32_t)(A.k + 1);
    it.pos = (int)(j - ri * (uint32_t)(A.k + 1));
    it.row = a_row(P, (int)ri);
    it.kind = 1;
    it.reread = (int)ri >= P.nT + P.nG ? 1 : 0;   // unfiltered: the B tiles or the bonus draw read it again
    it.n = min(G::EA, A.V - it.c * G::EA);
  } else {
    const uint32_t j = t / (uint32_t)P.NTB;
    it.c = (int)((t - j * (uint32_t)P.NTB + j) % (uint32_t)P.NTB);
    const uint32_t ri = j / (uint32_t)A.k;
    it.pos = (int)(j - ri * (uint32_t)A.k);
    it.row = (int)P.order[ri];
    it.kind = 2;
    it.reread = 0;
    it.n = min(G::EB, A.V - it.c * G::EB);
  }
  it.u = it.row * (A.k + 1) + it.pos;
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
      if ((threadIdx.x & 31) == 0) atomicOr(&A.ws->error, (uint32_t)ERR_COPY_WAIT);
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

// A stream warp in one pass (1: A tiles, 2: B tiles).  Item t of the pass
// belongs to CTA t mod n_ctas; a CTA's warps take its items j = 0, 1, ...
// (item blockIdx + n_ctas j): the first two by the warp's index, later ones
// from a shared-memory counter (no global counter for all SMs to contend
// on).  Of the warp's two buffers one is filled by the copy engine while the
// other is reduced; the barriers' parities carry over from pass to pass.
template <bool kBF16>
__device__ __noinline__ void stream_pass(const Args& A, Plan P0, VShm& S, uint32_t tag, int w, uint32_t gw,
                                         int pass, uint32_t n_items, uint32_t* ticket) {
  const int lane = threadIdx.x & 31;
  const Plan P = P0;
  unsigned char* bufa = S.s.buf[w][0];
  unsigned char* bufb = S.s.buf[w][1];
  unsigned long long* bara = &S.bar[w][0];
  unsigned long long* barb = &S.bar[w][1];
  uint32_t pa = S.par[w][0], pb = S.par[w][1];
  bool swapped = false;
  bool broken = S.broken[w] != 0u;
  const uint32_t nc = (uint32_t)A.n_ctas, cb = blockIdx.x;
  Item ia = map_item<kBF16>(A, P, pass, cb + nc * (uint32_t)w, n_items);
  Item ib = map_item<kBF16>(A, P, pass, cb + nc * (uint32_t)(kNW + w), n_items);
  // the first buffer alone: the first data arrives behind half the bytes a
  // second copy per warp would put in flight; the second copy is posted as
  // soon as it has (below)
  if (lane == 0 && !broken) issue<kBF16>(A, ia, bufa, bara);
  bool first = true;
  while (ia.kind != 0) {
    uint32_t tn = 0;
    const bool take = ib.kind != 0 && !broken;   // warp-uniform
    if (lane == 0 && take) tn = cb + nc * (2u * kNW + atomicAdd(ticket, 1u));
    const RowCfg cfg = plan_cfg(A, P, ia.row);
    u64 sw8[kStateWords];
    if (ia.kind == 2) state_load(A, ia.u, sw8);     // in flight during the copy wait
    const bool ok = !broken && wait_buffer(A, bara, pa);
    if (first) {
      if (lane == 0 && ok && pass == 1) TL(TL_FIRST_DATA, (int)gw, 2048);
      if (lane == 0 && ok) issue<kBF16>(A, ib, bufb, barb);
      first = false;
    }
#ifdef SPEC_TIMELINE
    if (lane == 0 && pass == 1) {
      TL(TL_ISTART, (int)ia.t, 16384);
      if (ia.t < 16384u) g_tl[TL_IWARP + ia.t] = gw + 1u;
    }
#endif
    if (!ok) {
      // the buffer's copy never completed: mark this tile and stop taking new ones
      broken = true;
      timeout_record(A, tag, ia, cfg.type == UT_TOPK);
    } else {
      pa ^= 1u;
      if (!A.vec_logits || (ia.kind == 2 && !A.vec_q) || ia.n != (ia.kind == 1 ? Geo<kBF16>::EA : Geo<kBF16>::EB))
        fill_tail<kBF16>(A, ia, bufa);
      if (ia.kind == 1) {
        if (cfg.type == UT_TOPK) a_list<kBF16>(A, tag, ia, bufa, S.s.stage[w]);
        else a_stats<kBF16>(A, tag, ia, cfg, bufa);
      } else {
        // the unit state, published before this pass (bounded wait all the same)
        long long spins = 0;
        bool st_ok = true;
        while (!__all_sync(kFull, state_ok(sw8, tag))) {
          if (++spins > kSpinLimit) {
            if (lane == 0) atomicOr(&A.ws->error, (uint32_t)ERR_STATE_WAIT);
            st_ok = false;
            break;
          }
          __nanosleep(128);
          state_load(A, ia.u, sw8);
        }
        if (!st_ok) {
          timeout_record(A, tag, ia, false);
        } else {
          const UnitState st = state_of(sw8);
          if (!st.invalid) b_tile<kBF16>(A, tag, ia, cfg, st, bufa);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && pass == 1) TL(TL_ITEM, (int)ia.t, 16384);
    tn = __shfl_sync(kFull, tn, 0);
    Item in;
    in.kind = 0;
    if (take) in = map_item<kBF16>(A, P, pass, tn, n_items);   // after a failed copy: mapped, marked, not copied
    if (lane == 0 && !broken) issue<kBF16>(A, in, bufa, bara);
    ia = ib;
    ib = in;
    unsigned char* tb = bufa;
    bufa = bufb;
    bufb = tb;
    unsigned long long* tr = bara;
    bara = barb;
    barb = tr;
    const uint32_t tp = pa;
    pa = pb;
    pb = tp;
    swapped = !swapped;
  }
  if (lane == 0) {
    S.par[w][0] = swapped ? pb : pa;
    S.par[w][1] = swapped ? pa : pb;
    S.broken[w] = broken ? 1u : 0u;
    if (pass == 1) TL(TL_STREAM_END, (int)gw, 2048);
  }
  __syncwarp();
}

// The settle pass after the A pass: small top-k units by whole CTAs (unit
// i by CTA i mod n_ctas), the other units by single warps from a counter.
template <bool kBF16>
__device__ __noinline__ void settle_pass_a(const Args& A, Plan P, VShm& S, uint32_t tag) {
  const int lane = threadIdx.x & 31;
  const int k1 = A.k + 1;
  const int nTU = P.nT * k1;
  for (int i = (int)blockIdx.x; i < nTU; i += A.n_ctas) {
    __syncthreads();   // warp 0 has finished the CTA's previous unit
    const int ri = i / k1, pos = i - (i / k1) * k1;
    const int row = a_row(P, ri);
    const int u = row * k1 + pos;
    const RowCfg cfg = plan_cfg(A, P, row);
    if (threadIdx.x == 0) TL(TL_SA_START, u, 2048);
    topk_settle_cta<kBF16>(A, tag, S.tkc, u, row, pos, cfg);
    if (threadIdx.x == 0) TL(TL_SA_END, u, 2048);
  }
  const uint32_t nu = (uint32_t)a_units(A, P);
  while (true) {
    uint32_t j = 0;
    if (lane == 0) j = atomicAdd(&A.ws->settle_next, 1u);
    j = __shfl_sync(kFull, j, 0) + (uint32_t)nTU;
    if (j >= nu) break;
    const uint32_t ri = j / (uint32_t)k1;
    const int pos = (int)(j - ri * (uint32_t)k1);
    const int row = a_row(P, (int)ri);
    const int u = row * k1 + pos;
    const RowCfg cfg = plan_cfg(A, P, row);
    if (lane == 0) TL(TL_SA_START, u, 2048);
    const Pre pr = load_pre<kBF16>(A, u, row, pos);
    fin_stats<kBF16>(A, tag, u, row, pos, cfg, pr);
    if (lane == 0) TL(TL_SA_END, u, 2048);
    __syncwarp();
  }
}

// The settle pass after the B pass: one warp per drafted unfiltered unit.
template <bool kBF16>
__device__ __noinline__ void settle_pass_b(const Args& A, Plan P, uint32_t tag, uint32_t gw, uint32_t nwarps) {
  const int lane = threadIdx.x & 31;
  const uint32_t nu = (uint32_t)b_units(A, P);
  for (uint32_t j = gw; j < nu; j += nwarps) {
    const uint32_t ri = j / (uint32_t)A.k;
    const int pos = (int)(j - ri * (uint32_t)A.k);
    const int row = (int)P.order[ri];
    const int u = row * (A.k + 1) + pos;
    const RowCfg cfg = plan_cfg(A, P, row);
    if (lane == 0) TL(TL_SB_START, u, 2048);
    StateWords sw8;
    state_load(A, u, sw8.w);
    fin_b<kBF16>(A, tag, u, row, pos, cfg, sw8);
    if (lane == 0) TL(TL_SB_END, u, 2048);
    __syncwarp();
  }
}

// Every CTA arrives before any leaves (the launch is cooperative, so all are
// resident).  The count only grows within a call: barrier i waits for
// i x n_ctas arrivals.  Bounded: a wait that gives up sets ERR_BARRIER and
// the CTA goes on (the record polls after it then give up too, and the rows
// come back with SPEC_F_TIMEOUT).
__device__ __noinline__ void grid_barrier(const Args& A, uint32_t target) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&A.ws->bar, 1u);
    long long spins = 0;
    while (load_acquire(&A.ws->bar) < target) {
      if (++spins > 16ll * kSpinLimit) {
        atomicOr(&A.ws->error, (uint32_t)ERR_BARRIER);
        break;
      }
      __nanosleep(spins > 16 ? 128 : 16);
    }
    __threadfence();
  }
  __syncthreads();
}

// General-path units, taken by the CTA's first kThreads threads.
template <bool kBF16>
__device__ __noinline__ void general_phase(const Args& A, Plan P, VShm& S, uint32_t tag) {
  const int k1 = A.k + 1;
  const int nGU = P.nX * k1;
  const int gbase = P.nD + P.nT;
  while (true) {
    if (ctid() == 0) S.gtask = (int)atomicAdd(&A.ws->gnext, 1u);
    csync();
    const int g = S.gtask;
    csync();
    if (g >= nGU) break;
    const int row = (int)P.order[gbase + g / k1], pos = g % k1;
    unit_general<kBF16>(A, S.gen, tag, row * k1 + pos, row, pos, plan_cfg(A, P, row));
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kAllThreads, 1) verify_kernel(const __grid_constant__ Args A) {
  using G = Geo<kBF16>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  VShm& S = *reinterpret_cast<VShm*>(smem_raw);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    S.tag = next_tag(__ldcg(&A.ws->epoch));
    S.gtask = 0;
    S.ticket[0] = 0u;
    S.ticket[1] = 0u;
  }
  if (lane == 0) {
    mbar_init(&S.bar[w][0], 1);    // issue() orders the inits before the copies (fence.proxy.async)
    mbar_init(&S.bar[w][1], 1);
    S.par[w][0] = 0u;
    S.par[w][1] = 0u;
    S.broken[w] = 0u;
  }
  Plan P;
  bool order_ok = true;
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
          atomicOr(&A.ws->error, (uint32_t)ERR_ORDER_WAIT);
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
  }
  const uint32_t tag = S.tag;
  P.NTA = ceil_div(A.V, G::EA);
  P.NTB = ceil_div(A.V, G::EB);
  __syncthreads();
  if (threadIdx.x == 0) TL(TL_CTA_START, (int)blockIdx.x, 160);
  // warp gw of nwarps: consecutive indices on different SMs
  const uint32_t nwarps = (uint32_t)A.n_ctas * kNW;
  const uint32_t gw = (uint32_t)w * (uint32_t)A.n_ctas + blockIdx.x;
  const uint32_t nb = (uint32_t)b_units(A, P) * (uint32_t)P.NTB;
  if (order_ok) {
    // A pass, then every unit's settle (the B pass's q into L2 meanwhile)
    stream_pass<kBF16>(A, P, S, tag, w, gw, 1, (uint32_t)a_units(A, P) * (uint32_t)P.NTA, &S.ticket[0]);
    grid_barrier(A, (uint32_t)A.n_ctas);
    settle_pass_a<kBF16>(A, P, S, tag);
    if (nb > 0) {
      // B pass over the drafted unfiltered units, then their settles
      grid_barrier(A, 2u * (uint32_t)A.n_ctas);
      stream_pass<kBF16>(A, P, S, tag, w, gw, 2, nb, &S.ticket[1]);
      grid_barrier(A, 3u * (uint32_t)A.n_ctas);
      settle_pass_b<kBF16>(A, P, tag, gw, nwarps);
    }
  }
  if (P.nX > 0 && order_ok) {
    __syncthreads();
    if (threadIdx.x < kThreads) general_phase<kBF16>(A, P, S, tag);
  }
  __syncthreads();
  if (A.fc.on && order_ok) {
    // the fused commit: every warp copies rows as they are finalized (not
    // after a copy wait that gave up: that copy may still land in a buffer)
    const bool copy_failed = (__shfl_sync(kFull, __ldcg(&A.ws->error), 0) & (uint32_t)ERR_COPY_WAIT) != 0u;
    if (!copy_failed) commit_phase(A, tag, S.s.buf[w][0], S.s.buf[w][1], S.cbar[w]);
    __syncthreads();
  }
  if (threadIdx.x == 0) TL(TL_CTA_END, (int)blockIdx.x, 160);
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t d = atomicAdd(&A.ws->ctas_done, 1u);
    if (d == (uint32_t)A.n_ctas - 1u) {
      __threadfence();
      A.ws->gnext = 0u;
      A.ws->bar = 0u;
      A.ws->settle_next = 0u;
      A.ws->commit_next = 0u;
      A.ws->done_count = 0u;
      A.ws->ctas_done = 0u;
      A.ws->last_error = __ldcg(&A.ws->error);
      A.ws->error = 0u;
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
      cached[dev] = sms;   // one CTA per SM
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
