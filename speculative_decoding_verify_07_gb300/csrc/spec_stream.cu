// spec_verify: the persistent verify kernel.
//
// Rows whose kept set needs a global threshold search (top-p without a small
// top-k, or a large top-k) run first, one (row, position) unit per CTA, on
// the general path (spec_general.cuh).  Greedy rows, rows with a small top-k
// (with or without top-p after it) and unfiltered rows then stream.
//
// Execution model: one persistent CTA per SM; every warp is an independent
// worker with two shared-memory buffers.  A warp pulls tickets from one
// counter, maps each ticket to a work item, and has the copy engine stream
// the item into a buffer (cp.async.bulk completed on an mbarrier) while it
// computes on the other buffer, so each SM keeps about 100 KB of HBM reads in
// flight without any block-wide barrier.
//
//   A item (unit, chunk of 6144 bf16 / 3072 fp32 entries): reduce the chunk
//     to a record -- max and first argmax, the softmax sum relative to the
//     chunk max, and at an unfiltered bonus position the level-1 race of the
//     chunk's 256-entry blocks; for a small top-k the maxima of its 64-entry
//     super-groups.  An atomic ticket per unit makes the warp that finishes
//     the last chunk the unit's finaliser.
//   B item (drafted unfiltered unit, chunk of 2048 / 1536 entries of logits
//     plus q): wait (bounded) for the unit state, then alpha = sum min(p, q)
//     and, after a rejection, the level-1 race of the residual max(p - q, 0).
//   Finalisers (one warp): merge records in chunk order; greedy and bonus
//     units are settled at once, a drafted unfiltered unit publishes its
//     accept decision for the B items, and a small top-k unit selects its
//     candidates from the super-group maxima, sorts them exactly and settles
//     top-p, the accept test, alpha and the draw on that list.
//
// Tickets are ordered: A items of drafted unfiltered units first, then top-k
// units and bonus unfiltered positions, then the B items, then greedy units,
// so the B items find their unit state ready and the expensive finalisers
// run early.
// A warp processes its tickets in increasing order and A items never wait, so
// every wait of a B item ends.  All reductions use a fixed order; no
// floating-point atomics are used, so results are bit-reproducible.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "spec_general.cuh"
#include "spec_host.h"
#include "spec_verify_common.cuh"

namespace specv {

constexpr int kSW = 8;                 // warps per streaming CTA
constexpr int kSThreads = kSW * 32;
constexpr int kOrderSmem = 1024;       // batches up to this many rows keep order and configs in shared memory
constexpr int kSgCap = 256;            // top-k finaliser: super-groups gathered
constexpr int kCandCap = 512;          // top-k finaliser: candidate entries
constexpr int kStage = 128;            // per-warp staging floats
constexpr int kStatic = 3;             // fixed tickets per warp before the counter is used
constexpr unsigned kFull = 0xffffffffu;

struct OrderScratch {
  int n_class[4];
  int run[4];
  int scan[kSW][4];
  int gtick;
};
static_assert(kSThreads == kThreads, "the general path runs on the streaming CTA");

struct alignas(128) StreamShm {
  unsigned char buf[kSW][2][kSlot];
  unsigned long long bar[kSW][2];
  float stage[kSW][kStage];
  uint32_t order[kOrderSmem];
  RowPack cfg[kOrderSmem];
  OrderScratch ord;
};
static_assert(sizeof(GenShm) <= kSW * 2 * kSlot, "general scratch exceeds the buffers");

// Top-k finaliser scratch inside a consumed buffer (byte offsets).  The
// unit's super-group maxima are staged at the start and turned into order
// keys while the threshold is found; once the super-groups are listed, the
// candidate list and then the kept list reuse that space.
constexpr int kScrMax = 10240;                      // staged maxima / keys (bytes)
constexpr int kScrHist = kScrMax;                   // 256 x u32
constexpr int kScrSg = kScrHist + 1024;             // kSgCap x u32
constexpr int kScrCand = 0;                         // kCandCap x u64
constexpr int kScrList = kScrCand + kCandCap * 8;   // kTopkSmall x 16 B entries, then cum and e
static_assert(kScrSg + kSgCap * 4 <= kSlot, "finaliser scratch exceeds a buffer");
static_assert(kScrList + kTopkSmall * 24 <= kScrHist, "list overlaps the histogram");

// ---------------------------------------------------------------------------
// Row order: rows of each class, stably, as [unfiltered][small top-k][greedy]
// [general].  Every thread of the CTA takes part.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int class_base(const OrderScratch& O, int cl) {
  const int nD = O.n_class[UT_DENSE], nT = O.n_class[UT_TOPK], nG = O.n_class[UT_GREEDY];
  return cl == UT_DENSE ? 0 : (cl == UT_TOPK ? nD : (cl == UT_GREEDY ? nD + nT : nD + nT + nG));
}

// Stable placement of one round of kSThreads rows (cl < 0: no row).
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

// Batches of up to kOrderSmem rows: one parameter load per row, the packed
// configs and the order in shared memory.
__device__ __noinline__ void build_order_smem(const Args& A, uint32_t* order, RowPack* cfgs, OrderScratch& O) {
  constexpr int kR = kOrderSmem / kSThreads;
  const int tid = threadIdx.x;
  if (tid < 4) {
    O.n_class[tid] = 0;
    O.run[tid] = 0;
  }
  __syncthreads();
  int cls[kR];
#pragma unroll
  for (int i = 0; i < kR; ++i) {
    const int r = tid + i * kSThreads;
    cls[i] = -1;
    if (r < A.B) {
      const RowCfg c = classify(A.params[r], A.V);
      cfgs[r] = pack_cfg(c);
      cls[i] = c.type;
      atomicAdd(&O.n_class[c.type], 1);
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kR; ++i)
    if (i * kSThreads < A.B) place_round(order, O, tid + i * kSThreads, cls[i]);
}

// Larger batches: one CTA writes the order and the class counts into the
// workspace before the streaming kernel runs.
__global__ void __launch_bounds__(kSThreads) plan_kernel(const Args A) {
  __shared__ OrderScratch O;
  const int tid = threadIdx.x;
  if (tid < 4) {
    O.n_class[tid] = 0;
    O.run[tid] = 0;
  }
  __syncthreads();
  for (int r = tid; r < A.B; r += kSThreads) atomicAdd(&O.n_class[classify(A.params[r], A.V).type], 1);
  __syncthreads();
  for (int base = 0; base < A.B; base += kSThreads) {
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
  int nD, nT, nG, NCA, NCB;
  int s0, s1, s2, s3, s4;   // segment sizes in tickets
};

struct Item {
  int kind;                 // 0 none, 1 A item, 2 B item
  int row, pos, u, c, n;    // unit, chunk, valid entries in the item
  RowCfg cfg;
};

template <bool kBF16>
__device__ __forceinline__ Item map_ticket(const Args& A, const Plan& P, uint32_t t) {
  using G = Geo<kBF16>;
  Item it;
  it.kind = 0;
  const int k = A.k, k1 = A.k + 1;
  if (t >= 0x7fffffffu) return it;
  int s = (int)t;
  int row, pos, c, kind;
  if (s < P.s0) {                       // drafted unfiltered units: A items
    const int j = s / P.NCA;
    c = s - j * P.NCA;
    row = (int)P.order[j / k];
    pos = j % k;
    kind = 1;
  } else if ((s -= P.s0) < P.s1) {      // small top-k units
    const int j = s / P.NCA;
    c = s - j * P.NCA;
    row = (int)P.order[P.nD + j / k1];
    pos = j % k1;
    kind = 1;
  } else if ((s -= P.s1) < P.s2) {      // unfiltered bonus positions
    const int j = s / P.NCA;
    c = s - j * P.NCA;
    row = (int)P.order[j];
    pos = k;
    kind = 1;
  } else if ((s -= P.s2) < P.s3) {      // drafted unfiltered units: B items
    const int j = s / P.NCB;
    c = s - j * P.NCB;
    row = (int)P.order[j / k];
    pos = j % k;
    kind = 2;
  } else if ((s -= P.s3) < P.s4) {      // greedy units
    const int j = s / P.NCA;
    c = s - j * P.NCA;
    row = (int)P.order[P.nD + P.nT + j / k1];
    pos = j % k1;
    kind = 1;
  } else {
    return it;
  }
  it.kind = kind;
  it.row = row;
  it.pos = pos;
  it.u = row * k1 + pos;
  it.c = c;
  const int E = kind == 1 ? G::EA : G::EB;
  it.n = min(E, A.V - c * E);
  it.cfg = P.cfg ? unpack_cfg(P.cfg[row]) : classify(A.params[row], A.V);
  return it;
}

// Lane 0: post the copies of an item into buffer `buf`, completing on `bar`.
template <bool kBF16>
__device__ __forceinline__ void issue(const Args& A, const Item& it, unsigned char* buf, unsigned long long* bar) {
  using G = Geo<kBF16>;
  if (it.kind == 0) return;
  const unsigned char* lg = reinterpret_cast<const unsigned char*>(A.logits);
  fence_proxy_async();
  if (it.kind == 1) {
    const uint32_t bl = A.vec_logits ? ((uint32_t)(it.n * G::es) & ~15u) : 0u;
    mbar_arrive_expect_tx(bar, bl);
    if (bl) bulk_g2s(buf, lg + ((size_t)it.u * A.V + (size_t)it.c * G::EA) * G::es, bl, bar);
  } else {
    const uint32_t bl = A.vec_logits ? ((uint32_t)(it.n * G::es) & ~15u) : 0u;
    const uint32_t bq = A.vec_q ? ((uint32_t)(it.n * 4) & ~15u) : 0u;
    mbar_arrive_expect_tx(bar, bl + bq);
    if (bl) bulk_g2s(buf, lg + ((size_t)it.u * A.V + (size_t)it.c * G::EB) * G::es, bl, bar);
    if (bq)
      bulk_g2s(buf + G::EB * G::es,
               A.q + ((size_t)it.row * A.k + it.pos) * (size_t)A.V + (size_t)it.c * G::EB, bq, bar);
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

// Maximum (NaN-propagating) of a lane's 8 slots of block b.
template <bool kBF16>
__device__ __forceinline__ float sgroup_max(const unsigned char* buf, int b, int l) {
  if (kBF16) {
    const uint2 a = *reinterpret_cast<const uint2*>(buf + (b * kRaceBlock + 4 * l) * 2);
    const uint2 c = *reinterpret_cast<const uint2*>(buf + (b * kRaceBlock + 128 + 4 * l) * 2);
    const uint32_t m2 = max_nan_bf16x2(max_nan_bf16x2(a.x, a.y), max_nan_bf16x2(c.x, c.y));
    return max_nan(bf16_lo(m2), bf16_hi(m2));
  } else {
    float v[8];
    sload<false>(buf, b, l, v);
    return group_max(v);
  }
}

// ---------------------------------------------------------------------------
// Unit finalisers (one warp each).
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ __noinline__ void fin_stats(const Args& A, const Item& it) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const RowCfg& cfg = it.cfg;
  const int u = it.u, row = it.row, pos = it.pos;
  const bool has_q = pos < A.k;
  const int NC = ceil_div(A.V, G::EA);
  const ChunkRec* R = A.crec + (size_t)u * A.NCA;
  bool nan = false;
  float m = -INFINITY;
  int cm = 0x7fffffff;
  for (int c = lane; c < NC; c += 32) {
    const float mc = __ldcg(&R[c].m);
    if (mc != mc) {
      nan = true;
    } else if (mc > m) {
      m = mc;
      cm = c;
    }
  }
  nan = __any_sync(kFull, nan);
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
  m = mw;
  const int am = (int)__ldcg(&R[cfirst].amax);
  // the softmax sum rescaled to the unit max (lane partials in chunk order)
  float Z = 0.f;
  for (int c = lane; c < NC; c += 32) {
    const float mc = __ldcg(&R[c].m);
    if (mc > -INFINITY) Z += __ldcg(&R[c].z) * ex2((mc - m) * cfg.c);
  }
  Z = warp_sum(Z);
  const float lnZ = logf(Z);
  if (cfg.type == UT_GREEDY) {
    if (lane == 0) {
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
    const AcceptInfo ai = accept_test(A, row, pos, kBF16, false, am, m, cfg.c, Z, nullptr);
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

// One warp: the bin of hist[0..256) where the count from bin 0 reaches
// `need`, and the count before it (255 when the bins never reach it).
__device__ __forceinline__ int warp_select_bin(const uint32_t* hist, uint32_t need, uint32_t* below) {
  const int lane = threadIdx.x & 31;
  uint32_t own = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) own += hist[8 * lane + i];
  uint32_t inc = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += y;
  }
  const unsigned ball = __ballot_sync(kFull, inc >= need);
  const int src = ball ? __ffs(ball) - 1 : 31;
  int chosen = 255;
  uint32_t bel = 0;
  if (lane == src) {
    uint32_t acc = inc - own;
    chosen = 8 * lane + 7;
    for (int i = 0; i < 8; ++i) {
      const uint32_t h = hist[8 * lane + i];
      if (acc + h >= need) {
        chosen = 8 * lane + i;
        break;
      }
      acc += h;
    }
    bel = acc;
  }
  chosen = __shfl_sync(kFull, chosen, src);
  *below = __shfl_sync(kFull, bel, src);
  return chosen;
}

__device__ __forceinline__ void warp_clear(uint32_t* h, int n) {
  for (int i = threadIdx.x & 31; i < n; i += 32) h[i] = 0u;
  __syncwarp();
}

template <bool kBF16>
__device__ __forceinline__ uint32_t kfk(float v) {
  return kBF16 ? (okey(v) >> 16) : okey(v);
}

// Key of super-group maximum s: from the staged keys in shared memory, or
// from the records in global memory when they were too many to stage.
template <bool kBF16, bool kStaged>
__device__ __forceinline__ uint32_t key_load(const uint32_t* skeys, const float* gvals, int s) {
  if (kStaged) return skeys[s];
  return kfk<kBF16>(__ldcg(gvals + s));
}

// Histogram of d = kmax - key over the entries with (d & mask) == prefix,
// bins (d >> shift) & 255 (or d >> shift below `lim` when lim != 0).
template <bool kBF16, bool kStaged>
__device__ __forceinline__ void warp_hist(const uint32_t* skeys, const float* gvals, int nsm, uint32_t kmax,
                                          uint32_t* hist, uint32_t lo, uint32_t span, int shift) {
  warp_clear(hist, 256);
  for (int base = threadIdx.x & 31; base < nsm; base += 128) {
    uint32_t d[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int s = base + 32 * j;
      d[j] = s < nsm ? kmax - key_load<kBF16, kStaged>(skeys, gvals, s) : 0xffffffffu;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (d[j] >= lo && d[j] - lo < span) atomicAdd(&hist[(d[j] - lo) >> shift], 1u);
  }
  __syncwarp();
}

// A key tau no larger than the K-th largest of the unit's super-group maxima
// (counting multiplicity): a histogram of the distance d = kmax - key, first
// with fine bins next to the maximum, refined 8 bits at a time while the bin
// holding rank K is wide and crowded; exact for bf16 in the usual case.
template <bool kBF16, bool kStaged>
__device__ __noinline__ uint32_t warp_kth_key(const uint32_t* skeys, const float* gvals, int nsm, uint32_t kmax,
                                              uint32_t K, uint32_t* hist) {
  const int s0 = kBF16 ? 0 : 16;
  const int dbits = kBF16 ? 16 : 32;
  uint32_t need = K;
  warp_hist<kBF16, kStaged>(skeys, gvals, nsm, kmax, hist, 0u, 255u << s0, s0);
  uint32_t below;
  const int b = warp_select_bin(hist, need, &below);
  if (b < 255) {
    need -= below;
    uint32_t cnt = hist[b];
    uint32_t lo = (uint32_t)b << s0;
    int sh = s0;
    while (sh > 0 && cnt > 64) {
      sh -= 8;
      __syncwarp();
      warp_hist<kBF16, kStaged>(skeys, gvals, nsm, kmax, hist, lo, 1u << (sh + 8), sh);
      uint32_t bl;
      const int bb = warp_select_bin(hist, need, &bl);
      need -= bl;
      cnt = hist[bb];
      lo += (uint32_t)bb << sh;
    }
    uint32_t dmax = lo + ((1u << sh) - 1u);
    if (dmax > kmax || dmax < lo) dmax = kmax;
    __syncwarp();
    return kmax - dmax;
  }
  // rank K lies far from the maximum: top-down radix over every bit of d
  uint32_t prefix = 0u;
  for (int shift = dbits - 8; shift >= 0; shift -= 8) {
    __syncwarp();
    // entries whose bits above `shift + 8` equal the prefix: d in [prefix, prefix + 2^(shift+8))
    const uint32_t span = (shift + 8 >= 32) ? 0xffffffffu : (1u << (shift + 8));
    warp_hist<kBF16, kStaged>(skeys, gvals, nsm, kmax, hist, prefix, span, shift);
    uint32_t bl;
    const int bb = warp_select_bin(hist, need, &bl);
    need -= bl;
    prefix |= (uint32_t)bb << shift;
    if (shift > 0 && hist[bb] <= 64) {
      uint32_t dmax = prefix | ((1u << shift) - 1u);
      if (dmax > kmax) dmax = kmax;
      __syncwarp();
      return kmax - dmax;
    }
  }
  __syncwarp();
  return kmax - prefix;
}

// Bitonic sort of s[0..n) in descending order, n a power of two, one warp.
__device__ __noinline__ void warp_bitonic_desc(unsigned long long* s, int n) {
  const int lane = threadIdx.x & 31;
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = lane; i < (n >> 1); i += 32) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long a = s[lo], b = s[hi];
        if ((a < b) == desc) {
          s[lo] = b;
          s[hi] = a;
        }
      }
      __syncwarp();
    }
  }
}

// Exact top-K list of a whole logit row by one warp (the fallback when the
// super-group candidates overflow, e.g. with massive ties): radix select of
// the K-th key over the row, then the entries above it and the first ties in
// index order.  Writes K sorted keys to cand and returns K.
template <bool kBF16>
__device__ __noinline__ int warp_row_topk(const Args& A, size_t lrow, uint32_t kmax, uint32_t K, uint32_t* hist,
                                          unsigned long long* cand) {
  const int lane = threadIdx.x & 31;
  const int G = (A.V + 7) / 8;
  const int dbits = kBF16 ? 16 : 32;
  uint32_t need = K, prefix = 0u, mask = 0u;
  for (int shift = dbits - 8; shift >= 0; shift -= 8) {
    __syncwarp();
    warp_clear(hist, 256);
    for (int g = lane; g < G; g += 32) {
      float v[8];
      load_group<kBF16>(A, lrow, g, true, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (g * 8 + j >= A.V) continue;
        const uint32_t d = kmax - kfk<kBF16>(v[j]);
        if ((d & mask) == prefix) atomicAdd(&hist[(d >> shift) & 255u], 1u);
      }
    }
    __syncwarp();
    uint32_t bl;
    const int bb = warp_select_bin(hist, need, &bl);
    need -= bl;
    prefix |= (uint32_t)bb << shift;
    mask |= 255u << shift;
  }
  const uint32_t tkey = kmax - prefix;   // K-th key; `need` ties at it are kept
  int n_above = 0;
  uint32_t ties_seen = 0;
  for (int base = 0; base < G; base += 32) {
    const int g = base + lane;
    float v[8];
    int nt = 0;
    if (g < G) {
      load_group<kBF16>(A, lrow, g, true, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (g * 8 + j >= A.V) continue;
        if (kfk<kBF16>(v[j]) == tkey) ++nt;
      }
    }
    // entries above the threshold: ballot-ordered appends
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool up = g < G && g * 8 + j < A.V && kfk<kBF16>(v[j]) > tkey;
      const unsigned b = __ballot_sync(kFull, up);
      if (up) cand[n_above + __popc(b & ((1u << lane) - 1u))] = key64(okey(v[j]), (uint32_t)(g * 8 + j));
      n_above += __popc(b);
    }
    // ties in index order (lanes hold consecutive groups)
    int inc = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += y;
    }
    const uint32_t exc = ties_seen + (uint32_t)(inc - nt);
    if (nt > 0 && exc < need) {
      uint32_t r = exc;
      for (int j = 0; j < 8; ++j) {
        if (g * 8 + j < A.V && kfk<kBF16>(v[j]) == tkey) {
          if (r < need) cand[(int)(K - need) + (int)r] = key64(okey(v[j]), (uint32_t)(g * 8 + j));
          ++r;
        }
      }
    }
    ties_seen += (uint32_t)__shfl_sync(kFull, inc, 31);
  }
  __syncwarp();
  int n = 1;
  while (n < (int)K) n <<= 1;
  for (int i = (int)K + lane; i < n; i += 32) cand[i] = 0ull;
  __syncwarp();
  warp_bitonic_desc(cand, n);
  return (int)K;
}

// Small top-k finaliser.  Every top-K entry lies in a 64-entry super-group
// whose maximum reaches tau (a lower bound of the K-th largest super-group
// maximum), so the entries >= tau of those super-groups hold the top K; they
// are gathered from L2, sorted exactly, and the first K settle the unit.
template <bool kBF16>
__device__ __noinline__ void fin_topk(const Args& A, const Item& it, unsigned char* scr, unsigned long long* bar,
                                      uint32_t& parity) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const RowCfg cfg = it.cfg;
  const int u = it.u, row = it.row, pos = it.pos;
  const bool has_q = pos < A.k;
  const int V = A.V;
  const int NC = ceil_div(V, G::EA);
  const int nsm = NC * G::SPI;
  const float* sm = A.smax + (size_t)u * A.NSM;
  const size_t lrow = (size_t)u * V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)V;
  uint32_t* hist = reinterpret_cast<uint32_t*>(scr + kScrHist);
  uint32_t* sg = reinterpret_cast<uint32_t*>(scr + kScrSg);
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(scr + kScrCand);
  float4* l4 = reinterpret_cast<float4*>(scr + kScrList);           // (index bits, w, w + tq, 0)
  float* l_cum = reinterpret_cast<float*>(scr + kScrList + kTopkSmall * 16);
  float* l_e = l_cum + kTopkSmall;
  // the draft token goes out first; its logit and q follow once it is back
  const int x = has_q ? A.drafts[(size_t)row * A.k + pos] : -1;
  // stage the maxima in shared memory with one bulk copy (the records were
  // published before the unit ticket this warp acquired)
  const bool staged = nsm * 4 <= kScrMax;
  if (staged) {
    if (lane == 0) {
      fence_proxy_async_all();
      mbar_arrive_expect_tx(bar, (uint32_t)(nsm * 4));
      bulk_g2s(scr, sm, (uint32_t)(nsm * 4), bar);
    }
    const bool ok = wait_buffer(A, bar, parity);
    parity ^= 1u;
    if (!ok) return;
  }
  uint32_t* keys = reinterpret_cast<uint32_t*>(scr);
  // order keys (in place when staged); the unit maximum; NaN
  uint32_t kmax = 0u;
  bool nan = false;
  for (int base = lane; base < nsm; base += 128) {
    float xv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int s = base + 32 * j;
      xv[j] = s < nsm ? (staged ? reinterpret_cast<const float*>(scr)[s] : __ldcg(sm + s)) : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int s = base + 32 * j;
      const uint32_t kk = kfk<kBF16>(xv[j]);
      if (xv[j] != xv[j]) nan = true;
      else kmax = max(kmax, kk);
      if (staged && s < nsm) keys[s] = kk;
    }
  }
  nan = __any_sync(kFull, nan);
  kmax = warp_max_u32(kmax);
  __syncwarp();
  const float m = from_okey(full_key<kBF16>(kmax));
  if (nan || !(m > -INFINITY) || !(m < INFINITY)) {
    if (lane == 0) commit_record(A, u, row, empty_record(SPEC_F_NAN));
    __syncwarp();
    return;
  }
  const uint32_t K = (uint32_t)cfg.K;
  uint32_t tau = 0u;
  if (K < (uint32_t)nsm)
    tau = staged ? warp_kth_key<kBF16, true>(keys, sm, nsm, kmax, K, hist)
                 : warp_kth_key<kBF16, false>(keys, sm, nsm, kmax, K, hist);
  // the accept test's loads overlap the gather below
  const bool xvalid = x >= 0 && x < V;
  const float lx = xvalid ? load_logit(A, kBF16, lrow + x) : 0.f;
  const float qx = xvalid ? A.q[qrow + x] : 0.f;
  // the qualifying super-groups
  int nsg = 0;
  for (int base = 0; base < nsm; base += 128) {
    uint32_t kk[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int s = base + 32 * j + lane;
      kk[j] = s >= nsm ? 0u : (staged ? key_load<kBF16, true>(keys, sm, s) : key_load<kBF16, false>(keys, sm, s));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int s = base + 32 * j + lane;
      const bool ok = s < nsm && kk[j] >= tau;
      const unsigned b = __ballot_sync(kFull, ok);
      if (ok) {
        const int p = nsg + __popc(b & ((1u << lane) - 1u));
        if (p < kSgCap) sg[p] = (uint32_t)s;
      }
      nsg += __popc(b);
    }
  }
  __syncwarp();
  bool overflow = nsg > kSgCap;
  int count = 0;
  if (!overflow) {
    // gather their entries >= tau; super-group r of a chunk is block r/4,
    // lanes 8(r%4)..8(r%4)+7, i.e. entries [32q, 32q+32) and [128+32q,
    // 128+32q+32) of the block with q = r%4
    const int ngr = nsg * 8;
    for (int base = 0; base < ngr; base += 128) {
      float v[4][8];
      int e[4];
      bool act[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int i = base + 32 * h + lane;
        act[h] = i < ngr;
        e[h] = 0;
        if (act[h]) {
          const int sgi = (int)sg[i >> 3];
          const int gi = i & 7;
          const int c = sgi / G::SPI, r = sgi - c * G::SPI;
          e[h] = c * G::EA + (r >> 2) * kRaceBlock + (gi >> 2) * 128 + (r & 3) * 32 + (gi & 3) * 8;
          load_group<kBF16>(A, lrow, e[h] >> 3, true, v[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < 4; ++h) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const bool up = act[h] && e[h] + j < V && kfk<kBF16>(v[h][j]) >= tau;
          const unsigned b = __ballot_sync(kFull, up);
          if (up) {
            const int p = count + __popc(b & ((1u << lane) - 1u));
            if (p < kCandCap) cand[p] = key64(okey(v[h][j]), (uint32_t)(e[h] + j));
          }
          count += __popc(b);
        }
      }
    }
    overflow = count > kCandCap;
  }
  __syncwarp();
  int n_k;
  if (!overflow) {
    int n = 1;
    while (n < count) n <<= 1;
    for (int i = count + lane; i < n; i += 32) cand[i] = 0ull;
    __syncwarp();
    warp_bitonic_desc(cand, n);
    n_k = min(count, (int)K);
  } else {
    n_k = warp_row_topk<kBF16>(A, lrow, kmax, K, hist, cand);
  }
  const int am = (int)key64_idx(cand[0]);

  // ---- the list: entries 4*lane .. 4*lane+3 of the first n_k ----
  float e4[4];
  uint32_t i4[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = 4 * lane + j;
    e4[j] = 0.f;
    i4[j] = 0u;
    if (i < n_k) {
      const unsigned long long key = cand[i];
      i4[j] = key64_idx(key);
      e4[j] = ex2((from_okey((uint32_t)(key >> 32)) - m) * cfg.c);
    }
  }
  __syncwarp();   // the candidate space is reused by the list from here on
  {
    // inclusive prefix sums in list order (fixed order)
    float run = 0.f;
    float cum4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      run += e4[j];
      cum4[j] = run;
    }
    float inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += y;
    }
    const float loc = inc - run;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = 4 * lane + j;
      if (i < n_k) {
        l_e[i] = e4[j];
        l_cum[i] = loc + cum4[j];
      }
    }
  }
  __syncwarp();
  const float Zk = l_cum[n_k - 1];
  uint32_t flags = cfg.bad_param ? SPEC_F_BAD_PARAM : 0u;
  int n_s = n_k;
  if (cfg.P < 1.0f) {
    const float target = cfg.P * Zk;
    uint32_t first = 0xffffffffu;
#pragma unroll
    for (int j = 3; j >= 0; --j) {
      const int i = 4 * lane + j;
      if (i < n_k && l_cum[i] >= target) first = (uint32_t)i;
    }
    first = warp_min_u32(first);
    n_s = (first == 0xffffffffu) ? n_k : (int)first + 1;
    const float at = l_cum[n_s - 1] / Zk;
    const float before = n_s >= 2 ? l_cum[n_s - 2] / Zk : 0.f;
    if (fabsf(at - cfg.P) < kMargin || fabsf(cfg.P - before) < kMargin) flags |= SPEC_F_MARGIN_TOPP;
  }
  const float Zs = l_cum[n_s - 1];
  const float invZ = 1.0f / Zs;
  const float lnZ = logf(Zs);
  float p4[4], q4[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = 4 * lane + j;
    const bool mine = i < n_s;
    p4[j] = mine ? e4[j] * invZ : 0.f;
    q4[j] = (mine && has_q) ? A.q[qrow + i4[j]] : 0.f;
  }
  float alpha_v = 0.f;
  bool need_race = !has_q;
  bool accept = false, margin = false;
  if (has_q) {
    int xi = -1;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (4 * lane + j < n_s && i4[j] == (uint32_t)x) xi = 4 * lane + j;
    const unsigned hb = __ballot_sync(kFull, xi >= 0);
    xi = hb ? __shfl_sync(kFull, xi, __ffs(hb) - 1) : -1;
    float al = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) al += fminf(p4[j], q4[j]);
    alpha_v = warp_sum(al);
    const float px = xi >= 0 ? l_e[xi] / Zs : 0.f;
    const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)pos, (uint32_t)row, 0u), A.key0, A.key1);
    const float uu = uniform_of(w.x);
    const float d = fmaf(uu, qx, -px);
    accept = d < 0.0f;
    margin = (px > 0.0f && px < 1.0f && fabsf(d) < kMargin);
    need_race = !accept;
  }
  // the draw: the two-level race over the kept entries (blocks by index)
  uint32_t draw_flags = 0;
  uint32_t y = 0xffffffffu;
  if (need_race) {
    for (int attempt = 0; attempt < 2; ++attempt) {
      const bool use_p = attempt == 1;          // empty residual: draw from p
      float w4[4], t4[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 4 * lane + j;
        w4[j] = (has_q && !use_p) ? fmaxf(p4[j] - q4[j], 0.f) : p4[j];
        t4[j] = (has_q && !use_p) ? 2.0f * q4[j] : 0.f;
        if (i < n_s) l4[i] = make_float4(__uint_as_float(i4[j]), w4[j], w4[j] + t4[j], 0.f);
      }
      __syncwarp();
      // level 1: the first list entry of each block races for its block, with
      // the block's weights summed in list order
      Race r1;
      race_init(r1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 4 * lane + j;
        if (i < n_s && w4[j] > 0.f) {
          const uint32_t b = i4[j] / kRaceBlock;
          bool rep = true;
          float W = 0.f, U = 0.f;
#pragma unroll 4
          for (int jj = 0; jj < n_s; ++jj) {
            const float4 L = l4[jj];
            if (__float_as_uint(L.x) / kRaceBlock == b && L.y > 0.f) {
              if (jj < i) rep = false;
              W += L.y;
              U += L.z;
            }
          }
          if (rep) race_consider(r1, W, U - W, b, block_word(A, row, pos, b));
        }
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
      for (int j = 0; j < 4; ++j) {
        const int i = 4 * lane + j;
        if (i < n_s && w4[j] > 0.f && i4[j] / kRaceBlock == r1.v1)
          race_consider(r2, w4[j], t4[j], i4[j], race_word(A, row, pos, i4[j]));
      }
      warp_race_merge(r2);
      y = r2.v1;
      if (draw_margin(r1) || draw_margin(r2)) draw_flags |= SPEC_F_MARGIN_DRAW;
      break;
    }
  }
  if (lane == 0) {
    UnitRecord rec = empty_record(flags);
    if (has_q) {
      if (!xvalid) rec.flags |= SPEC_F_BAD_TOKEN;
      if (margin) rec.flags |= SPEC_F_MARGIN_ACCEPT;
      rec.accept = accept ? 1 : 0;
      rec.lp_x = xvalid ? (lx - m) * cfg.invT - lnZ : 0.f;
      rec.alpha = alpha_v;
    }
    if (need_race) {
      const uint32_t yy = y < (uint32_t)V ? y : (uint32_t)am;
      rec.y = (int32_t)yy;
      rec.lp_y = (load_logit(A, kBF16, lrow + yy) - m) * cfg.invT - lnZ;
      rec.draw_flags = draw_flags;
    }
    commit_record(A, u, row, rec);
  }
  __syncwarp();
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

template <bool kBF16>
__device__ __noinline__ void fin_b(const Args& A, const Item& it) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int u = it.u, row = it.row, pos = it.pos;
  const RowCfg& cfg = it.cfg;
  const UnitState st = load_state(A, u);
  if (st.invalid) {   // the A finaliser wrote the record already
    if (lane == 0) {
      A.b_ticket[u] = 0;
      A.ready[u] = 0;
    }
    __syncwarp();
    return;
  }
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

// ---------------------------------------------------------------------------
// Item processing (one warp).  An item's record is stored when the item ends;
// its unit ticket is taken one item later (the release then finds the store
// long completed) and read one item after that, when the finaliser of a
// completed unit runs with the buffer just consumed as scratch.
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ void a_compute(const Args& A, const Item& it, const unsigned char* buf, float* stage, ChunkRec& rec) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int nb = ceil_div(it.n, kRaceBlock);
  const int e0 = it.c * G::EA;
  const RowCfg& cfg = it.cfg;
  if (cfg.type == UT_TOPK) {
    // maxima of the 64-entry super-groups (8 consecutive lanes of a block)
#pragma unroll 4
    for (int b = 0; b < nb; ++b) {
      float gm = sgroup_max<kBF16>(buf, b, lane);
      gm = max_nan(gm, __shfl_xor_sync(kFull, gm, 1));
      gm = max_nan(gm, __shfl_xor_sync(kFull, gm, 2));
      gm = max_nan(gm, __shfl_xor_sync(kFull, gm, 4));
      if ((lane & 7) == 0) stage[b * 4 + (lane >> 3)] = gm;
    }
    __syncwarp();
    float* dst = A.smax + (size_t)it.u * A.NSM + (size_t)it.c * G::SPI;
    for (int s = lane; s < G::SPI; s += 32) dst[s] = s < nb * 4 ? stage[s] : -INFINITY;
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
    const float gm = sgroup_max<kBF16>(buf, b, lane);
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
        race_consider(r, myW, 0.f, blk, block_word(A, it.row, it.pos, blk));
      }
      warp_race_merge(r);
    }
  }
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

template <bool kBF16>
__device__ void b_compute(const Args& A, const Item& it, const unsigned char* buf, BRec& br) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int nb = ceil_div(it.n, kRaceBlock);
  const int e0 = it.c * G::EB;
  const RowCfg& cfg = it.cfg;
  // the unit state (bounded wait; every A item was claimed before any B item,
  // and a warp resolves its pending A tickets before it starts a B item)
  if (lane == 0) {
    long long spins = 0;
    while (load_acquire(&A.ready[it.u]) == 0u) {
      if (++spins > kSpinLimit) {
        atomicOr(&A.ws->error, 1u);
        break;
      }
      __nanosleep(64);
    }
  }
  __syncwarp();
  const UnitState st = load_state(A, it.u);
  const bool need_race = !st.accept;
  const float* qb = reinterpret_cast<const float*>(buf + G::EB * G::es);
  float alpha_c = 0.f, myW = 0.f, myU = 0.f;
  if (!st.invalid) {
    const float m = st.m, invZ = st.invZ, c = cfg.c;
    for (int b = 0; b < nb; ++b) {
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
      if (need_race) {
        const float Wb = warp_sum(w8), Ub = warp_sum(u8);
        if (lane == b) {
          myW = Wb;
          myU = Ub;
        }
      }
    }
  }
  Race r;
  race_init(r);
  if (need_race && myW > 0.f) {
    const uint32_t blk = (uint32_t)(e0 / kRaceBlock + lane);
    race_consider(r, myW, myU - myW, blk, block_word(A, it.row, it.pos, blk));
  }
  warp_race_merge(r);
  br.alpha = alpha_c;
  br.s1 = r.s1;
  br.t1 = r.t1;
  br.s2 = r.s2;
  br.t2 = r.t2;
  br.v1 = r.v1;
  br.pad[0] = br.pad[1] = 0;
}

// A processed item whose unit ticket is still to be taken or read.
struct Pending {
  Item it;                  // kind 0: none
  uint32_t t;               // the ticket value (lane 0), once taken
};

template <bool kBF16>
__device__ __forceinline__ uint32_t* ticket_of(const Args& A, const Item& it) {
  return it.kind == 1 ? A.a_ticket + it.u : A.b_ticket + it.u;
}
template <bool kBF16>
__device__ __forceinline__ uint32_t last_ticket(const Args& A, const Item& it) {
  return (uint32_t)(it.kind == 1 ? ceil_div(A.V, Geo<kBF16>::EA) : ceil_div(A.V, Geo<kBF16>::EB)) - 1u;
}

// Lane 0's ticket value t (valid in lane 0 only) decides whether this warp
// settles the item's unit; the finaliser's scratch is a consumed buffer.
template <bool kBF16>
__device__ void settle(const Args& A, const Item& it, uint32_t t, unsigned char* scr, unsigned long long* bar,
                       uint32_t& parity) {
  t = __shfl_sync(kFull, t, 0);
  if (t != last_ticket<kBF16>(A, it)) return;
  if (it.kind == 1) {
    if ((threadIdx.x & 31) == 0) A.a_ticket[it.u] = 0;
    __syncwarp();
    if (it.cfg.type == UT_TOPK) fin_topk<kBF16>(A, it, scr, bar, parity);
    else fin_stats<kBF16>(A, it);
  } else {
    fin_b<kBF16>(A, it);
  }
}

// Take the pending tickets now and settle what they complete.
template <bool kBF16>
__device__ void flush(const Args& A, Pending& p0, Pending& p1, unsigned char* scr, unsigned long long* bar,
                      uint32_t& parity) {
  uint32_t t0 = 0;
  if ((threadIdx.x & 31) == 0 && p0.it.kind != 0) t0 = atomic_add_acq_rel(ticket_of<kBF16>(A, p0.it), 1u);
  if (p1.it.kind != 0) settle<kBF16>(A, p1.it, p1.t, scr, bar, parity);
  if (p0.it.kind != 0) settle<kBF16>(A, p0.it, t0, scr, bar, parity);
  p0.it.kind = 0;
  p1.it.kind = 0;
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <bool kBF16>
__global__ void __launch_bounds__(kSThreads, 1) stream_kernel(const Args A) {
  using G = Geo<kBF16>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StreamShm& S = *reinterpret_cast<StreamShm*>(smem_raw);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) {
    mbar_init(&S.bar[w][0], 1);
    mbar_init(&S.bar[w][1], 1);
  }
  Plan P;
  int nX;
  if (!A.global_order) {
    build_order_smem(A, S.order, S.cfg, S.ord);
    P.order = S.order;
    P.cfg = S.cfg;
    P.nD = S.ord.n_class[UT_DENSE];
    P.nT = S.ord.n_class[UT_TOPK];
    P.nG = S.ord.n_class[UT_GREEDY];
    nX = S.ord.n_class[UT_GENERAL];
  } else {
    P.order = A.order;
    P.cfg = nullptr;
    P.nD = (int)__ldcg(&A.ws->n_class[UT_DENSE]);
    P.nT = (int)__ldcg(&A.ws->n_class[UT_TOPK]);
    P.nG = (int)__ldcg(&A.ws->n_class[UT_GREEDY]);
    nX = (int)__ldcg(&A.ws->n_class[UT_GENERAL]);
  }
  fence_mbar_init();
  __syncthreads();
  // general rows first: whole CTAs claim their units; the buffers are free
  // until the first streaming copy is posted
  if (nX > 0) {
    GenShm& Sg = *reinterpret_cast<GenShm*>(&S.buf[0][0][0]);
    const int nGU = nX * (A.k + 1);
    const int gbase = P.nD + P.nT + P.nG;
    while (true) {
      if (threadIdx.x == 0) S.ord.gtick = (int)atomicAdd(&A.ws->gnext, 1u);
      __syncthreads();
      const int g = S.ord.gtick;
      __syncthreads();
      if (g >= nGU) break;
      const int row = (int)P.order[gbase + g / (A.k + 1)], pos = g % (A.k + 1);
      const RowCfg cfg = P.cfg ? unpack_cfg(P.cfg[row]) : classify(A.params[row], A.V);
      unit_general<kBF16>(A, Sg, row * (A.k + 1) + pos, row, pos, cfg);
    }
  }
  P.NCA = ceil_div(A.V, G::EA);
  P.NCB = ceil_div(A.V, G::EB);
  P.s0 = P.nD * A.k * P.NCA;
  P.s1 = P.nT * (A.k + 1) * P.NCA;
  P.s2 = P.nD * P.NCA;
  P.s3 = P.nD * A.k * P.NCB;
  P.s4 = P.nG * (A.k + 1) * P.NCA;
  // The first kStatic tickets of each warp are fixed (warp g takes g, g + NW,
  // g + 2 NW, with NW warps in the grid), so the launch starts without a
  // burst of atomics on one counter; later tickets come from the counter.
  const uint32_t nw = (uint32_t)A.n_ctas * kSW;
  const uint32_t gw = (uint32_t)blockIdx.x * kSW + (uint32_t)w;
  int nstat = 2;   // static tickets used so far
  // slot a holds the oldest outstanding ticket, slot b the next one
  Item ia = map_ticket<kBF16>(A, P, gw);
  Item ib = map_ticket<kBF16>(A, P, gw + nw);
  unsigned char* bufa = S.buf[w][0];
  unsigned char* bufb = S.buf[w][1];
  unsigned long long* bara = &S.bar[w][0];
  unsigned long long* barb = &S.bar[w][1];
  uint32_t para = 0u, parb = 0u;
  uint32_t tn = gw + 2 * nw;
  if (lane == 0) {
    issue<kBF16>(A, ia, bufa, bara);
    issue<kBF16>(A, ib, bufb, barb);
  }
  Pending p0, p1;
  p0.it.kind = 0;
  p1.it.kind = 0;
  p0.t = p1.t = 0;
  bool ok = true;
  while (ia.kind != 0) {
    if (!wait_buffer(A, bara, para)) {
      ok = false;
      break;
    }
    para ^= 1u;
    if (!A.vec_logits || (ia.kind == 2 && !A.vec_q) || (ia.n & (kRaceBlock - 1)) != 0)
      fill_tail<kBF16>(A, ia, bufa);
    ChunkRec rec;
    BRec br;
    if (ia.kind == 1) a_compute<kBF16>(A, ia, bufa, S.stage[w], rec);
    else b_compute<kBF16>(A, ia, bufa, br);
    // the ticket of the item before (its record was stored an item ago)
    uint32_t t0 = 0;
    if (lane == 0 && p0.it.kind != 0) t0 = atomic_add_acq_rel(ticket_of<kBF16>(A, p0.it), 1u);
    // this item's record
    if (lane == 0) {
      if (ia.kind == 2) A.brec[(size_t)ia.u * A.NCB + ia.c] = br;
      else if (ia.cfg.type != UT_TOPK) A.crec[(size_t)ia.u * A.NCA + ia.c] = rec;
    }
    __syncwarp();
    // the ticket taken an item ago
    if (p1.it.kind != 0) settle<kBF16>(A, p1.it, p1.t, bufa, bara, para);
    p1.it = p0.it;
    p1.t = t0;
    p0.it = ia;
    // B items wait on A finalisers: settle pending A items before one starts
    if (ib.kind == 2 && (p0.it.kind == 1 || p1.it.kind == 1)) flush<kBF16>(A, p0, p1, bufa, bara, para);
    // refill the consumed buffer with the next ticket, then rotate the slots
    const uint32_t t = __shfl_sync(kFull, tn, 0);
    Item in;
    in.kind = 0;
    if (ib.kind != 0) in = map_ticket<kBF16>(A, P, t);
    if (lane == 0) {
      issue<kBF16>(A, in, bufa, bara);
      if (in.kind != 0) {
        if (nstat + 1 < kStatic) {
          tn = gw + (uint32_t)(nstat + 1) * nw;
        } else {
          tn = atomicAdd(&A.ws->next, 1u) + (uint32_t)kStatic * nw;
        }
      }
    }
    ++nstat;
    ia = ib;
    ib = in;
    unsigned char* tb = bufa;
    bufa = bufb;
    bufb = tb;
    unsigned long long* tr = bara;
    bara = barb;
    barb = tr;
    const uint32_t tp = para;
    para = parb;
    parb = tp;
  }
  if (ok) flush<kBF16>(A, p0, p1, bufa, bara, para);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t d = atomicAdd(&A.ws->ctas_done, 1u);
    if (d == (uint32_t)A.n_ctas - 1u) {
      A.ws->next = 0u;
      A.ws->ctas_done = 0u;
      A.ws->gnext = 0u;
      for (int i = 0; i < 4; ++i) A.ws->n_class[i] = 0u;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
template <bool kBF16>
int launch_stream(const Args& A0, cudaStream_t stream) {
  static std::mutex mu;
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  int n = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
      auto kern = stream_kernel<kBF16>;
      int per_sm = 0, sms = 0;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(StreamShm)) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSThreads, sizeof(StreamShm)) !=
              cudaSuccess ||
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
  if (A.global_order) {
    plan_kernel<<<1, kSThreads, 0, stream>>>(A);
    if (cudaGetLastError() != cudaSuccess) return SPEC_E_CUDA;
  }
  stream_kernel<kBF16><<<A.n_ctas, kSThreads, sizeof(StreamShm), stream>>>(A);
  if (cudaGetLastError() != cudaSuccess) return SPEC_E_CUDA;
  return SPEC_OK;
}

template int launch_stream<true>(const Args&, cudaStream_t);
template int launch_stream<false>(const Args&, cudaStream_t);

}  // namespace specv
