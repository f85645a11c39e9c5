// spec_verify, streaming kernels (sm_103a).
//
// Both kernels run one persistent CTA of 16 warps per SM; every warp is an
// independent worker with two 6 KB shared-memory buffers.  A warp takes the
// items t = g, g + NW, g + 2 NW, ... (g its index in the grid, NW the warps
// in the grid), has the copy engine stream each item into a buffer
// (cp.async.bulk completed on an mbarrier) while it computes on the other
// one, and reduces it with warp collectives only: no block-wide barrier and
// no atomics on the streaming path.
//
//   Stats kernel, A item (unit, chunk of 3072 bf16 / 1536 fp32 entries):
//     max and first argmax, the softmax sum relative to the chunk max, and at
//     an unfiltered bonus position the level-1 race of the chunk's 256-entry
//     blocks; for a small top-k the maxima of its 64-entry super-groups.
//     The unit kernel (spec_unit.cu) then settles every unit from these
//     records.
//   B-pass kernel, B item (drafted unfiltered unit, chunk of 1024 / 768
//     entries of logits plus q): alpha = sum min(p, q) and, after a
//     rejection, the level-1 race of the residual max(p - q, 0).  An atomic
//     ticket per unit makes the warp that finishes the last chunk settle the
//     unit: level 2 of the race, the unit record, the row.
//
// All reductions use a fixed order; no floating-point atomics are used, so
// results are bit-reproducible.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "spec_host.h"
#include "spec_verify_common.cuh"

namespace specv {

constexpr int kSW = 16;                // warps per streaming CTA
constexpr int kSThreads = kSW * 32;
constexpr int kCfgSmem = 1024;         // batches up to this many rows keep their configs in shared memory
constexpr int kStage = 64;             // per-warp staging floats (super-group maxima of an item)
constexpr unsigned kFull = 0xffffffffu;
static_assert(Geo<true>::SPI <= kStage && Geo<false>::SPI <= kStage, "staging too small");

struct alignas(128) StreamShm {
  unsigned char buf[kSW][2][kSlot];
  unsigned long long bar[kSW][2];
  float stage[kSW][kStage];
  RowPack cfg[kCfgSmem];
};

// Per-row configurations in shared memory (one parameter load per row).
__device__ void build_cfg(const Args& A, RowPack* cfgs) {
  if (A.B <= kCfgSmem)
    for (int r = threadIdx.x; r < A.B; r += kSThreads) cfgs[r] = pack_cfg(classify(A.params[r], A.V));
  __syncthreads();
}

__device__ __forceinline__ RowCfg row_cfg(const Args& A, const RowPack* cfgs, int row) {
  return A.B <= kCfgSmem ? unpack_cfg(cfgs[row]) : classify(A.params[row], A.V);
}

// A work item.  kind: 0 none, 1 A item, 2 B item.
struct Item {
  int kind;
  int row, pos, u, c, n;    // unit, chunk, valid entries in the item
  RowCfg cfg;
  UnitState st;             // B items: the unit state, read when the item is mapped
};

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

// ---------------------------------------------------------------------------
// Stats kernel.
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ __forceinline__ Item map_a(const Args& A, const RowPack* cfgs, uint32_t t, uint32_t total) {
  using G = Geo<kBF16>;
  Item it;
  it.kind = 0;
  if (t >= total) return it;
  const int NC = ceil_div(A.V, G::EA);
  const int u = (int)(t / (uint32_t)NC);
  it.c = (int)t - u * NC;
  it.u = u;
  it.row = u / (A.k + 1);
  it.pos = u - it.row * (A.k + 1);
  it.n = min(G::EA, A.V - it.c * G::EA);
  it.kind = 1;   // the row configuration is looked up when the item is reduced
  return it;
}

template <bool kBF16>
__device__ void a_compute(const Args& A, const Item& it, const unsigned char* buf, float* stage, const RowPack* cfgs) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int nb = ceil_div(it.n, kRaceBlock);
  const int e0 = it.c * G::EA;
  const RowCfg cfg = row_cfg(A, cfgs, it.row);
  if (cfg.type == UT_GENERAL) return;   // general rows are read by the unit kernel itself
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
        race_consider(r, myW, 0.f, blk, block_word(A, it.row, it.pos, blk));
      }
      warp_race_merge(r);
    }
  }
  if (lane == 0) {
    ChunkRec rec;
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
    A.crec[(size_t)it.u * A.NCA + it.c] = rec;
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kSThreads, 1) stats_kernel(const Args A) {
  using G = Geo<kBF16>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StreamShm& S = *reinterpret_cast<StreamShm*>(smem_raw);
  // the unit kernel may be scheduled now; it waits for this grid's results
  pdl_trigger();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t nw = (uint32_t)A.n_ctas * kSW;
  const uint32_t total = (uint32_t)A.U * (uint32_t)ceil_div(A.V, G::EA);
  uint32_t t = (uint32_t)blockIdx.x * kSW + (uint32_t)w;
  Item ia = map_a<kBF16>(A, S.cfg, t, total);
  Item ib = map_a<kBF16>(A, S.cfg, t + nw, total);
  t += 2 * nw;
  unsigned char* bufa = S.buf[w][0];
  unsigned char* bufb = S.buf[w][1];
  unsigned long long* bara = &S.bar[w][0];
  unsigned long long* barb = &S.bar[w][1];
  uint32_t para = 0u, parb = 0u;
  // the first two copies go out before the row configurations are read
  if (lane == 0) {
    mbar_init(bara, 1);
    mbar_init(barb, 1);
    fence_mbar_init();
    issue<kBF16>(A, ia, bufa, bara);
    issue<kBF16>(A, ib, bufb, barb);
  }
  build_cfg(A, S.cfg);
  while (ia.kind != 0) {
    if (!wait_buffer(A, bara, para)) break;
    para ^= 1u;
    if (!A.vec_logits || (ia.n & (kRaceBlock - 1)) != 0) fill_tail<kBF16>(A, ia, bufa);
    a_compute<kBF16>(A, ia, bufa, S.stage[w], S.cfg);
    __syncwarp();
    Item in;
    in.kind = 0;
    if (ib.kind != 0) {
      in = map_a<kBF16>(A, S.cfg, t, total);
      t += nw;
    }
    if (lane == 0) issue<kBF16>(A, in, bufa, bara);
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
}

// ---------------------------------------------------------------------------
// B-pass kernel.
// ---------------------------------------------------------------------------
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

// B item t (t < end); `prev` is the item mapped before it (kind 0: none),
// whose unit, configuration and state are reused when t is in the same unit.
template <bool kBF16>
__device__ __forceinline__ Item map_b(const Args& A, const RowPack* cfgs, uint32_t t, uint32_t end, const Item& prev) {
  using G = Geo<kBF16>;
  Item it;
  it.kind = 0;
  if (t >= end) return it;
  const int NC = ceil_div(A.V, G::EB);
  const int j = (int)(t / (uint32_t)NC);
  it.c = (int)t - j * NC;
  if (prev.kind == 2 && it.c > 0) {   // item t - 1 was `prev`, in the same unit
    it.u = prev.u;
    it.row = prev.row;
    it.pos = prev.pos;
    it.cfg = prev.cfg;
    it.st = prev.st;
  } else {
    it.u = (int)__ldcg(A.dlist + j);
    it.row = it.u / (A.k + 1);
    it.pos = it.u - it.row * (A.k + 1);
    it.cfg = row_cfg(A, cfgs, it.row);
    it.st = load_state(A, it.u);
  }
  it.n = min(G::EB, A.V - it.c * G::EB);
  it.kind = 2;
  return it;
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
__device__ __noinline__ void fin_b(const Args& A, const Item& it) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int u = it.u, row = it.row, pos = it.pos;
  const RowCfg& cfg = it.cfg;
  const UnitState& st = it.st;
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
    commit_record(A, u, row, rec);
  }
  __syncwarp();
}

template <bool kBF16>
__device__ void b_compute(const Args& A, const Item& it, const unsigned char* buf, BRec& br) {
  using G = Geo<kBF16>;
  const int lane = threadIdx.x & 31;
  const int nb = ceil_div(it.n, kRaceBlock);
  const int e0 = it.c * G::EB;
  const RowCfg& cfg = it.cfg;
  const UnitState& st = it.st;
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

template <bool kBF16>
__global__ void __launch_bounds__(kSThreads, 1) bpass_kernel(const Args A) {
  using G = Geo<kBF16>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StreamShm& S = *reinterpret_cast<StreamShm*>(smem_raw);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) {
    mbar_init(&S.bar[w][0], 1);
    mbar_init(&S.bar[w][1], 1);
  }
  build_cfg(A, S.cfg);
  fence_mbar_init();
  // the unit states and the unit list come from the unit kernel
  pdl_wait();
  __syncthreads();
  // each warp takes a contiguous range of items, so it reads a unit's state
  // once and takes the unit's ticket once per run of chunks
  const uint32_t nw = (uint32_t)A.n_ctas * kSW;
  const uint32_t total = __ldcg(&A.ws->n_dense) * (uint32_t)ceil_div(A.V, G::EB);
  const uint32_t per = (total + nw - 1) / nw;
  const uint32_t gw = (uint32_t)blockIdx.x * kSW + (uint32_t)w;
  uint32_t t = min(total, gw * per);
  const uint32_t end = min(total, t + per);
  Item none;
  none.kind = 0;
  Item ia = map_b<kBF16>(A, S.cfg, t, end, none);
  Item ib = map_b<kBF16>(A, S.cfg, t + 1, end, ia);
  t += 2;
  unsigned char* bufa = S.buf[w][0];
  unsigned char* bufb = S.buf[w][1];
  unsigned long long* bara = &S.bar[w][0];
  unsigned long long* barb = &S.bar[w][1];
  uint32_t para = 0u, parb = 0u;
  if (lane == 0) {
    issue<kBF16>(A, ia, bufa, bara);
    issue<kBF16>(A, ib, bufb, barb);
  }
  Item run = none;           // the unit whose chunks this warp is processing
  uint32_t run_n = 0;        // chunks of it processed so far
  const uint32_t last = (uint32_t)ceil_div(A.V, G::EB);
  // add this warp's chunks of the run's unit to its ticket; the warp that
  // completes the unit settles it
  auto close_run = [&]() {
    if (run.kind == 0) return;
    uint32_t old = 0;
    if (lane == 0) old = atomic_add_acq_rel(&A.b_ticket[run.u], run_n);
    old = __shfl_sync(kFull, old, 0);
    __syncwarp();
    if (old + run_n == last) fin_b<kBF16>(A, run);
    run.kind = 0;
    run_n = 0;
  };
  while (ia.kind != 0) {
    if (!wait_buffer(A, bara, para)) break;
    para ^= 1u;
    if (!A.vec_logits || !A.vec_q || (ia.n & (kRaceBlock - 1)) != 0) fill_tail<kBF16>(A, ia, bufa);
    BRec br;
    b_compute<kBF16>(A, ia, bufa, br);
    if (lane == 0) A.brec[(size_t)ia.u * A.NCB + ia.c] = br;
    __syncwarp();
    if (run.kind != 0 && run.u != ia.u) close_run();
    if (run.kind == 0) run = ia;
    ++run_n;
    Item in = map_b<kBF16>(A, S.cfg, t, end, ib);
    ++t;
    if (lane == 0) issue<kBF16>(A, in, bufa, bara);
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
  close_run();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t d = atomicAdd(&A.ws->ctas_done, 1u);
    if (d == (uint32_t)A.n_ctas - 1u) {
      A.ws->n_dense = 0u;
      A.ws->ctas_done = 0u;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
template <bool kStats, bool kBF16>
static int stream_grid(int* n) {
  static std::mutex mu;
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    auto kern = kStats ? stats_kernel<kBF16> : bpass_kernel<kBF16>;
    int per_sm = 0, sms = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(StreamShm)) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSThreads, sizeof(StreamShm)) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || per_sm <= 0) {
      cudaGetLastError();
      return SPEC_E_CUDA;
    }
    cached[dev] = per_sm * sms;
  }
  *n = cached[dev];
  return SPEC_OK;
}

template <bool kBF16>
int launch_stats(const Args& A0, cudaStream_t stream) {
  Args A = A0;
  const int rc = stream_grid<true, kBF16>(&A.n_ctas);
  if (rc != SPEC_OK) return rc;
  stats_kernel<kBF16><<<A.n_ctas, kSThreads, sizeof(StreamShm), stream>>>(A);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_E_CUDA;
}

template <bool kBF16>
int launch_bpass(const Args& A0, cudaStream_t stream) {
  Args A = A0;
  const int rc = stream_grid<false, kBF16>(&A.n_ctas);
  if (rc != SPEC_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)A.n_ctas);
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = sizeof(StreamShm);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, bpass_kernel<kBF16>, A) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  return SPEC_OK;
}

template int launch_stats<true>(const Args&, cudaStream_t);
template int launch_stats<false>(const Args&, cudaStream_t);
template int launch_bpass<true>(const Args&, cudaStream_t);
template int launch_bpass<false>(const Args&, cudaStream_t);

}  // namespace specv
