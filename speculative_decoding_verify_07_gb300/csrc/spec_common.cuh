// Device-side pieces shared by the verify kernel (sm_103a): tile geometry,
// workspace layout, kernel arguments, row classification, loads, the accept
// test, the exponential race and the per-row finalize.
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
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#include "../../include/spec_verify.h"
#include "spec_device.cuh"

namespace specv {

constexpr int kRaceBlock = 256;            // entries per block of the two-level race
constexpr int kTopkSmall = 128;            // top_k <= this: candidate-list path
constexpr int kMaxListCand = 640;          // ... when the tiles' candidate lists of a row fit a settle warp
// Polls of a bounded wait before it gives up (with a short sleep per poll:
// a few hundred milliseconds in all).
constexpr long long kSpinLimit = 1ll << 21;
constexpr int kCtaWarps = 12;              // warps of a verify CTA

// Tile geometry.  Every stream warp owns two shared buffers of kSlot bytes.
// An A tile is one buffer of logits; a B tile is logits (read again, from
// L2) plus the matching draft probabilities.  Tiles cover whole race blocks
// of 256 entries.
constexpr int kSlot = 8192;
template <bool kBF16>
struct Geo {
  static constexpr int es = kBF16 ? 2 : 4;                         // logit bytes
  static constexpr int EA = kBF16 ? 4096 : 2048;                   // A tile entries (16 / 8 blocks; 8 KB)
  static constexpr int EB = kBF16 ? 1280 : 1024;                   // B tile entries (5 / 4 blocks)
  static constexpr int NBA = EA / kRaceBlock;
  static constexpr int NBB = EB / kRaceBlock;
  static_assert(EA * es <= kSlot, "A tile exceeds a buffer");
  static_assert(EB * (es + 4) <= kSlot, "B tile exceeds a buffer");
  static_assert((EB * es) % 16 == 0, "q part of a B tile must start 16-byte aligned");
};

// Row classes: greedy, small top-k (candidate lists), unfiltered, a top-k
// above the list limit (general path), top-p alone (grid-wide passes).
enum { UT_GREEDY = 0, UT_TOPK = 1, UT_DENSE = 2, UT_GENERAL = 3, UT_TOPP = 4 };
constexpr int kClasses = 5;

// Error bits of CallWords::error (OR-ed during a call, kept until the call
// after next starts).
enum {
  ERR_STATE_WAIT = 1,      // a B tile gave up waiting for its unit's state
  ERR_COPY_WAIT = 2,       // a tile's bulk copy did not complete
  ERR_RECORD_WAIT = 4,     // a settle or finalize gave up waiting for records
  ERR_ORDER_WAIT = 8,      // a CTA gave up waiting for the row order
  ERR_BARRIER = 16         // a CTA gave up waiting at a grid barrier of the top-p passes
};

// The counters of one call.  Calls alternate between two sets: call n
// counts in set n & 1 and zeroes set (n + 1) & 1 for the call after it, so
// no call has to wait at its end for the last CTA to reset anything.
struct CallWords {
  uint32_t gnext;         // next general-path unit
  uint32_t commit_next;   // fused commit: next copy job
  uint32_t done_count;    // fused commit: rows finalized so far (entries of the done queue)
  uint32_t bar;           // top-p passes: arrivals at the grid barriers
  uint32_t tp_more;       // top-p passes: bit L set when refinement level L is needed
  uint32_t error;         // ERR_* bits of the waits that gave up
  uint32_t pad[2];
};
static_assert(sizeof(CallWords) == 32, "call words");

struct WsHeader {
  unsigned long long arrivals;  // CTAs that have entered a call on this workspace, over all calls
  uint32_t order_tag;     // the row order in the workspace is this call's (large batches)
  uint32_t pad_a[2];
  uint32_t inject;        // test hooks: bit 0 makes the finalize of row 0 wait for a tag nothing
                          // writes; bit 1 makes CTA 0 reach the first grid barrier of the top-p
                          // passes 1.5 s late, after the others' wait has given up
  uint32_t last_set;      // the counter set of the last call to start (written by its CTA 0)
  uint32_t pad_b;
  CallWords call[2];      // by the parity of the call's number
  uint32_t n_class[kClasses];   // rows per class (large batches)
  uint32_t pad[30];
  uint32_t epoch;         // tag of the last call to start (written by its CTA 0)
  uint32_t pad1[4];
};
static_assert(sizeof(WsHeader) == 256, "workspace header");
static_assert(offsetof(WsHeader, inject) == 20, "test hook word");
static_assert(offsetof(WsHeader, last_set) == 24, "last call's counter set");
static_assert(offsetof(WsHeader, call) == 32, "call words");
static_assert(offsetof(WsHeader, epoch) == 236, "epoch word");

// The parity of the running call's number, set by each CTA as it enters the
// verify kernel; selects the call's counter set.
static __shared__ uint32_t s_call_parity;

// General-path group: the CTA's first kThreads (256) threads run the
// group-wide code on a named barrier of their own.
__device__ __forceinline__ int ctid() { return (int)(threadIdx.x & 255u); }
__device__ __forceinline__ void csync() {
  asm volatile("bar.sync %0, 256;" ::"r"(1 + (int)(threadIdx.x >> 8)) : "memory");
}

// Records pass between warps without fences: every 64-bit word carries the
// call's tag in its high half and one 32-bit value in its low half, and a
// reader takes a word as written once it carries the current tag (aligned
// 64-bit accesses are single-copy atomic).
//   A record, per (unit, A tile), 16 words:
//     greedy / unfiltered: [0] tile max (NaN when the tile holds a NaN, the
//       timeout NaN when the tile's copy gave up), [1] first index of the
//       tile max (greedy), [2] sum of exp2((l - m) c) relative to the tile
//       max, [3..7] level-1 race of the tile's blocks relative to the tile
//       max (s1, t1, s2, t2, v1; bonus positions);
//     small top-k: [2j] order key and [2j + 1] tile-local index of one of
//       the tile's 8 largest entries in the total order (j < 8; the
//       smallest at j = 7 when there are 8; key 0 = none), with the flags
//       kListNaN / kListPartial / kListTimeout in word 1.
//   B record, per (unit, B tile), 8 words: [0] alpha (the timeout NaN when
//     the tile gave up), [1..5] level-1 race of the residual.
//   Unit state of a drafted unfiltered unit, 8 words: see UnitState.
//   Unit record of a settled unit, 8 words: see UnitRecord.
constexpr int kRecWords = 16;
constexpr int kBRecWords = 8;
constexpr int kStateWords = 8;
constexpr int kURecWords = 8;
constexpr int kList = 8;                   // entries listed per top-k A tile
constexpr uint32_t kListNaN = 1u << 31;    // the tile holds a NaN
constexpr uint32_t kListPartial = 1u << 30;   // the list may miss entries above its last (re-scan the tile)
constexpr uint32_t kListTimeout = 1u << 29;   // the tile's copy gave up
constexpr uint32_t kListIdx = (1u << 29) - 1u;
constexpr uint32_t kTimeoutNaN = 0x7fbadbadu;  // a quiet NaN marking a tile that gave up
typedef unsigned long long u64;
__device__ __forceinline__ u64 tagw(uint32_t tag, uint32_t v) { return ((u64)tag << 32) | v; }
__device__ __forceinline__ u64 tagf(uint32_t tag, float v) { return tagw(tag, __float_as_uint(v)); }
__device__ __forceinline__ bool tag_ok(u64 w, uint32_t tag) { return (uint32_t)(w >> 32) == tag; }
__device__ __forceinline__ float wf(u64 w) { return __uint_as_float((uint32_t)w); }
__device__ __forceinline__ uint32_t wu(u64 w) { return (uint32_t)w; }

struct UnitState {        // what the B tiles of a drafted unfiltered unit need
  float m, invZ, lnZ, lp_x;
  int32_t accept;
  uint32_t flags;         // BAD_TOKEN | MARGIN_ACCEPT | BAD_PARAM | TIMEOUT of this unit
  uint32_t invalid;       // the unit is invalid (NaN or timeout); its record is already written
  int32_t am;
};

struct UnitRecord {       // one per unit, published as kURecWords tagged words
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
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Per-unit record counts, sized for the logit dtype with more tiles (fp32).
__host__ __device__ inline int max_nta(int V) { return ceil_div(V, Geo<false>::EA); }
__host__ __device__ inline int max_ntb(int V) { return ceil_div(V, Geo<false>::EB); }

struct Layout {
  size_t row_ticket, ucnt, rec, brec, ust, urec, order, done, tp, total;
};

// Scratch of the top-p passes, per top-p unit (u64 words, zeroed by every
// call that has top-p rows): 32 unit words (summary and threshold states),
// the mass histogram of 256 bins, then kTpLevels refinement histograms.
constexpr int kTpBins = 256;
constexpr int kTpLevels = 4;             // 8 key bits a level: two for bf16 keys, four for fp32
constexpr int kTpUnitWords = 32;
constexpr int kTpStride = kTpUnitWords + kTpBins * (1 + kTpLevels);
static_assert(kTpStride % 2 == 0, "the top-p scratch is zeroed in 16-byte stores");

__host__ __device__ inline Layout ws_layout(int B, int k, int V) {
  const size_t U = (size_t)B * (k + 1);
  Layout L;
  size_t off = sizeof(WsHeader);
  L.row_ticket = off; off = align_up(off + (size_t)B * 4, 256);
  L.ucnt = off; off = align_up(off + U * 2 * 4, 256);
  L.rec = off; off = align_up(off + U * max_nta(V) * kRecWords * 8, 256);
  L.brec = off; off = align_up(off + U * max_ntb(V) * kBRecWords * 8, 256);
  L.ust = off; off = align_up(off + U * kStateWords * 8, 256);
  L.urec = off; off = align_up(off + U * kURecWords * 8, 256);
  L.order = off; off = align_up(off + (size_t)B * 4, 256);
  L.done = off; off = align_up(off + (size_t)B * 8, 256);
  L.tp = off; off = align_up(off + U * kTpStride * 8, 256);
  L.total = off;
  return L;
}

// The commit fused into the verify launch (spec_verify_commit): each row's
// accepted state, gathered as in spec_commit once the row is finalized.
constexpr long long kJobBytes = 64 * 1024;   // fused commit: bytes of one copy job

struct FusedCommit {
  const unsigned char* vrec;    // verify_rec [L, B, S, H, Dk, Dv] fp32 (null: none)
  const unsigned char* vconv;   // verify_conv [L, B, S, W, C] 16-bit (null: none)
  const int32_t* slot;          // cache_slot [B] (null: slot r)
  unsigned char* crec;          // cache_rec [L, slots, H, Dk, Dv]
  unsigned char* cconv;         // cache_conv [L, slots, W, C]
  long long rec_bytes, conv_bytes;   // bytes of one (layer, row, state) blob
  int L, slots;
  int rec_jobs, conv_jobs;      // copy jobs per blob
  int bulk;                     // pointers and blob sizes 16-byte aligned: bulk copies through shared memory
  int on;
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
  uint32_t* row_ticket;
  uint32_t* ucnt;         // per unit: tiles done, A pass [U] then B pass [U]
  u64* rec;               // A records
  u64* brec;              // B records
  u64* ust;               // unit states of drafted unfiltered units
  u64* urec;              // unit records
  uint32_t* order;        // rows by class (batches above the shared-memory order limit)
  uint32_t key0, key1;
  uint32_t row_base;      // row r of this call draws as row row_base + r of the stream
  int B, k, V, U;
  int NTA, NTB;           // record strides per unit: A tiles, B tiles
  int n_ctas;             // CTAs of the kernel
  int n_settle;           // settle CTAs: blocks 0, stride, 2 stride, ... (n_settle of them)
  int settle_stride;
  int global_order;       // the row order lives in the workspace
  int vec_logits;
  int vec_q;
  int l2_stage;           // the logits fit L2 with room to spare: top-p rows are staged there at entry
  u64* done;              // fused commit: finalized rows in order, tagged (row << 5 | accept_len)
  u64* tp;                // top-p passes: per-unit scratch (kTpStride words per top-p unit)
  u64* desc;              // draft sampling: per-unit kept-set descriptors (null: not written)
  uint32_t race_stream;   // Philox stream word of the entries' race uniforms (blocks: the next one)
  uint32_t pos_base;      // added to a unit's position in the Philox counters
  FusedCommit fc;
};

// The running call's counters (in the verify kernel, after its prologue).
__device__ __forceinline__ CallWords& cur(const Args& A) { return A.ws->call[s_call_parity]; }


// Timeline stamps (global timer, ns) of an instrumented build compiled with
// SPEC_TIMELINE; empty otherwise.  Slots: per CTA start and end, per stream
// warp first data and end, per settle warp end, per unit the last A ticket,
// settle-A start and end, last B ticket, settle-B start and end, per row the
// finalize, per item its end.
enum {
  TL_CTA_START = 0, TL_CTA_END = 160, TL_FIRST_DATA = 320, TL_STREAM_END = 2368, TL_SETTLE_END = 4416,
  TL_ATICK = 4672, TL_SA_START = 6720, TL_SA_END = 8768, TL_BTICK = 10816, TL_SB_START = 12864,
  TL_SB_END = 14912, TL_FINAL = 16960, TL_ITEM = 17984, TL_PHASE = 34368, TL_ISTART = 34368 + 2048 * 8,
  TL_IWARP = TL_ISTART + 16384, TL_ISTATE = TL_IWARP + 16384, TL_SUB = TL_ISTATE + 16384,
  TL_TP = TL_SUB + 2048 * 8, TL_TP_WARP = TL_TP + 16, TL_SIZE = TL_TP_WARP + 8 * 2048
};
#ifdef SPEC_TIMELINE
static __device__ unsigned long long g_tl[TL_SIZE];
__device__ __forceinline__ void tl_stamp(int slot, int i, int lim) {
  if (i >= 0 && i < lim) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_tl[slot + i] = t;
  }
}
#define TL(slot, i, lim) tl_stamp((slot), (i), (lim))
// phase p (0..7) of the settle of unit u
#define TLP(u, p) do { if ((threadIdx.x & 31) == 0 && (u) < 2048) tl_stamp(TL_PHASE + (u) * 8 + (p), 0, 1); } while (0)
#define TLS(u, p) do { if ((threadIdx.x & 31) == 0 && (u) < 2048) tl_stamp(TL_SUB + (u) * 8 + (p), 0, 1); } while (0)
#else
#define TL(slot, i, lim) ((void)0)
#define TLP(u, p) ((void)0)
#define TLS(u, p) ((void)0)
#endif

// The row index the random streams are keyed by.
__device__ __forceinline__ uint32_t srow(const Args& A, int row) { return A.row_base + (uint32_t)row; }

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

__device__ __forceinline__ RowCfg classify(const spec_params_t& prm, int V) {
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
  else if (r.K > 0 && r.K <= kTopkSmall && max_nta(V) * kList <= kMaxListCand) r.type = UT_TOPK;
  else if (r.K == 0 && r.P >= 1.0f) r.type = UT_DENSE;
  else if (r.K == 0) r.type = UT_TOPP;
  else r.type = UT_GENERAL;
  return r;
}

// Row configuration packed in 16 bytes (kept in shared memory per row).
struct RowPack {
  float c, invT, P;
  uint32_t tk;            // type | bad_param << 3 | K << 8
};
__device__ __forceinline__ RowPack pack_cfg(const RowCfg& r) {
  RowPack p;
  p.c = r.c;
  p.invT = r.invT;
  p.P = r.P;
  p.tk = (uint32_t)r.type | (r.bad_param ? 8u : 0u) | ((uint32_t)r.K << 8);
  return p;
}
__device__ __forceinline__ RowCfg unpack_cfg(const RowPack& p) {
  RowCfg r;
  r.c = p.c;
  r.invT = p.invT;
  r.P = p.P;
  r.type = (int)(p.tk & 7u);
  r.bad_param = (p.tk & 8u) != 0;
  r.K = (int)(p.tk >> 8);
  return r;
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
    const float4 a = __ldcg(reinterpret_cast<const float4*>(p + e0));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(p + e0 + 4));
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
// One warp, lane j reading unit j's record (k + 1 <= 32; bounded wait for
// its tag): the accepted prefix ends at the first rejected draft; its tokens
// are the drafts, then the draw of the first rejected unit (or the bonus
// draw).  A row whose records did not all arrive, or that holds a unit that
// gave up a wait, is written as invalid with SPEC_F_TIMEOUT.
// Fused commit: append a finalized row to the done queue (lane 0), after
// its outputs (the commit ORs SPEC_F_BAD_IDX into the row's flags later).
__device__ __forceinline__ void enqueue_done(const Args& A, int row, int acc_len, uint32_t tag) {
  if ((threadIdx.x & 31) == 0) {
    __threadfence();
    const uint32_t i = atomicAdd(&cur(A).done_count, 1u);
    __stcg(A.done + i, tagw(tag, ((uint32_t)row << 5) | (uint32_t)acc_len));
  }
}

// w[] holds words 0..6 of unit `lane` of the row as loaded before the
// row's ticket was taken; they are used if they all carry the tag already.
static __device__ __forceinline__ void finalize_row(const Args& A, int row, uint32_t tag, const u64 (&w0)[7]) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int k = A.k;
  const u64* R = A.urec + ((size_t)row * (k + 1) + lane) * kURecWords;
  // test hook: row 0 waits for a tag that no record carries
  const uint32_t want = (row == 0 && (__ldcg(&A.ws->inject) & 1u) != 0u) ? (tag ^ 0x80000000u) : tag;
  u64 w[7];
#pragma unroll
  for (int i = 0; i < 7; ++i) w[i] = w0[i];
  long long spins = 0;
  bool timed_out = false;
  for (bool first = true;; first = false) {
    bool ok = true;
    if (lane <= k) {
#pragma unroll
      for (int i = 0; i < 7; ++i) {
        if (!first) w[i] = __ldcg(R + i);
        ok = ok && tag_ok(w[i], want);
      }
    }
    if (__all_sync(full, ok)) break;
    if (++spins > kSpinLimit) {
      if (lane == 0) atomicOr(&cur(A).error, (uint32_t)ERR_RECORD_WAIT);
      timed_out = true;
      break;
    }
    __nanosleep(64);
  }
  const uint32_t f = wu(w[0]);
  const bool acc = wu(w[1]) != 0u;
  const float lp_x = wf(w[2]), alpha = wf(w[3]);
  const int32_t y = (int32_t)wu(w[4]);
  const float lp_y = wf(w[5]);
  const uint32_t draw_flags = wu(w[6]);
  uint32_t uflags = __reduce_or_sync(
      full, lane <= k ? (f & (SPEC_F_NAN | SPEC_F_BAD_PARAM | SPEC_F_BAD_TOKEN | SPEC_F_MARGIN_TOPP | SPEC_F_TIMEOUT)) : 0u);
  int32_t* tok = A.tokens + (size_t)row * (k + 1);
  float* lp = A.logprobs + (size_t)row * (k + 1);
  if (timed_out || (uflags & (SPEC_F_NAN | SPEC_F_TIMEOUT))) {
    const uint32_t rf = timed_out || (uflags & SPEC_F_TIMEOUT) ? (SPEC_F_TIMEOUT | (uflags & SPEC_F_NAN))
                                                                : SPEC_F_NAN;
    if (lane <= k) {
      tok[lane] = -1;
      lp[lane] = 0.f;
    }
    if (lane < k) A.alpha[(size_t)row * k + lane] = 0.f;
    if (lane == 0) {
      A.accept_len[row] = 0;
      A.flags[row] = rf;
    }
    if (A.fc.on) enqueue_done(A, row, 0, tag);
    return;
  }
  const unsigned rej = __ballot_sync(full, lane < k && !acc);
  const int a = rej ? __ffs(rej) - 1 : k;
  uflags |= __reduce_or_sync(full, (lane < k && lane <= a) ? (f & SPEC_F_MARGIN_ACCEPT) : 0u);
  uflags |= __shfl_sync(full, draw_flags, a);
  if (lane < a) {
    tok[lane] = A.drafts[(size_t)row * k + lane];
    lp[lane] = lp_x;
  } else if (lane == a) {
    tok[lane] = y;
    lp[lane] = lp_y;
  } else if (lane <= k) {
    tok[lane] = -1;
    lp[lane] = 0.f;
  }
  if (lane < k) A.alpha[(size_t)row * k + lane] = alpha;
  if (lane == 0) {
    A.accept_len[row] = a + 1;
    A.flags[row] = uflags;
  }
  if (A.fc.on) enqueue_done(A, row, a + 1, tag);
}

// One warp (converged): lanes 0..7 publish the unit's record (lane 0's
// `rec`) as tagged words and lane 0 takes the row's ticket (relaxed: the
// finaliser waits for the tags, not for an ordering); the warp whose unit is
// the row's last finalizes the row.
static __device__ __noinline__ void commit_record(const Args& A, uint32_t tag, int u, int row, UnitRecord rec) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const uint32_t v = lane_word8(lane, __shfl_sync(full, rec.flags, 0), __shfl_sync(full, (uint32_t)rec.accept, 0),
                                __shfl_sync(full, __float_as_uint(rec.lp_x), 0),
                                __shfl_sync(full, __float_as_uint(rec.alpha), 0), __shfl_sync(full, (uint32_t)rec.y, 0),
                                __shfl_sync(full, __float_as_uint(rec.lp_y), 0), __shfl_sync(full, rec.draw_flags, 0),
                                0u);
  if (lane < kURecWords) __stcg(A.urec + (size_t)u * kURecWords + lane, tagw(tag, v));
  // the row's records, in flight with the ticket: the last unit usually
  // finds the others' already written and finalizes without another load
  u64 w[7];
  const int ul = row * (A.k + 1) + (lane <= A.k ? lane : 0);
#pragma unroll
  for (int i = 0; i < 7; ++i) w[i] = __ldcg(A.urec + (size_t)ul * kURecWords + i);
  uint32_t old = 0u;
  if (lane == 0) old = atomicAdd(&A.row_ticket[row], 1u);
  old = __shfl_sync(full, old, 0);
  if (old == (uint32_t)A.k) {
    finalize_row(A, row, tag, w);
    if (lane == 0) TL(TL_FINAL, row, 1024);
    if (lane == 0) A.row_ticket[row] = 0;   // leave the workspace clean for the next call
  }
  __syncwarp();
}

// Draft sampling (spec_draft_sample): the settled unit's kept set and
// normaliser, for the kernel that writes q afterwards.  Tagged words:
// [0] mode, [1] m, [2] 1 / Z_S, [3] threshold order key (full 32-bit key),
// [4] threshold index (the last kept entry at that key) or the argmax.
enum { DESC_ALL = 1, DESC_THRESH = 2, DESC_GREEDY = 3 };
constexpr int kDescWords = 8;
__device__ __forceinline__ void publish_desc(const Args& A, uint32_t tag, int u, uint32_t mode, float m, float invZ,
                                             uint32_t tkey, uint32_t tidx) {
  if (A.desc == nullptr) return;
  const int lane = threadIdx.x & 31;
  const uint32_t v = lane == 0 ? mode
                   : lane == 1 ? __float_as_uint(m)
                   : lane == 2 ? __float_as_uint(invZ)
                   : lane == 3 ? tkey
                               : tidx;
  if (lane < 5) __stcg(A.desc + (size_t)u * kDescWords + lane, tagw(tag, v));
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

// The kept set is a prefix of the total order: entries with a larger key,
// and the entries at the threshold key up to index tidx.
struct Thresh {
  uint32_t tkey;
  uint32_t tidx;
};
__device__ __forceinline__ bool kept(const Thresh& t, uint32_t key, uint32_t v) {
  return key > t.tkey || (key == t.tkey && v <= t.tidx);
}

// The accept uniform u_j of draft `pos` in row `row`: Philox counter
// (0, pos, row, 0), word 0.
__device__ __forceinline__ float accept_uniform(const Args& A, int row, int pos) {
  const uint4 w = philox4x32_10(make_uint4(0u, (uint32_t)pos + A.pos_base, srow(A, row), 0u), A.key0, A.key1);
  return uniform_of(w.x);
}

// Accept test of the draft at (row, pos): accept iff u*q(x) < p(x), with the
// sign of u*q - p taken exactly by one fma.  p(x) = exp((l_x - m) / T) / Z
// when x is kept (kept_th == nullptr keeps everything); greedy: p(x) = 1 if
// x is the argmax, else 0.
// The decision itself, for a draft whose x, validity, l_x and q(x) are in ai.
static __device__ __noinline__ AcceptInfo accept_decide(const Args& A, int row, int pos, AcceptInfo ai, bool greedy,
                                                        int am, float m, float c, float Zs, const Thresh* kept_th) {
  ai.px = 0.f;
  if (ai.valid) {
    if (greedy) {
      ai.px = (ai.x == am) ? 1.0f : 0.0f;
    } else {
      const bool in = kept_th ? kept(*kept_th, okey(ai.lx), (uint32_t)ai.x) : true;
      ai.px = in ? ex2((ai.lx - m) * c) / Zs : 0.0f;
    }
  }
  const float u = accept_uniform(A, row, pos);
  const float d = fmaf(u, ai.qx, -ai.px);
  ai.accept = d < 0.0f;
  ai.margin = (ai.px > 0.0f && ai.px < 1.0f && fabsf(d) < kMargin);
  return ai;
}
// x, l_x and q(x) of the draft at (row, pos) (ai.valid: x in [0, V)).
__device__ __forceinline__ AcceptInfo accept_load(const Args& A, int row, int pos, bool bf16, int x) {
  AcceptInfo ai;
  ai.x = x;
  ai.valid = x >= 0 && x < A.V;
  ai.lx = 0.f;
  ai.qx = 0.f;
  ai.px = 0.f;
  ai.accept = false;
  ai.margin = false;
  if (ai.valid) {
    ai.lx = load_logit(A, bf16, ((size_t)row * (A.k + 1) + pos) * (size_t)A.V + x);
    ai.qx = A.q[((size_t)row * A.k + pos) * (size_t)A.V + x];
  }
  return ai;
}
static __device__ __noinline__ AcceptInfo accept_test(const Args& A, int row, int pos, bool bf16, bool greedy, int am,
                                                      float m, float c, float Zs, const Thresh* kept_th) {
  const AcceptInfo ai = accept_load(A, row, pos, bf16, A.drafts[(size_t)row * A.k + pos]);
  return accept_decide(A, row, pos, ai, greedy, am, m, c, Zs, kept_th);
}

// Race uniform words.  Entry v at position pos: counter (v >> 2, pos, row,
// 1), word v & 3.  Block b (level 1): counter (b >> 2, pos, row, 2), word b & 3.
__device__ __forceinline__ uint32_t race_word(const Args& A, int row, int pos, uint32_t v) {
  const uint4 w = philox4x32_10(make_uint4(v >> 2, (uint32_t)pos + A.pos_base, srow(A, row), A.race_stream),
                                A.key0, A.key1);
  return word_of(w, v & 3);
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
  const uint4 w = philox4x32_10(make_uint4(b >> 2, (uint32_t)pos + A.pos_base, srow(A, row), A.race_stream + 1u),
                                A.key0, A.key1);
  return word_of(w, b & 3);
}

enum { RW_BONUS = 0, RW_RESIDUAL = 1, RW_P = 2 };

// Weights of the 8 entries of group g from its logits v[] (and q[] for
// RW_RESIDUAL): RW_BONUS / RW_P use exp2((l - m) c) (margin weight: the
// same), RW_RESIDUAL uses max(p - q, 0) with p = exp2((l - m) c) * invZ
// (margin weight p + q).  Entries outside the kept set (th) or past V weigh
// 0.  Returns in w[] and tq[] = margin - w.
__device__ __forceinline__ void group_weights(const Args& A, int g, const float v[8], const float qv[8], float m,
                                              float c, float invZ, int mode, const Thresh* th, float w[8],
                                              float tq[8]) {
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
  group_weights(A, g, v, qv, m, c, invZ, mode, th, w, tq);
}

// Level 2: the race among the entries of block b, run by one warp (the
// result is in every lane).  The group's two Philox blocks are computed
// while its loads are in flight.  *ly (if given) receives the logit of the
// winning entry.  kInline runs race_consider's steps unrolled and inline:
// the same race, without the latency of an out-of-line update per entry,
// for a warp that runs it alone (the top-p settles, one unit an SM); where
// settles share SMs and are throughput-bound, the rolled loop's smaller
// code and out-of-line updates are faster.
template <bool kBF16, bool kInline = false>
__device__ __noinline__ Race race_in_block(const Args& A, int row, int pos, uint32_t b, float m, float c, float invZ,
                                           int mode, const Thresh* th, float* ly = nullptr) {
  const int lane = threadIdx.x & 31;
  const size_t lrow = ((size_t)row * (A.k + 1) + pos) * (size_t)A.V;
  const size_t qrow = ((size_t)row * A.k + pos) * (size_t)A.V;
  const int G = (A.V + 7) / 8;
  Race r;
  race_init(r);
  if (b >= (uint32_t)((A.V + kRaceBlock - 1) / kRaceBlock)) return r;   // no block won (all weights 0)
  const int g = (int)b * (kRaceBlock / 8) + lane;
  float v[8], qv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[j] = 0.f;
    qv[j] = 0.f;
  }
  if (g < G) {
    load_group<kBF16>(A, lrow, g, true, v);
    if (mode == RW_RESIDUAL) load_q8(A, qrow, g * 8, qv);
    // the Philox blocks of entries 8g..8g+3 and 8g+4..8g+7
    const uint32_t blk = (uint32_t)g * 2u;
    const uint32_t cp = (uint32_t)pos + A.pos_base;
    const uint4 p0 = philox4x32_10(make_uint4(blk, cp, srow(A, row), A.race_stream), A.key0, A.key1);
    const uint4 p1 = philox4x32_10(make_uint4(blk + 1u, cp, srow(A, row), A.race_stream), A.key0, A.key1);
    float w[8], tq[8];
    group_weights(A, g, v, qv, m, c, invZ, mode, th, w, tq);
    if constexpr (kInline) {
      // zero weights skip the score (its division would take the slow path)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float om = one_minus_uniform_of(j < 4 ? word_of(p0, j) : word_of(p1, j - 4));
        if (w[j] > 0.f && w[j] >= r.s1lo * om) {
          float sj, uj;
          race_score(w[j], tq[j], om, sj, uj);
          race_apply(r, sj, uj, (uint32_t)(g * 8 + j));
        }
      }
    } else {
      // one race step per entry, in a rolled loop (small code)
#pragma unroll 1
      for (int j = 0; j < 8; ++j) {
        float wj = w[0], tj = tq[0];
        uint32_t pj = p0.x;
#pragma unroll
        for (int t = 1; t < 8; ++t)
          if (j == t) {
            wj = w[t];
            tj = tq[t];
            pj = t < 4 ? word_of(p0, t) : word_of(p1, t - 4);
          }
        if (wj > 0.f) race_consider(r, wj, tj, (uint32_t)(g * 8 + j), pj);
      }
    }
  }
  warp_race_merge(r);
  if (ly != nullptr && r.s1 >= 0.f) {
    // the winner's lane holds its logit
    const int src = (int)(r.v1 >> 3) - (int)b * (kRaceBlock / 8);
    const uint32_t jj = r.v1 & 7u;
    float lv = v[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) lv = jj == (uint32_t)j ? v[j] : lv;
    *ly = __shfl_sync(0xffffffffu, lv, src & 31);
  }
  return r;
}

__device__ __forceinline__ void race_scale(Race& r, float sc) {
  if (r.s1 >= 0.f) r.s1 *= sc;
  if (r.s2 >= 0.f) r.s2 *= sc;
  r.t1 *= sc;
  r.t2 *= sc;
}

// ---------------------------------------------------------------------------
// Launcher.
// ---------------------------------------------------------------------------
template <bool kBF16>
int launch_verify(const Args& A, cudaStream_t stream);

}  // namespace specv
