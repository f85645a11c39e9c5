// Device helpers shared by the verify and commit kernels (sm_103a).
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMargin = 1e-6f;

// ---------------------------------------------------------------------------
// Philox4x32-10, written from J. K. Salmon et al., "Parallel random numbers:
// as easy as 1, 2, 3" (SC'11), section 3: each round multiplies counter words
// 0 and 2 by the two Philox-4x32 multipliers, permutes
// (X0,X1,X2,X3) -> (hi(M1 X2)^X1^K0, lo(M1 X2), hi(M0 X0)^X3^K1, lo(M0 X0)),
// and bumps the key by the Weyl constants; ten rounds.
// ---------------------------------------------------------------------------
// Out of line with a rolled loop: the verify kernel runs it from many
// places, and a small body keeps the instruction stream short.
static __device__ __noinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll 1
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ uint32_t word_of(const uint4& w, int i) {
  return i == 0 ? w.x : (i == 1 ? w.y : (i == 2 ? w.z : w.w));
}

// U = ((w >> 9) + 1/2) * 2^-23 and 1 - U, both exact: 1 + m*2^-23 is built
// from the bits and (1 - 2^-24) subtracted (an exact subtraction, Sterbenz).
__device__ __forceinline__ float uniform_of(uint32_t w) {
  return __uint_as_float(0x3f800000u | (w >> 9)) - __uint_as_float(0x3f7fffffu);
}
__device__ __forceinline__ float one_minus_uniform_of(uint32_t w) {
  return __uint_as_float(0x3f800000u | ((w >> 9) ^ 0x7fffffu)) - __uint_as_float(0x3f7fffffu);
}

// ---------------------------------------------------------------------------
// Asynchronous global->shared copies (16 bytes per instruction, L1 bypassed).
// Completion is awaited with cp.async.wait_group, a hardware wait.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------------------
// Bulk asynchronous global->shared copies completed on an mbarrier (the
// copy engine moves the bytes; the issuing thread only posts the request).
// Addresses and sizes are multiples of 16 bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same with an L2 cache policy (createpolicy), e.g. evict-first for data
// read once, so streamed inputs do not push reused lines out of L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, unsigned long long* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, unsigned long long* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------------------
// Device-scope load-acquire and store-release (one instruction instead of a
// full fence plus a relaxed access).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t load_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// A relaxed device-scope load that the compiler may not merge with another
// (for polling a word other warps update).
__device__ __forceinline__ uint32_t load_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void store_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Floating point helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Warp-wide maximum that propagates NaN (one instruction on sm_100 and later).
__device__ __forceinline__ float warp_max_nan(float v) {
  float r;
  asm("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Packed bf16x2 maximum that propagates NaN.
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Order-preserving key of a float: larger value -> larger key; -0 and +0 map
// to the same key.  NaN never reaches it (rows with NaN are rejected first).
__device__ __forceinline__ uint32_t okey(float f) {
  uint32_t b = __float_as_uint(f);
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_okey(uint32_t k) {
  const uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(b);
}

// 64-bit total-order key: (value key, then smaller index first).
__device__ __forceinline__ unsigned long long key64(uint32_t vkey, uint32_t idx) {
  return ((unsigned long long)vkey << 32) | (unsigned long long)(0xffffffffu - idx);
}
__device__ __forceinline__ uint32_t key64_idx(unsigned long long k) {
  return 0xffffffffu - (uint32_t)(k & 0xffffffffull);
}

// Word `lane` of eight (lanes 8..31 get a0): a chain of selects, so a warp
// writing a small record does not branch per lane.
__device__ __forceinline__ uint32_t lane_word8(int lane, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
  uint32_t v = a0;
  v = lane == 1 ? a1 : v;
  v = lane == 2 ? a2 : v;
  v = lane == 3 ? a3 : v;
  v = lane == 4 ? a4 : v;
  v = lane == 5 ? a5 : v;
  v = lane == 6 ? a6 : v;
  v = lane == 7 ? a7 : v;
  return v;
}

// ---------------------------------------------------------------------------
// Warp and block reductions with a fixed combination order (deterministic).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ uint32_t warp_min_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Transposed warp sum of N (a power of two <= 32) values per lane: lane L
// returns the sum over all lanes of their value number L mod N.  A butterfly:
// at each level a lane keeps the half of its values its lane bit selects
// and adds its partner's copy of them (N - 1 shuffles), then the groups of
// N lanes are summed.  t is overwritten.  The combination order is fixed.
template <int N>
__device__ __forceinline__ float warp_transpose_sum(float (&t)[N]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int h = N / 2; h >= 1; h >>= 1) {
    const bool up = (lane & h) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? t[i] : t[i + h];
      const float keep = up ? t[i + h] : t[i];
      t[i] = keep + __shfl_xor_sync(0xffffffffu, send, h);
    }
  }
  float r = t[0];
#pragma unroll
  for (int o = N; o < 32; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

// ---------------------------------------------------------------------------
// Exponential-race state: best score s1 (entry v1) and runner-up s2, with the
// margin weights t = (p + q) / E of both.
// ---------------------------------------------------------------------------
struct Race {
  float s1, t1, s2, t2, s1lo;
  uint32_t v1;
};

// Start bringing the line holding *p into L2 (no result, no fault on a
// valid address).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// The GPU's global timer, in nanoseconds.
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Start bringing `bytes` (a multiple of 16, from a 16-byte aligned address)
// into L2 with the copy engine.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void race_init(Race& r) {
  r.s1 = -1.0f;
  r.t1 = 0.0f;
  r.s2 = -1.0f;
  r.t2 = 0.0f;
  r.s1lo = 0.0f;
  r.v1 = 0xffffffffu;
}

// Score s = w / E with E = -ln U.  Because E >= 1 - U, an entry with
// w < s1 * (1 - 2^-20) * (1 - U) cannot beat the current best and needs no
// logarithm; the factor (1 - 2^-20) absorbs the rounding of the test itself.
__device__ __forceinline__ void race_apply(Race& r, float s, float t, uint32_t v) {
  if (s > r.s1 || (s == r.s1 && v < r.v1)) {
    if (v != r.v1) {
      r.s2 = r.s1;
      r.t2 = r.t1;
    }
    r.s1 = s;
    r.t1 = t;
    r.v1 = v;
    r.s1lo = s * 0.99999905f;
  } else if (v != r.v1 && s > r.s2) {
    r.s2 = s;
    r.t2 = t;
  }
}
// The score and margin weight of an entry of weight w: s = w / E, t = (w + tq) / E.
__device__ __forceinline__ void race_score(float w, float tq, float om, float& s, float& t) {
  const float E = -log1pf(-om);
  s = w / E;
  t = (w + tq) / E;
}
static __device__ __noinline__ Race race_update(Race r, float w, float tq, uint32_t v, float om) {
  float s, t;
  race_score(w, tq, om, s, t);
  race_apply(r, s, t, v);
  return r;
}
// The cheap bound test inline, the logarithm out of line (the state stays
// in registers either way).
__device__ __forceinline__ void race_consider(Race& r, float w, float tq, uint32_t v, uint32_t word) {
  const float om = one_minus_uniform_of(word);
  if (w >= r.s1lo * om) r = race_update(r, w, tq, v, om);
}
__device__ __forceinline__ void race_merge(Race& a, const Race& b) {
  if (b.v1 == a.v1) {
    if (b.s2 > a.s2) { a.s2 = b.s2; a.t2 = b.t2; }
    return;
  }
  const bool b_wins = (b.s1 > a.s1) || (b.s1 == a.s1 && b.v1 < a.v1);
  if (b_wins) {
    // old a.s1 competes with b.s2 for second place
    float s2 = a.s1, t2 = a.t1;
    if (b.s2 > s2) { s2 = b.s2; t2 = b.t2; }
    a.s1 = b.s1; a.t1 = b.t1; a.v1 = b.v1; a.s2 = s2; a.t2 = t2;
  } else {
    if (b.s1 > a.s2) { a.s2 = b.s1; a.t2 = b.t1; }
  }
  a.s1lo = a.s1 * 0.99999905f;
}

// Warp merge by reductions: the winner is the largest score, ties to the
// smaller entry; the runner-up is the largest of the other entries' best
// scores and the winning entry's second score (a lane that raced the winning
// entry too contributes its second).  Scores are positive, so their float
// bits order like unsigned integers.  Every lane gets the result; it does not
// depend on the lanes' order (ties of the runner-up go to the lowest lane).
static __device__ __noinline__ Race warp_race_merged(Race r) {
  const unsigned full = 0xffffffffu;
  const uint32_t sk = r.s1 >= 0.f ? __float_as_uint(r.s1) : 0u;
  const uint32_t top = __reduce_max_sync(full, sk);
  Race o;
  race_init(o);
  if (top == 0u) return o;
  const uint32_t vb = __reduce_max_sync(full, sk == top ? ~r.v1 : 0u);
  o.v1 = ~vb;
  const int wl = __ffs(__ballot_sync(full, sk == top && r.v1 == o.v1)) - 1;
  o.s1 = __shfl_sync(full, r.s1, wl);
  o.t1 = __shfl_sync(full, r.t1, wl);
  const bool same = r.v1 == o.v1;
  const float cs = same ? r.s2 : r.s1;
  const float ct = same ? r.t2 : r.t1;
  const uint32_t ck = cs >= 0.f ? __float_as_uint(cs) : 0u;
  const uint32_t sec = __reduce_max_sync(full, ck);
  if (sec != 0u) {
    const int sl = __ffs(__ballot_sync(full, ck == sec)) - 1;
    o.s2 = __shfl_sync(full, cs, sl);
    o.t2 = __shfl_sync(full, ct, sl);
  }
  o.s1lo = o.s1 * 0.99999905f;
  return o;
}
__device__ __forceinline__ void warp_race_merge(Race& r) { r = warp_race_merged(r); }

}  // namespace specv
