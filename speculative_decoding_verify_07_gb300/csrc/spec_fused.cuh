// spec_verify_commit, the commit phase of the fused launch (sm_103a).
//
// inclusionAI/AReno PR #550, "What does this PR do?" Phase 2 and table
// "Per-step optimizations": after the verify step the accepted position's
// recurrent and conv state of every linear-attention layer is copied into the
// row's cache slot.  Fused into the verify launch, the copy of a row starts
// as soon as the row is finalized instead of after the whole batch: every
// warp, once its verify work is done, takes copy jobs from one counter.
// Jobs are numbered in the order rows were finalized (the done queue), so
// the first jobs belong to the rows that finished first.  A job is up to
// kJobBytes of one (layer, row) blob, moved through the warp's two 8 KB
// shared-memory buffers by bulk copies (a bulk load into one buffer while
// the other is bulk-stored), or by plain loads and stores when a pointer or
// a blob size is not 16-byte aligned.  Rows outside the ranges spec_commit
// accepts get SPEC_F_BAD_IDX and are skipped, exactly as there.
#pragma once

#include "spec_common.cuh"

namespace specv {

__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The warp's earlier bulk stores have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The warp's earlier bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Lane 0: copy n bytes (a multiple of 16, 16-byte aligned ends) from global
// src to global dst through the two buffers.  False if a load's wait gave up
// (the warp then stops copying: a copy may still be landing in a buffer).
__device__ __forceinline__ bool bulk_job(const Args& A, unsigned char* dst, const unsigned char* src, long long n,
                                         unsigned char* const buf[2], unsigned long long* bar, uint32_t* par) {
  const int np = (int)((n + kSlot - 1) / kSlot);
  auto piece = [&](int p) { return (uint32_t)min((long long)kSlot, n - (long long)p * kSlot); };
  bulk_wait_read_all();   // the buffers are free
  fence_proxy_async();
  mbar_arrive_expect_tx(&bar[0], piece(0));
  bulk_g2s(buf[0], src, piece(0), &bar[0]);
  for (int p = 0; p < np; ++p) {
    const int b = p & 1;
    long long spins = 0;
    while (!mbar_try_wait(&bar[b], par[b])) {
      if (++spins > kSpinLimit) {
        atomicOr(&cur(A).error, (uint32_t)ERR_COPY_WAIT);
        return false;
      }
      if (spins > 64) __nanosleep(32);
    }
    par[b] ^= 1u;
    if (p + 1 < np) {
      bulk_wait_read_all();   // the store of piece p - 1 has read the other buffer
      mbar_arrive_expect_tx(&bar[b ^ 1], piece(p + 1));
      bulk_g2s(buf[b ^ 1], src + (long long)(p + 1) * kSlot, piece(p + 1), &bar[b ^ 1]);
    }
    fence_proxy_async();
    bulk_s2g(dst + (long long)p * kSlot, buf[b], piece(p));
    bulk_commit_group();
  }
  return true;
}

// One warp: copy jobs until none is left.  `bufs` are the warp's two
// buffers and `bar` two mbarriers it owns (initialized here).
__device__ __noinline__ void commit_phase(const Args& A, uint32_t tag, unsigned char* buf0, unsigned char* buf1,
                                          unsigned long long* bar) {
  const int lane = threadIdx.x & 31;
  const FusedCommit& F = A.fc;
  unsigned char* const buf[2] = {buf0, buf1};
  uint32_t par[2] = {0u, 0u};
  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
  }
  __syncwarp();
  const int S = A.k + 1;
  const long long jpl = (long long)F.rec_jobs + F.conv_jobs;   // jobs per (row, layer)
  const long long jpr = jpl * F.L;                              // jobs per row
  const long long total = jpr * A.B;
  long long cur_q = -1;
  int row = 0, acc = 0, slot = 0;
  bool bad = true, broken = false;
  while (!broken) {
    uint32_t jt = 0;
    if (lane == 0) jt = atomicAdd(&cur(A).commit_next, 1u);
    const long long j = (long long)__shfl_sync(0xffffffffu, jt, 0);
    if (j >= total) break;
    const long long q = j / jpr;
    const long long rem = j - q * jpr;
    if (q != cur_q) {
      // the q-th finalized row (bounded wait: every row is finalized, or the
      // verify gave up and then the wait does too)
      uint32_t w = 0;
      bool ok = false;
      if (lane == 0) {
        long long spins = 0;
        while (true) {
          const u64 d = __ldcg(A.done + q);
          if (tag_ok(d, tag)) {
            w = (uint32_t)d;
            ok = true;
            break;
          }
          if (++spins > 16ll * kSpinLimit) {
            atomicOr(&cur(A).error, (uint32_t)ERR_RECORD_WAIT);
            break;
          }
          __nanosleep(spins > 64 ? 256 : 32);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      w = __shfl_sync(0xffffffffu, w, 0);
      cur_q = q;
      row = (int)(w >> 5);
      acc = (int)(w & 31u);
      slot = F.slot ? F.slot[row] : row;
      bad = slot < 0 || slot >= F.slots;   // accept_len comes from the verify: within [0, S]
    }
    const int l = (int)(rem / jpl);
    const int jj = (int)(rem - (long long)l * jpl);
    if (bad) {
      if (lane == 0 && l == 0 && jj == 0) atomicOr(&A.flags[row], (uint32_t)SPEC_F_BAD_IDX);
      continue;
    }
    if (acc == 0) continue;
    const bool is_rec = jj < F.rec_jobs;
    const long long blob = is_rec ? F.rec_bytes : F.conv_bytes;
    const long long off = (long long)(is_rec ? jj : jj - F.rec_jobs) * kJobBytes;
    const long long n = min(kJobBytes, blob - off);
    const unsigned char* src = (is_rec ? F.vrec : F.vconv) + (((long long)l * A.B + row) * S + (acc - 1)) * blob + off;
    unsigned char* dst = (is_rec ? F.crec : F.cconv) + ((long long)l * F.slots + slot) * blob + off;
    if (F.bulk) {
      bool ok = true;
      if (lane == 0) ok = bulk_job(A, dst, src, n, buf, bar, par);
      broken = __shfl_sync(0xffffffffu, ok ? 0 : 1, 0) != 0;
    } else {
      // 2-byte units cover both the fp32 and the bf16 blobs
      const uint16_t* s2 = reinterpret_cast<const uint16_t*>(src);
      uint16_t* d2 = reinterpret_cast<uint16_t*>(dst);
      for (long long i = lane; i < n / 2; i += 32) d2[i] = s2[i];
    }
  }
  if (lane == 0 && F.bulk) bulk_wait_all();
  __syncwarp();
}

}  // namespace specv
