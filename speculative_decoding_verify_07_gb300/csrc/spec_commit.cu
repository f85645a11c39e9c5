// spec_commit: gather of each row's accepted verify state into the cache.
//
// inclusionAI/AReno PR #550, "feat(engine): MTP training loss and speculative
// decoding for bailing_v3", "What does this PR do?" Phase 2: the recurrent
// and conv caches of the linear-attention layers are stacked across layers
// and the verify forward writes one state per fed token into one shared
// verify-state buffer; table "Per-step optimizations" ("KDA caches stacked
// across layers, commit in 4 kernels").  Here the whole commit is one launch:
// a copy job is a 16 KiB chunk of one (layer, row) state blob, recurrent or
// conv, and each CTA moves one job with 128-bit streaming loads and stores.
// Rows whose accept_len is 0 are skipped; bad indices set SPEC_F_BAD_IDX.
//
// spec_commit_swap is the zero-copy variant of InfiniTensor/InfiniLM PR #588,
// "feat: add mtp draft models for speculative decoding", section 2 item 5
// (scratch state slot, O(1) slot swap on full accept, replay on partial
// accept): the last state of a row already sits in its scratch cache slot,
// so a fully accepted row only trades slot numbers, and the same kernel
// gathers the accepted state of the other rows.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/spec_verify.h"
#include "spec_host.h"

namespace specv {

constexpr int kCopyThreads = 256;
constexpr int kVecPerThread = 4;
constexpr long long kChunk = (long long)kCopyThreads * kVecPerThread * 16;   // 16 KiB

struct CommitArgs {
  const unsigned char* vrec;
  const unsigned char* vconv;
  const int32_t* accept_len;
  const int32_t* slot;
  int32_t* swap_slot;     // swap mode: each row's committed slot (traded on full accept)
  int32_t* swap_scratch;  // swap mode: each row's scratch slot
  unsigned char* crec;
  unsigned char* cconv;
  uint32_t* flags;
  long long rec_bytes;    // bytes of one (layer, row, state) recurrent blob
  long long conv_bytes;   // bytes of one conv blob
  int L, B, S, slots;
  int SV;                              // states per row in the verify buffers (S, or S - 1 in swap mode)
  int swap;
  long long rec_chunks, conv_chunks;   // chunks per blob
  int rec_vec, conv_vec;               // 16-byte vector path allowed
};

__global__ void __launch_bounds__(kCopyThreads) commit_kernel(const CommitArgs A) {
  const long long per_row = A.rec_chunks + A.conv_chunks;
  const long long job = blockIdx.x + (long long)blockIdx.y * gridDim.x;
  const long long total = (long long)A.L * A.B * per_row;
  if (job >= total) return;
  const long long lr = job / per_row;
  long long c = job - lr * per_row;
  const int l = (int)(lr / A.B);
  const int r = (int)(lr - (long long)l * A.B);

  const int acc = A.accept_len[r];
  int slot, scratch = -1;
  if (A.swap) {
    // a full accept's first job trades the slots while the row's other jobs
    // read them: either value pair passes the same range check
    slot = A.swap_slot[r];
    scratch = A.swap_scratch[r];
  } else {
    slot = A.slot ? A.slot[r] : r;
  }
  bool bad = acc < 0 || acc > A.S || slot < 0 || slot >= A.slots;
  if (A.swap) bad = bad || scratch < 0 || scratch >= A.slots || scratch == slot;
  const bool lead = l == 0 && c == 0 && threadIdx.x == 0;
  if (A.flags && lead && bad) atomicOr(&A.flags[r], (uint32_t)SPEC_F_BAD_IDX);
  if (bad || acc == 0) return;
  if (A.swap && acc == A.S) {
    if (lead) {
      A.swap_slot[r] = scratch;
      A.swap_scratch[r] = slot;
    }
    return;
  }
  const int s = acc - 1;

  const bool is_rec = c < A.rec_chunks;
  if (!is_rec) c -= A.rec_chunks;
  const long long blob = is_rec ? A.rec_bytes : A.conv_bytes;
  const unsigned char* src = (is_rec ? A.vrec : A.vconv) +
                             (((long long)l * A.B + r) * A.SV + s) * blob;
  unsigned char* dst = (is_rec ? A.crec : A.cconv) + ((long long)l * A.slots + slot) * blob;
  const long long off = c * kChunk;
  const long long n = min(kChunk, blob - off);
  const bool vec = is_rec ? A.rec_vec : A.conv_vec;
  if (vec) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + off);
    uint4* d4 = reinterpret_cast<uint4*>(dst + off);
    const int nv = (int)(n / 16);
    uint4 buf[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int idx = threadIdx.x + i * kCopyThreads;
      if (idx < nv) buf[i] = __ldcs(s4 + idx);
    }
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int idx = threadIdx.x + i * kCopyThreads;
      if (idx < nv) __stcs(d4 + idx, buf[i]);
    }
  } else {
    // element-granular path (2-byte units cover both fp32 and bf16 blobs)
    const uint16_t* s2 = reinterpret_cast<const uint16_t*>(src + off);
    uint16_t* d2 = reinterpret_cast<uint16_t*>(dst + off);
    const int nh = (int)(n / 2);
    for (int i = threadIdx.x; i < nh; i += kCopyThreads) d2[i] = s2[i];
  }
}

}  // namespace specv

static inline bool aligned_to(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int specv::commit_check(const float* verify_rec, const uint16_t* verify_conv, const int32_t* accept_len,
                        const int32_t* cache_slot, const int32_t* swap_slot, const int32_t* swap_scratch,
                        const float* cache_rec, const uint16_t* cache_conv, int L, int B, int S, int H, int Dk,
                        int Dv, int W, int C, int slots, const uint32_t* flags) {
  const bool swap = swap_slot != nullptr;
  if (L < 0 || B < 0 || S < 1 || slots < 0) return SPEC_E_DIM;
  if (verify_rec && (H < 1 || Dk < 1 || Dv < 1)) return SPEC_E_DIM;
  if (verify_conv && (W < 1 || C < 1)) return SPEC_E_DIM;
  if (L == 0 || B == 0) return SPEC_OK;
  if (!accept_len) return SPEC_E_NULL;
  if (!verify_rec && !verify_conv) return SPEC_E_NULL;
  if (verify_rec && !cache_rec) return SPEC_E_NULL;
  if (verify_conv && !cache_conv) return SPEC_E_NULL;
  if (swap && !swap_scratch) return SPEC_E_NULL;
  if (!swap && !cache_slot && slots < B) return SPEC_E_DIM;
  if (!aligned_to(accept_len, 4) || (cache_slot && !aligned_to(cache_slot, 4)) ||
      (flags && !aligned_to(flags, 4)) || (swap && (!aligned_to(swap_slot, 4) || !aligned_to(swap_scratch, 4))))
    return SPEC_E_ALIGN;
  if (verify_rec && (!aligned_to(verify_rec, 4) || !aligned_to(cache_rec, 4))) return SPEC_E_ALIGN;
  if (verify_conv && (!aligned_to(verify_conv, 2) || !aligned_to(cache_conv, 2))) return SPEC_E_ALIGN;
  return SPEC_OK;
}

static int commit_launch(const float* verify_rec, const uint16_t* verify_conv, const int32_t* accept_len,
                         const int32_t* cache_slot, int32_t* swap_slot, int32_t* swap_scratch, float* cache_rec,
                         uint16_t* cache_conv, int L, int B, int S, int H, int Dk, int Dv, int W, int C, int slots,
                         uint32_t* flags, void* cuda_stream) {
  using namespace specv;
  const bool swap = swap_slot != nullptr;
  const int rc = commit_check(verify_rec, verify_conv, accept_len, cache_slot, swap_slot, swap_scratch, cache_rec,
                              cache_conv, L, B, S, H, Dk, Dv, W, C, slots, flags);
  if (rc != SPEC_OK || L == 0 || B == 0) return rc;
  const int arc = check_arch();
  if (arc != SPEC_OK) return arc;

  CommitArgs A;
  memset(&A, 0, sizeof(A));
  A.vrec = reinterpret_cast<const unsigned char*>(verify_rec);
  A.vconv = reinterpret_cast<const unsigned char*>(verify_conv);
  A.accept_len = accept_len;
  A.slot = cache_slot;
  A.swap_slot = swap_slot;
  A.swap_scratch = swap_scratch;
  A.swap = swap ? 1 : 0;
  A.crec = reinterpret_cast<unsigned char*>(cache_rec);
  A.cconv = reinterpret_cast<unsigned char*>(cache_conv);
  A.flags = flags;
  A.rec_bytes = verify_rec ? (long long)H * Dk * Dv * 4 : 0;
  A.conv_bytes = verify_conv ? (long long)W * C * 2 : 0;
  A.L = L;
  A.B = B;
  A.S = S;
  A.SV = swap ? S - 1 : S;
  A.slots = slots;
  A.rec_chunks = (A.rec_bytes + kChunk - 1) / kChunk;
  A.conv_chunks = (A.conv_bytes + kChunk - 1) / kChunk;
  A.rec_vec = verify_rec && aligned_to(verify_rec, 16) && aligned_to(cache_rec, 16) && A.rec_bytes % 16 == 0;
  A.conv_vec = verify_conv && aligned_to(verify_conv, 16) && aligned_to(cache_conv, 16) &&
               A.conv_bytes % 16 == 0;
  const long long jobs = (long long)L * B * (A.rec_chunks + A.conv_chunks);
  if (jobs == 0) return SPEC_OK;
  const long long gx = jobs < 65535 ? jobs : 65535;
  const long long gy = (jobs + gx - 1) / gx;
  if (gy > 65535) return SPEC_E_DIM;
  commit_kernel<<<dim3((unsigned)gx, (unsigned)gy, 1), kCopyThreads, 0,
                  reinterpret_cast<cudaStream_t>(cuda_stream)>>>(A);
  if (cudaGetLastError() != cudaSuccess) return SPEC_E_CUDA;
  return SPEC_OK;
}

extern "C" int spec_commit(const float* verify_rec, const uint16_t* verify_conv,
                           const int32_t* accept_len, const int32_t* cache_slot, float* cache_rec,
                           uint16_t* cache_conv, int L, int B, int S, int H, int Dk, int Dv, int W,
                           int C, int slots, uint32_t* flags, void* cuda_stream) {
  return commit_launch(verify_rec, verify_conv, accept_len, cache_slot, nullptr, nullptr, cache_rec, cache_conv, L, B,
                       S, H, Dk, Dv, W, C, slots, flags, cuda_stream);
}

extern "C" int spec_commit_swap(const float* verify_rec, const uint16_t* verify_conv, const int32_t* accept_len,
                                int32_t* slot_of_row, int32_t* scratch_slot, float* cache_rec,
                                uint16_t* cache_conv, int L, int B, int S, int H, int Dk, int Dv, int W, int C,
                                int slots, uint32_t* flags, void* cuda_stream) {
  if (L < 0 || B < 0 || S < 1 || slots < 0) return SPEC_E_DIM;
  if (L == 0 || B == 0) return SPEC_OK;
  if (!slot_of_row || !scratch_slot) return SPEC_E_NULL;
  return commit_launch(verify_rec, verify_conv, accept_len, nullptr, slot_of_row, scratch_slot, cache_rec,
                       cache_conv, L, B, S, H, Dk, Dv, W, C, slots, flags, cuda_stream);
}
