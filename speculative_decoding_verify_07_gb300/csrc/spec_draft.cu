// spec_draft_sample: the draft-side sampler (sm_103a).
//
// inclusionAI/AReno PR #550, "What does this PR do?" Phase 2: the MTP head
// drafts EAGLE-style, one position at a time, with the same sampler
// settings as the target; the verify then needs each draft token x and the
// draft distribution q it was drawn from.  One draft step over B rows is
// the verify launch with k = 0 on the draft logits (its bonus draw is a draw
// from the sampler-equivalent distribution of those logits), with the
// Philox streams moved to words 3 (entries) and 4 (blocks) at counter
// position `pos`, so that draft draws and verify draws are independent, and
// with every settled unit publishing its kept set and normaliser.  A second
// kernel then writes q = that distribution over all V entries, one pass of
// coalesced loads and stores (HBM-bound).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "spec_common.cuh"
#include "spec_host.h"

namespace specv {

struct DraftLayout {
  size_t desc, acc, total;
};
static DraftLayout draft_layout(int B, int V) {
  DraftLayout L;
  size_t off = ws_layout(B, 0, V).total;
  L.desc = off;
  off = align_up(off + (size_t)B * kDescWords * 8, 256);
  L.acc = off;
  off = align_up(off + (size_t)B * 4, 256);
  L.total = off;
  return L;
}

constexpr int kQThreads = 256;
constexpr int kQEntries = kQThreads * 8;   // entries a CTA writes per round

// q for row blockIdx.y: p(v) = exp2((l_v - m) c) / Z_S on the kept set
// (every entry, or the prefix of the total order up to the threshold), the
// one-hot argmax under greedy decoding, 0 elsewhere and for invalid rows.
template <bool kBF16>
__global__ void __launch_bounds__(kQThreads) draft_q_kernel(const void* logits, const spec_params_t* params,
                                                            const u64* desc, const WsHeader* ws, int V,
                                                            int vec_in, int vec_out, float* q) {
  __shared__ uint32_t d[5];
  __shared__ int ok;
  const int row = blockIdx.y;
  if (threadIdx.x < 32) {
    // the verify launch before this one wrote its tag as the epoch
    const uint32_t tag = __ldcg(&ws->epoch);
    const int lane = threadIdx.x;
    const u64 w = lane < 5 ? __ldcg(desc + (size_t)row * kDescWords + lane) : 0ull;
    const bool good = __all_sync(0xffffffffu, lane >= 5 || tag_ok(w, tag));
    if (lane < 5) d[lane] = (uint32_t)w;
    if (lane == 0) ok = good ? 1 : 0;
  }
  __syncthreads();
  const uint32_t mode = ok ? d[0] : 0u;
  const float m = __uint_as_float(d[1]), invZ = __uint_as_float(d[2]);
  const uint32_t tkey = d[3], tidx = d[4];
  const float c = classify(params[row], V).c;
  const size_t base = (size_t)row * (size_t)V;
  for (int e0 = (blockIdx.x * kQThreads + threadIdx.x) * 8; e0 < V; e0 += gridDim.x * kQEntries) {
    float v[8];
    if (kBF16) {
      const uint16_t* p = reinterpret_cast<const uint16_t*>(logits) + base;
      if (vec_in && e0 + 8 <= V) {
        const uint4 x = __ldcs(reinterpret_cast<const uint4*>(p + e0));
        v[0] = bf16_lo(x.x); v[1] = bf16_hi(x.x); v[2] = bf16_lo(x.y); v[3] = bf16_hi(x.y);
        v[4] = bf16_lo(x.z); v[5] = bf16_hi(x.z); v[6] = bf16_lo(x.w); v[7] = bf16_hi(x.w);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = e0 + i < V ? __uint_as_float((uint32_t)p[e0 + i] << 16) : -INFINITY;
      }
    } else {
      const float* p = reinterpret_cast<const float*>(logits) + base;
      if (vec_in && e0 + 8 <= V) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(p + e0));
        const float4 b = __ldcs(reinterpret_cast<const float4*>(p + e0 + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = e0 + i < V ? p[e0 + i] : -INFINITY;
      }
    }
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t idx = (uint32_t)(e0 + i);
      float pv = 0.f;
      if (mode == DESC_GREEDY) {
        pv = idx == tidx ? 1.0f : 0.0f;
      } else if (mode == DESC_ALL || mode == DESC_THRESH) {
        const uint32_t key = okey(v[i]);
        const bool in = mode == DESC_ALL || key > tkey || (key == tkey && idx <= tidx);
        pv = in ? ex2((v[i] - m) * c) * invZ : 0.0f;
      }
      o[i] = pv;
    }
    float* qo = q + base;
    if (vec_out && e0 + 8 <= V) {
      __stcs(reinterpret_cast<float4*>(qo + e0), make_float4(o[0], o[1], o[2], o[3]));
      __stcs(reinterpret_cast<float4*>(qo + e0 + 4), make_float4(o[4], o[5], o[6], o[7]));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (e0 + i < V) qo[e0 + i] = o[i];
    }
  }
}

}  // namespace specv

static inline bool aligned_to(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

extern "C" size_t spec_draft_workspace_size(int B, int V) {
  if (B < 0 || V < 1) return 0;
  return specv::draft_layout(B, V).total;
}

extern "C" int spec_draft_sample(const void* logits, int logits_dtype, const spec_params_t* params, uint64_t seed,
                                 uint32_t row_base, uint32_t pos, int B, int V, float* q, int32_t* tokens,
                                 float* logprobs, uint32_t* flags, void* workspace, size_t workspace_bytes,
                                 void* cuda_stream) {
  using namespace specv;
  if (B < 0 || V < 1 || V > SPEC_MAX_V || B > (1 << 24)) return SPEC_E_DIM;
  if (logits_dtype != SPEC_F32 && logits_dtype != SPEC_BF16) return SPEC_E_DTYPE;
  if (B == 0) return SPEC_OK;
  if (!workspace) return SPEC_E_NULL;
  if (!aligned_to(workspace, 16) || (q && !aligned_to(q, 4))) return SPEC_E_ALIGN;
  const DraftLayout DL = draft_layout(B, V);
  if (workspace_bytes < DL.total) return SPEC_E_WORKSPACE;
  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  int32_t* acc = reinterpret_cast<int32_t*>(ws + DL.acc);
  // the verify's own checks (k = 0: no draft arrays), ending with the device query
  int rc = verify_check(logits, logits_dtype, nullptr, nullptr, params, B, 0, V, tokens, acc, logprobs, nullptr,
                        flags, true, workspace, workspace_bytes);
  if (rc != SPEC_OK) return rc;
  DraftOpts dr;
  dr.desc = reinterpret_cast<unsigned long long*>(ws + DL.desc);
  dr.race_stream = 3u;
  dr.pos_base = pos;
  rc = verify_launch(logits, logits_dtype, nullptr, nullptr, params, seed, row_base, B, 0, V, tokens, acc, logprobs,
                     nullptr, flags, workspace, cuda_stream, nullptr, &dr);
  if (rc != SPEC_OK || !q) return rc;
  const size_t es = logits_dtype == SPEC_BF16 ? 2 : 4;
  const int vec_in = aligned_to(logits, 16) && ((size_t)V * es) % 16 == 0;
  const int vec_out = aligned_to(q, 16) && V % 4 == 0;
  const dim3 grid((unsigned)ceil_div(V, kQEntries), (unsigned)B);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
  const WsHeader* hdr = reinterpret_cast<const WsHeader*>(workspace);
  const u64* desc = reinterpret_cast<const u64*>(dr.desc);
  if (logits_dtype == SPEC_BF16)
    draft_q_kernel<true><<<grid, kQThreads, 0, st>>>(logits, params, desc, hdr, V, vec_in, vec_out, q);
  else
    draft_q_kernel<false><<<grid, kQThreads, 0, st>>>(logits, params, desc, hdr, V, vec_in, vec_out, q);
  if (cudaGetLastError() != cudaSuccess) return SPEC_E_CUDA;
  return SPEC_OK;
}
