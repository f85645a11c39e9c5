// spec_verify: batched speculative-decoding verify sampler for sm_103a --
// argument checks, workspace carving and the launch.
//
// One persistent kernel on the caller's stream, with no host
// synchronisation (spec_kernel.cu): streaming warps reduce every logit row
// once and stream the draft probabilities of drafted positions over
// unfiltered distributions, while a settle group per CTA settles each
// (row, position) as soon as its chunks are reduced (spec_settle.cuh; rows
// that need a global threshold search take the general path,
// spec_general.cuh).  Batches beyond 512 rows get a one-CTA planning kernel
// first.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "spec_host.h"
#include "spec_verify_common.cuh"

extern "C" size_t spec_verify_workspace_size(int B, int k, int V) {
  if (B < 0 || k < 0 || V < 1) return 0;
  return specv::ws_layout(B, k, V).total;
}

static inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

extern "C" int spec_verify(const void* logits, int logits_dtype, const float* draft_probs,
                           const int32_t* draft_tokens, const spec_params_t* params, uint64_t seed,
                           int B, int k, int V, int32_t* tokens, int32_t* accept_len,
                           float* logprobs, float* alpha, uint32_t* flags, void* workspace,
                           size_t workspace_bytes, void* cuda_stream) {
  if (B < 0 || k < 0 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return SPEC_E_DIM;
  if ((long long)B * (k + 1) > (1ll << 24)) return SPEC_E_DIM;
  if (logits_dtype != SPEC_F32 && logits_dtype != SPEC_BF16) return SPEC_E_DTYPE;
  if (B == 0) return SPEC_OK;
  if (!logits || !params || !tokens || !accept_len || !logprobs || !flags || !workspace)
    return SPEC_E_NULL;
  if (k > 0 && (!draft_probs || !draft_tokens || !alpha)) return SPEC_E_NULL;
  const size_t es = logits_dtype == SPEC_BF16 ? 2 : 4;
  if (!aligned(logits, es) || !aligned(params, 4) || !aligned(tokens, 4) || !aligned(accept_len, 4) ||
      !aligned(logprobs, 4) || !aligned(flags, 4) || !aligned(workspace, 16))
    return SPEC_E_ALIGN;
  if (k > 0 && (!aligned(draft_probs, 4) || !aligned(draft_tokens, 4) || !aligned(alpha, 4)))
    return SPEC_E_ALIGN;
  const specv::Layout L = specv::ws_layout(B, k, V);
  if (workspace_bytes < L.total) return SPEC_E_WORKSPACE;
  // items of the streaming kernels (A items of every unit, B items of every drafted unit)
  const long long items = (long long)B * (k + 1) * specv::max_nca(V) + (long long)B * k * specv::max_ncb(V);
  if (items > 0x7fffffffLL) return SPEC_E_DIM;
  const int arc = specv::check_arch();
  if (arc != SPEC_OK) return arc;

  specv::Args A;
  memset(&A, 0, sizeof(A));
  A.logits = logits;
  A.q = draft_probs;
  A.drafts = draft_tokens;
  A.params = params;
  A.tokens = tokens;
  A.accept_len = accept_len;
  A.logprobs = logprobs;
  A.alpha = alpha;
  A.flags = flags;
  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  A.ws = reinterpret_cast<specv::WsHeader*>(ws);
  A.row_ticket = reinterpret_cast<uint32_t*>(ws + L.row_ticket);
  A.rec = reinterpret_cast<specv::u64*>(ws + L.rec);
  A.ust = reinterpret_cast<specv::u64*>(ws + L.ust);
  A.brec = reinterpret_cast<specv::u64*>(ws + L.brec);
  A.urec = reinterpret_cast<specv::u64*>(ws + L.urec);
  A.order = reinterpret_cast<uint32_t*>(ws + L.order);
  A.key0 = (uint32_t)(seed & 0xffffffffull);
  A.key1 = (uint32_t)(seed >> 32);
  A.B = B;
  A.k = k;
  A.V = V;
  A.U = B * (k + 1);
  A.NCA = specv::max_nca(V);
  A.NCB = specv::max_ncb(V);
  A.vec_logits = aligned(logits, 16) && ((size_t)V * es) % 16 == 0;
  A.vec_q = k > 0 && aligned(draft_probs, 16) && (V % 4) == 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
  return logits_dtype == SPEC_BF16 ? specv::launch_verify<true>(A, st) : specv::launch_verify<false>(A, st);
}
