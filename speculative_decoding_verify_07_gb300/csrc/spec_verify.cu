// spec_verify: batched speculative-decoding verify sampler for sm_103a --
// argument checks, workspace carving and the launch.
//
// One persistent kernel on the caller's stream, with no host
// synchronisation (spec_kernel.cu): stream warps reduce every logit row
// once in tiles and stream the draft probabilities of drafted positions over
// unfiltered distributions, while settle warps settle each (row, position)
// as soon as its last tile is reduced (spec_settle.cuh); rows that need a
// global threshold search take the general path (spec_general.cuh).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "spec_common.cuh"
#include "spec_host.h"

extern "C" size_t spec_verify_workspace_size(int B, int k, int V) {
  if (B < 0 || k < 0 || V < 1) return 0;
  return specv::ws_layout(B, k, V).total;
}

static inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

namespace specv {

int verify_check(const void* logits, int logits_dtype, const float* draft_probs, const int32_t* draft_tokens,
                 const spec_params_t* params, int B, int k, int V, const int32_t* tokens, const int32_t* accept_len,
                 const float* logprobs, const float* alpha, const uint32_t* flags, bool need_workspace,
                 const void* workspace, size_t workspace_bytes) {
  if (B < 0 || k < 0 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return SPEC_E_DIM;
  if ((long long)B * (k + 1) > (1ll << 24)) return SPEC_E_DIM;
  if (logits_dtype != SPEC_F32 && logits_dtype != SPEC_BF16) return SPEC_E_DTYPE;
  if (B == 0) return SPEC_OK;
  if (!logits || !params || !tokens || !accept_len || !logprobs || !flags) return SPEC_E_NULL;
  if (need_workspace && !workspace) return SPEC_E_NULL;
  if (k > 0 && (!draft_probs || !draft_tokens || !alpha)) return SPEC_E_NULL;
  const size_t es = logits_dtype == SPEC_BF16 ? 2 : 4;
  if (!aligned(logits, es) || !aligned(params, 4) || !aligned(tokens, 4) || !aligned(accept_len, 4) ||
      !aligned(logprobs, 4) || !aligned(flags, 4))
    return SPEC_E_ALIGN;
  if (need_workspace && !aligned(workspace, 16)) return SPEC_E_ALIGN;
  if (k > 0 && (!aligned(draft_probs, 4) || !aligned(draft_tokens, 4) || !aligned(alpha, 4)))
    return SPEC_E_ALIGN;
  if (need_workspace && workspace_bytes < ws_layout(B, k, V).total) return SPEC_E_WORKSPACE;
  // items of the stream sequence (A tiles of every unit, B tiles of every drafted unit)
  const long long items = (long long)B * (k + 1) * max_nta(V) + (long long)B * k * max_ntb(V);
  if (items > 0x7fffffffLL) return SPEC_E_DIM;
  return check_arch();
}

int verify_launch(const void* logits, int logits_dtype, const float* draft_probs, const int32_t* draft_tokens,
                  const spec_params_t* params, uint64_t seed, uint32_t row_base, int B, int k, int V,
                  int32_t* tokens, int32_t* accept_len, float* logprobs, float* alpha, uint32_t* flags,
                  void* workspace, void* cuda_stream, const FusedCommit* fc, const DraftOpts* dr) {
  const size_t es = logits_dtype == SPEC_BF16 ? 2 : 4;
  const Layout L = ws_layout(B, k, V);
  Args A;
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
  A.ws = reinterpret_cast<WsHeader*>(ws);
  A.row_ticket = reinterpret_cast<uint32_t*>(ws + L.row_ticket);
  A.ucnt = reinterpret_cast<uint32_t*>(ws + L.ucnt);
  A.rec = reinterpret_cast<u64*>(ws + L.rec);
  A.brec = reinterpret_cast<u64*>(ws + L.brec);
  A.ust = reinterpret_cast<u64*>(ws + L.ust);
  A.urec = reinterpret_cast<u64*>(ws + L.urec);
  A.order = reinterpret_cast<uint32_t*>(ws + L.order);
  A.done = reinterpret_cast<u64*>(ws + L.done);
  A.tp = reinterpret_cast<u64*>(ws + L.tp);
  if (fc) A.fc = *fc;
  A.race_stream = 1u;   // entries on Philox stream 1, blocks on stream 2
  if (dr) {
    A.desc = dr->desc;
    A.race_stream = dr->race_stream;
    A.pos_base = dr->pos_base;
  }
  A.key0 = (uint32_t)(seed & 0xffffffffull);
  A.key1 = (uint32_t)(seed >> 32);
  A.row_base = row_base;
  A.B = B;
  A.k = k;
  A.V = V;
  A.U = B * (k + 1);
  A.NTA = max_nta(V);
  A.NTB = max_ntb(V);
  A.vec_logits = aligned(logits, 16) && ((size_t)V * es) % 16 == 0;
  A.l2_stage = A.vec_logits && (size_t)B * (size_t)(k + 1) * (size_t)V * es <= ((size_t)64 << 20);
  A.vec_q = k > 0 && aligned(draft_probs, 16) && (V % 4) == 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
  return logits_dtype == SPEC_BF16 ? launch_verify<true>(A, st) : launch_verify<false>(A, st);
}

}  // namespace specv

extern "C" int spec_verify(const void* logits, int logits_dtype, const float* draft_probs,
                           const int32_t* draft_tokens, const spec_params_t* params, uint64_t seed,
                           uint32_t row_base, int B, int k, int V, int32_t* tokens, int32_t* accept_len,
                           float* logprobs, float* alpha, uint32_t* flags, void* workspace,
                           size_t workspace_bytes, void* cuda_stream) {
  const int rc = specv::verify_check(logits, logits_dtype, draft_probs, draft_tokens, params, B, k, V, tokens,
                                     accept_len, logprobs, alpha, flags, true, workspace, workspace_bytes);
  if (rc != SPEC_OK || B == 0) return rc;
  return specv::verify_launch(logits, logits_dtype, draft_probs, draft_tokens, params, seed, row_base, B, k, V,
                              tokens, accept_len, logprobs, alpha, flags, workspace, cuda_stream, nullptr);
}

extern "C" int spec_verify_commit(const void* logits, int logits_dtype, const float* draft_probs,
                                  const int32_t* draft_tokens, const spec_params_t* params, uint64_t seed,
                                  uint32_t row_base, int B, int k, int V, int32_t* tokens, int32_t* accept_len,
                                  float* logprobs, float* alpha, uint32_t* flags, void* workspace,
                                  size_t workspace_bytes, const float* verify_rec, const uint16_t* verify_conv,
                                  const int32_t* cache_slot, float* cache_rec, uint16_t* cache_conv, int L, int H,
                                  int Dk, int Dv, int W, int C, int slots, void* cuda_stream) {
  using namespace specv;
  // the commit's argument checks, then the verify's (which end with the device query)
  if (B < 0 || k < 0 || k > SPEC_MAX_K) return SPEC_E_DIM;
  int rc = commit_check(verify_rec, verify_conv, accept_len, cache_slot, nullptr, nullptr, cache_rec, cache_conv, L, B,
                        k + 1, H, Dk, Dv, W, C, slots, flags);
  if (rc != SPEC_OK) return rc;
  rc = verify_check(logits, logits_dtype, draft_probs, draft_tokens, params, B, k, V, tokens, accept_len, logprobs,
                    alpha, flags, true, workspace, workspace_bytes);
  if (rc != SPEC_OK || B == 0) return rc;
  FusedCommit F;
  memset(&F, 0, sizeof(F));
  if (L > 0) {
    F.vrec = reinterpret_cast<const unsigned char*>(verify_rec);
    F.vconv = reinterpret_cast<const unsigned char*>(verify_conv);
    F.slot = cache_slot;
    F.crec = reinterpret_cast<unsigned char*>(cache_rec);
    F.cconv = reinterpret_cast<unsigned char*>(cache_conv);
    F.rec_bytes = verify_rec ? (long long)H * Dk * Dv * 4 : 0;
    F.conv_bytes = verify_conv ? (long long)W * C * 2 : 0;
    F.L = L;
    F.slots = slots;
    F.rec_jobs = (int)((F.rec_bytes + kJobBytes - 1) / kJobBytes);
    F.conv_jobs = (int)((F.conv_bytes + kJobBytes - 1) / kJobBytes);
    F.bulk = (!verify_rec || (aligned(verify_rec, 16) && aligned(cache_rec, 16) && F.rec_bytes % 16 == 0)) &&
             (!verify_conv || (aligned(verify_conv, 16) && aligned(cache_conv, 16) && F.conv_bytes % 16 == 0));
    const long long jobs = (long long)B * L * (F.rec_jobs + F.conv_jobs);
    if (jobs > 0x7fffffffLL) return SPEC_E_DIM;
    F.on = jobs > 0 ? 1 : 0;
  }
  return verify_launch(logits, logits_dtype, draft_probs, draft_tokens, params, seed, row_base, B, k, V, tokens,
                       accept_len, logprobs, alpha, flags, workspace, cuda_stream, &F);
}
