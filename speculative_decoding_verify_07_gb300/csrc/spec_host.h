// Host-side helpers shared by the library's translation units.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/spec_verify.h"

namespace specv {

struct FusedCommit;

// Draft sampling options of a verify launch (spec_draft_sample): where the
// settled units' kept-set descriptors go, the Philox stream word of the
// entries' race uniforms (blocks use the next one) and the position added to
// every Philox counter.
struct DraftOpts {
  unsigned long long* desc;
  uint32_t race_stream;
  uint32_t pos_base;
};

// SPEC_OK when the current device is an sm_103 GPU, SPEC_E_ARCH otherwise,
// SPEC_E_CUDA when the device cannot be queried.  Cached per device.
int check_arch();

// The argument checks of spec_verify (need_workspace: a caller workspace is
// required and checked).  Enqueues nothing.  SPEC_OK for B == 0 without
// further checks.
int verify_check(const void* logits, int logits_dtype, const float* draft_probs, const int32_t* draft_tokens,
                 const spec_params_t* params, int B, int k, int V, const int32_t* tokens, const int32_t* accept_len,
                 const float* logprobs, const float* alpha, const uint32_t* flags, bool need_workspace,
                 const void* workspace, size_t workspace_bytes);

// The launch of spec_verify on arguments verify_check accepted (B > 0),
// with a workspace of at least spec_verify_workspace_size(B, k, V) bytes.
// fc (or null): the commit to fuse into the launch (spec_verify_commit);
// dr (or null): draft sampling options (spec_draft_sample).
int verify_launch(const void* logits, int logits_dtype, const float* draft_probs, const int32_t* draft_tokens,
                  const spec_params_t* params, uint64_t seed, uint32_t row_base, int B, int k, int V,
                  int32_t* tokens, int32_t* accept_len, float* logprobs, float* alpha, uint32_t* flags,
                  void* workspace, void* cuda_stream, const FusedCommit* fc, const DraftOpts* dr = nullptr);

// The argument checks of spec_commit (swap_slot non-null: spec_commit_swap).
// Enqueues nothing; SPEC_OK for L == 0 or B == 0 after the dimension checks.
int commit_check(const float* verify_rec, const uint16_t* verify_conv, const int32_t* accept_len,
                 const int32_t* cache_slot, const int32_t* swap_slot, const int32_t* swap_scratch,
                 const float* cache_rec, const uint16_t* cache_conv, int L, int B, int S, int H, int Dk, int Dv,
                 int W, int C, int slots, const uint32_t* flags);

}  // namespace specv
