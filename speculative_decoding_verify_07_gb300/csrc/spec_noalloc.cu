// spec_verify_noalloc: spec_verify for callers that cannot allocate device memory.
//
// Some callers cannot allocate device memory when they run the verify step:
// plugin or custom-op hosts that hand a kernel only its input and output
// buffers and offer no scratch allocator, serving engines whose caching
// allocator has already reserved all of HBM (for KV cache) so that a
// cudaMalloc would fail, and tight decode loops that cannot afford the device
// synchronisation a cudaMalloc/cudaFree pair implies.  For them this entry
// point runs the verify step with scratch that the library itself holds: a
// file-scope device array of SPEC_NOALLOC_MAX_WORKSPACE bytes, present on
// every GPU that loads the library until the process exits.  The caller still
// passes every input and output buffer.  The verify step itself is the same
// kernel spec_verify launches, handed this array as its workspace.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/spec_verify.h"
#include "spec_host.h"

namespace {

static __device__ __align__(256) unsigned char g_verify_scratch[SPEC_NOALLOC_MAX_WORKSPACE];

std::mutex g_mu;
void* g_addr[64];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current and reused afterwards.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  if (dev < 0 || dev >= 64) return SPEC_E_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SPEC_E_CUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_verify_noalloc(const void* logits, int logits_dtype, const float* draft_probs,
                                   const int32_t* draft_tokens, const spec_params_t* params,
                                   uint64_t seed, uint32_t row_base, int B, int k, int V, int32_t* tokens,
                                   int32_t* accept_len, float* logprobs, float* alpha,
                                   uint32_t* flags, void* cuda_stream) {
  // every argument check of spec_verify first: a refused call enqueues nothing
  if (B < 0 || k < 0 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return SPEC_E_DIM;
  const size_t need = spec_verify_workspace_size(B, k, V);
  if (need > (size_t)SPEC_NOALLOC_MAX_WORKSPACE) return SPEC_E_WORKSPACE;
  const int rc = specv::verify_check(logits, logits_dtype, draft_probs, draft_tokens, params, B, k, V, tokens,
                                     accept_len, logprobs, alpha, flags, false, nullptr, 0);
  if (rc != SPEC_OK || B == 0) return rc;
  void* scratch = nullptr;
  const int ra = scratch_address(&scratch);
  if (ra != SPEC_OK) return ra;
  // The array keeps the previous call's contents; clear the part this call uses.
  if (cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  return specv::verify_launch(logits, logits_dtype, draft_probs, draft_tokens, params, seed, row_base, B, k, V,
                              tokens, accept_len, logprobs, alpha, flags, scratch, cuda_stream, nullptr);
}
