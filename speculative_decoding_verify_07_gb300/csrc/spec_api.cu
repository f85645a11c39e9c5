// Status strings, version, device check and the Philox diagnostic entry point.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/spec_verify.h"
#include "spec_device.cuh"
#include "spec_host.h"

namespace specv {

int check_arch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_E_CUDA;
  }
  static std::mutex mu;
  static int known[64];   // 0 unknown, 1 ok, 2 wrong arch
  if (dev < 0 || dev >= 64) return SPEC_E_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (known[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return SPEC_E_CUDA;
    }
    known[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return known[dev] == 1 ? SPEC_OK : SPEC_E_ARCH;
}

__global__ void philox_kernel(const uint4* ctr, uint32_t k0, uint32_t k1, uint4* out, long long n) {
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i < n) out[i] = philox4x32_10(ctr[i], k0, k1);
}

}  // namespace specv

extern "C" int spec_philox4x32_10(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n,
                                  void* cuda_stream) {
  if (n < 0) return SPEC_E_DIM;
  if (n == 0) return SPEC_OK;
  if (!ctr || !out) return SPEC_E_NULL;
  if (((uintptr_t)ctr % 16) || ((uintptr_t)out % 16)) return SPEC_E_ALIGN;
  const int arc = specv::check_arch();
  if (arc != SPEC_OK) return arc;
  const long long blocks = (n + 255) / 256;
  if (blocks > 0x7fffffffLL) return SPEC_E_DIM;
  specv::philox_kernel<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(cuda_stream)>>>(
      reinterpret_cast<const uint4*>(ctr), (uint32_t)(seed & 0xffffffffull), (uint32_t)(seed >> 32),
      reinterpret_cast<uint4*>(out), (long long)n);
  if (cudaGetLastError() != cudaSuccess) return SPEC_E_CUDA;
  return SPEC_OK;
}

extern "C" const char* spec_status_string(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_E_NULL: return "a required pointer is NULL";
    case SPEC_E_DIM: return "a size argument is out of range";
    case SPEC_E_DTYPE: return "unknown logits dtype";
    case SPEC_E_ALIGN: return "a pointer is not aligned to its element size";
    case SPEC_E_WORKSPACE: return "workspace missing or too small";
    case SPEC_E_CUDA: return "CUDA runtime call or kernel launch failed";
    case SPEC_E_ARCH: return "the current device is not an sm_103 GPU";
    default: return "unknown status code";
  }
}

extern "C" int spec_version(void) { return SPEC_ABI_VERSION; }
