// verify_static.cu — dspark_verify for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they run
// verification: code running inside another framework's memory pool that must not be
// bypassed, real-time paths that forbid allocation after start-up, or plugins whose
// host process owns all device memory.  For them this entry point takes its scratch
// from a fixed array compiled into the library instead of a caller workspace.
//
// The scratch is a file-scope __device__ array of kScratchBytes (8 MiB).  Every GPU
// that loads the library keeps one copy until the process exits.  Its device address
// is looked up once per device (cudaGetSymbolAddress, with that device current) by the
// first call made on that device; that first call should therefore happen before any
// stream capture begins.  All calls share the one array: calls that overlap on the GPU
// (different streams, or different host threads on the same device) race on it, so the
// caller must order them.  The array keeps the previous call's contents; this entry
// point clears the part that must start at zero (the status block) on the call's
// stream before the kernels run.
#include <stdio.h>

#include <mutex>

#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" dspark_status dspark_verify_static(
    int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w, const void* target, const void* U,
    const void* W1, const void* W2, const int32_t* x0, const int32_t* x, const float* logq, const float* lse_q,
    const int32_t* ell, float temperature, const int64_t* req_id, uint64_t seed, uint64_t round, int32_t* n_acc_out,
    int32_t* tokens_out, int32_t* n_out, void* stream) {
  const size_t need = dspark_verify_workspace_size(R, gamma, V, rank, dtype_w);
  if (need == 0)  // invalid sizes: let the regular entry point report them
    return dspark_verify(R, gamma, V, rank, dtype_t, dtype_u, dtype_w, target, U, W1, W2, x0, x, logq, lse_q, ell,
                         temperature, req_id, seed, round, n_acc_out, tokens_out, n_out, nullptr, 0, stream);
  if (need > kScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof msg, "dspark_verify_static: this shape needs %zu bytes of scratch, the static scratch holds %zu",
             need, kScratchBytes);
    return dspark::record_error(DSPARK_UNSUPPORTED_SHAPE, msg);
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return dspark::record_error(DSPARK_CUDA_ERROR, "dspark_verify_static: no usable current device");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_verify_scratch);
      if (e != cudaSuccess || p == nullptr) {
        char msg[200];
        snprintf(msg, sizeof msg, "dspark_verify_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        return dspark::record_error(DSPARK_CUDA_ERROR, msg);
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 256, s) != cudaSuccess)
    return dspark::record_error(DSPARK_CUDA_ERROR, "dspark_verify_static: clearing the status block failed");
  return dspark_verify(R, gamma, V, rank, dtype_t, dtype_u, dtype_w, target, U, W1, W2, x0, x, logq, lse_q, ell,
                       temperature, req_id, seed, round, n_acc_out, tokens_out, n_out, scratch, need, stream);
}
