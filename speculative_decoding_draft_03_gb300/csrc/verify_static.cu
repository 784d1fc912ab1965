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
// is looked up (cudaGetSymbolAddress, with the calling device current) by every call
// made outside stream capture; a call on a stream being captured reuses the address the
// last uncaptured call on that device looked up, so the first call on a device should
// happen before any stream capture begins.  All calls share the one array: calls that
// overlap on the GPU (different streams, or different host threads on the same device)
// race on it, so the caller must order them.  The array keeps the previous call's
// contents; this entry point clears the part that must start at zero (the status block)
// on the call's stream before the kernels run.  dspark_verify_static_status() reads
// that status block back (device-side reports of bad token ids, verify lengths or
// timeouts of the last call).
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

// The static array's device address on the current device.  Outside stream capture the
// address is looked up again on every call (cheap), so a context that was torn down and
// re-created (cudaDeviceReset) never leaves a stale pointer behind; while `s` is being
// captured the last address looked up on this device is used, because the lookup may
// not be legal during capture.
dspark_status scratch_address(cudaStream_t s, void** out, const char* who) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    char msg[160];
    snprintf(msg, sizeof msg, "%s: no usable current device", who);
    return dspark::record_error(DSPARK_CUDA_ERROR, msg);
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) cap = cudaStreamCaptureStatusNone;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap == cudaStreamCaptureStatusNone || g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[200];
      snprintf(msg, sizeof msg, "%s: cudaGetSymbolAddress failed: %s", who, cudaGetErrorString(e));
      return dspark::record_error(DSPARK_CUDA_ERROR, msg);
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DSPARK_OK;
}

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
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  const dspark_status st = scratch_address(s, &scratch, "dspark_verify_static");
  if (st != DSPARK_OK) return st;
  if (cudaMemsetAsync(scratch, 0, 256, s) != cudaSuccess)
    return dspark::record_error(DSPARK_CUDA_ERROR, "dspark_verify_static: clearing the status block failed");
  return dspark_verify(R, gamma, V, rank, dtype_t, dtype_u, dtype_w, target, U, W1, W2, x0, x, logq, lse_q, ell,
                       temperature, req_id, seed, round, n_acc_out, tokens_out, n_out, scratch, need, stream);
}

// The device status word of the static scratch on the current device: what the last
// dspark_verify_static call's kernels reported (DSPARK_INVALID_ARG for a token id,
// verify length or target row out of range, DSPARK_TIMEOUT for a bounded wait that gave
// up).  Each dspark_verify_static call clears the word on its stream before its kernels
// run, so read it after the call and before the next one.
extern "C" dspark_status dspark_verify_static_status(int reset, int* status, void* stream) {
  if (status == nullptr) return dspark::record_error(DSPARK_INVALID_ARG, "dspark_verify_static_status: status is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  const dspark_status st = scratch_address(s, &scratch, "dspark_verify_static_status");
  if (st != DSPARK_OK) return st;
  return dspark_workspace_status(scratch, reset, status, stream);
}
