// draft_tc.cu — tensor-core (tcgen05 / TMEM / TMA) draft step (placeholder until the
// fused kernel lands: every shape runs the CUDA-core step).
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

int tc_supported(int V, int rank, int dtype_w) {
  (void)V;
  (void)rank;
  (void)dtype_w;
  return 0;
}

int tc_grid_size() { return 1; }

cudaError_t launch_draft_step_tc(const DraftArgs& a, int k, cudaStream_t s) {
  (void)a;
  (void)k;
  (void)s;
  return cudaErrorNotSupported;
}

}  // namespace dspark
