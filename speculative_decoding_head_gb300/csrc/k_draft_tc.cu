// k_draft_tc.cu -- persistent tcgen05 Markov-head draft kernel (sm_103a).
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

int draft_tc_supported(const dspark_dims& d) {
  (void)d;
  return 0;
}

cudaError_t draft_tc_configure(dspark_ws* ws) {
  (void)ws;
  return cudaErrorNotSupported;
}

size_t draft_tc_scratch_rows(const dspark_dims& d, int grid) {
  (void)d;
  (void)grid;
  return 0;
}

cudaError_t launch_draft_tc(const dspark_ws* ws, const DraftArgs& a, cudaStream_t st, int* launches) {
  (void)ws;
  (void)a;
  (void)st;
  (void)launches;
  return cudaErrorNotSupported;
}

}  // namespace dspark
