// Tensor-core split kernel instantiated for 16 query rows per CTA.
#include "split_tc.cuh"

namespace mlav {
cudaError_t launch_split_tc_16(const SplitArgs& a, const TcMaps& m, dim3 grid, cudaStream_t stream) {
  return launch_split_tc_nq<16>(a, m, grid, stream);
}
int split_tc_smem_16() { return tc_smem_bytes<16>(); }
}  // namespace mlav
