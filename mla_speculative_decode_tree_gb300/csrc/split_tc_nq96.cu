// Tensor-core split kernel instantiated for 96 query rows per CTA (value
// blocks fetched twice: a resident tile does not fit beside 96 rows of Q).
#include "split_tc.cuh"

namespace mlav {
cudaError_t launch_split_tc_96(const SplitArgs& a, const TcMaps& m, dim3 grid, cudaStream_t stream, bool resident) {
  if (resident) return cudaErrorInvalidValue;
  return launch_split_tc_nq<96, kRefetch>(a, m, grid, stream);
}
int split_tc_smem_96(bool resident) { return resident ? -1 : tc_smem_bytes<96, kRefetch>(); }
}  // namespace mlav
