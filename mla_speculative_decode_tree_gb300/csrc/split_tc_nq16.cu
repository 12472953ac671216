// Tensor-core split kernel instantiated for 16 query rows per CTA, in both
// modes (value blocks fetched twice, or the whole tile resident).
#include "split_tc.cuh"

namespace mlav {
cudaError_t launch_split_tc_16(const SplitArgs& a, const TcMaps& m, dim3 grid, cudaStream_t stream, bool resident) {
  return resident ? launch_split_tc_nq<16, kResident>(a, m, grid, stream)
                  : launch_split_tc_nq<16, kRefetch>(a, m, grid, stream);
}
int split_tc_smem_16(bool resident) {
  return resident ? tc_smem_bytes<16, kResident>() : tc_smem_bytes<16, kRefetch>();
}
}  // namespace mlav
