// Tensor-core split kernel instantiated for 64 query rows per CTA, in both
// modes (value blocks fetched twice, or the whole tile resident).
#include "split_tc.cuh"

namespace mlav {
cudaError_t launch_split_tc_64(const SplitArgs& a, const TcMaps& m, dim3 grid, cudaStream_t stream, bool resident) {
  return resident ? launch_split_tc_nq<64, kResident>(a, m, grid, stream)
                  : launch_split_tc_nq<64, kRefetch>(a, m, grid, stream);
}
int split_tc_smem_64(bool resident) {
  return resident ? tc_smem_bytes<64, kResident>() : tc_smem_bytes<64, kRefetch>();
}
}  // namespace mlav
