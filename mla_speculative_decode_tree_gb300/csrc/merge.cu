// Merge kernel: combines the nsplit partials of every query row by
// log-sum-exp -- the second reduction kernel of the split-K verify
// [Custom sm_120 Verify Kernel, §"Building the Custom Kernel: From Occupancy
// Starvation to Flash-Decode"].  Two warps per row, one per half of the 512
// latent columns; the per-row arithmetic is merge_row_half (merge_row.cuh).
#include "merge_row.cuh"

namespace mlav {
namespace {

constexpr int kRowsPerBlock = 4;

__global__ void __launch_bounds__(64 * kRowsPerBlock) merge_kernel(MergeArgs a) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // The split kernels of this call have finished (stream order): hand their
    // status bits to the "last call" word and reset the accumulator.
    const uint32_t st = a.status[0];
    if (st) atomicOr(a.status + 1, st);
    a.status[0] = 0u;
  }
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int row = blockIdx.x * kRowsPerBlock + (warp >> 1);
  const int half = warp & 1;
  if (row >= a.rows) return;
  if (a.qo_indptr && (int64_t)row >= (int64_t)a.qo_indptr[a.batch] * a.H) return;  // past the call's tokens
  merge_row_half<false>(a.part_lse, a.part_o, a.rows_max, a.nsplit, row, half, lane, a.o, a.lse);
}

}  // namespace

int merge_blocks(int rows) { return (rows + kRowsPerBlock - 1) / kRowsPerBlock; }

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int blocks = merge_blocks(a.rows);
  if (blocks == 0) return cudaSuccess;
  merge_kernel<<<blocks, 64 * kRowsPerBlock, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlav
