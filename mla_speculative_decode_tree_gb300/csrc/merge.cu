// Merge kernel: combines the nsplit partials of every query row by
// log-sum-exp -- the second reduction kernel of the split-K verify
// [Custom sm_120 Verify Kernel, §"Building the Custom Kernel: From Occupancy
// Starvation to Flash-Decode"].  The per-row arithmetic is merge_row_half or
// merge_row_quarter (merge_row.cuh), bit for bit that of the split kernel's
// fused merge.
#include "merge_row.cuh"

namespace mlav {
namespace {

// Two layouts.  Many rows (the grid spans several waves): two warps per row,
// one per half of the 512 latent columns, four rows per block -- more bytes in
// flight per thread for a merge bound by reading the partials.  At most one
// wave of rows: four warps per row, one per quarter of the columns, two rows
// per block -- shorter per-row latency for a merge bound by its round trips.
// Both compute the same bits (merge_row.cuh).
constexpr int kHalfRowsPerBlock = 4;
constexpr int kQuarterRowsPerBlock = 2;

__global__ void __launch_bounds__(64 * kHalfRowsPerBlock) merge_half_kernel(MergeArgs a) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // The split kernels of this call have finished (stream order): hand their
    // status bits to the "last call" word and reset the accumulator.
    const uint32_t st = a.status[0];
    if (st) atomicOr(a.status + 1, st);
    a.status[0] = 0u;
  }
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int row = blockIdx.x * kHalfRowsPerBlock + (warp >> 1);
  const int half = warp & 1;
  if (row >= a.rows) return;
  if (a.qo_indptr && (int64_t)row >= (int64_t)a.qo_indptr[a.batch] * a.H) return;  // past the call's tokens
  merge_row_half<false>(a.part_lse, a.part_o, a.rows_max, a.nsplit, row, half, lane, a.o, a.lse);
}

template <bool kSpec>
__global__ void __launch_bounds__(128 * kQuarterRowsPerBlock, 2) merge_quarter_kernel(MergeArgs a) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const uint32_t st = a.status[0];
    if (st) atomicOr(a.status + 1, st);
    a.status[0] = 0u;
  }
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int row = blockIdx.x * kQuarterRowsPerBlock + (warp >> 2);
  const int quarter = warp & 3;
  if (row >= a.rows) return;
  if (a.qo_indptr && (int64_t)row >= (int64_t)a.qo_indptr[a.batch] * a.H) return;  // past the call's tokens
  merge_row_quarter<kSpec>(a.part_lse, a.part_o, a.rows_max, a.nsplit, row, quarter, lane, a.o, a.lse);
}

}  // namespace

int merge_blocks(int rows, bool quarter) {
  const int per = quarter ? kQuarterRowsPerBlock : kHalfRowsPerBlock;
  return (rows + per - 1) / per;
}

// Quarter layout while its blocks (two rows each, two per SM) fit one wave.
bool merge_quarter_fits(int64_t rows, int sms) {
  return (rows + kQuarterRowsPerBlock - 1) / kQuarterRowsPerBlock <= 2 * (int64_t)sms;
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int blocks = merge_blocks(a.rows, a.quarter != 0);
  if (blocks == 0) return cudaSuccess;
  if (!a.quarter)
    merge_half_kernel<<<blocks, 64 * kHalfRowsPerBlock, 0, stream>>>(a);
  else if (a.speculative)
    merge_quarter_kernel<true><<<blocks, 128 * kQuarterRowsPerBlock, 0, stream>>>(a);
  else
    merge_quarter_kernel<false><<<blocks, 128 * kQuarterRowsPerBlock, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlav
