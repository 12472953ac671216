// Merge kernel: combines the nsplit partials of every query row by
// log-sum-exp -- the second reduction kernel of the split-K verify
// [Custom sm_120 Verify Kernel, §"Building the Custom Kernel: From Occupancy
// Starvation to Flash-Decode"].
//
//   M = max_s lse_s,  w_s = exp(lse_s - M),
//   O = sum_s w_s O_s / sum_s w_s  (bf16, round-to-nearest-even),
//   LSE = M + ln sum_s w_s;        M = -inf  ->  O = 0, LSE = -inf.
//
// One warp per row; lane l owns latent columns [16l, 16l+16).  Splits with
// lse_s = -inf (empty chunk or nothing visible) are skipped without touching
// their O_s, which the split kernel does not write.
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kRowsPerBlock = 8;

__global__ void __launch_bounds__(32 * kRowsPerBlock) merge_kernel(MergeArgs a) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // The split kernels of this call have finished (stream order): hand their
    // status bits to the "last call" word and reset the accumulator.
    const uint32_t st = a.status[0];
    if (st) atomicOr(a.status + 1, st);
    a.status[0] = 0u;
  }
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= a.rows) return;

  float M = -INFINITY;
  for (int s = lane; s < a.nsplit; s += 32) M = fmaxf(M, a.part_lse[(int64_t)s * a.rows_max + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  uint4* o = reinterpret_cast<uint4*>(a.o + (int64_t)row * kDLatent) + 2 * lane;
  if (M == -INFINITY) {
    o[0] = make_uint4(0, 0, 0, 0);
    o[1] = make_uint4(0, 0, 0, 0);
    if (lane == 0) a.lse[row] = -INFINITY;
    return;
  }

  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float W = 0.f;
  for (int s = 0; s < a.nsplit; ++s) {
    const float ls = a.part_lse[(int64_t)s * a.rows_max + row];
    if (ls == -INFINITY) continue;
    const float w = expf(ls - M);
    W += w;
    const float4* src = reinterpret_cast<const float4*>(a.part_o + ((int64_t)s * a.rows_max + row) * kDLatent) +
                        4 * lane;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = src[q];
      acc[4 * q + 0] = fmaf(w, v.x, acc[4 * q + 0]);
      acc[4 * q + 1] = fmaf(w, v.y, acc[4 * q + 1]);
      acc[4 * q + 2] = fmaf(w, v.z, acc[4 * q + 2]);
      acc[4 * q + 3] = fmaf(w, v.w, acc[4 * q + 3]);
    }
  }
  const float inv = 1.f / W;
  uint32_t packed[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * k] * inv, acc[2 * k + 1] * inv);
    packed[k] = *reinterpret_cast<uint32_t*>(&h2);
  }
  o[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  o[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  if (lane == 0) a.lse[row] = M + logf(W);
}

}  // namespace

int merge_blocks(int rows) { return (rows + kRowsPerBlock - 1) / kRowsPerBlock; }

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int blocks = merge_blocks(a.rows);
  if (blocks == 0) return cudaSuccess;
  merge_kernel<<<blocks, 32 * kRowsPerBlock, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlav
