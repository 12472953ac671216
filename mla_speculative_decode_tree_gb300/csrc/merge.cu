// Merge kernel: combines the nsplit partials of every query row by
// log-sum-exp -- the second reduction kernel of the split-K verify
// [Custom sm_120 Verify Kernel, §"Building the Custom Kernel: From Occupancy
// Starvation to Flash-Decode"].
//
//   M = max_s lse_s,  w_s = exp(lse_s - M),
//   O = sum_s w_s O_s / sum_s w_s  (bf16, round-to-nearest-even),
//   LSE = M + ln sum_s w_s;        M = -inf  ->  O = 0, LSE = -inf.
//
// Two warps per row, one per half of the 512 latent columns; lane l owns 8
// columns of its half.  The lanes first take one split each (lse, weight),
// then the warp walks the splits kUnroll at a time with all their loads in
// flight, the weights broadcast by shuffle.  Splits with lse_s = -inf (empty
// chunk or nothing visible) are skipped without touching their O_s, which the
// split kernel does not write.
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kRowsPerBlock = 4;
constexpr int kUnroll = 8;  // divides 32

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

  float M = -INFINITY;
  for (int s = lane; s < a.nsplit; s += 32) M = fmaxf(M, a.part_lse[(int64_t)s * a.rows_max + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  const int col = half * (kDLatent / 2) + 8 * lane;
  uint4* o = reinterpret_cast<uint4*>(a.o + (int64_t)row * kDLatent + col);
  if (M == -INFINITY) {
    *o = make_uint4(0, 0, 0, 0);
    if (half == 0 && lane == 0) a.lse[row] = -INFINITY;
    return;
  }

  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
  float W = 0.f;
  const int64_t split_stride = a.rows_max * kDLatent;
  const float* base = a.part_o + (int64_t)row * kDLatent + col;
  for (int s0 = 0; s0 < a.nsplit; s0 += 32) {
    const int s = s0 + lane;
    const float ls = s < a.nsplit ? a.part_lse[(int64_t)s * a.rows_max + row] : -INFINITY;
    const float wl = ls == -INFINITY ? 0.f : expf(ls - M);
    W += wl;
    const int n = (a.nsplit - s0 < 32) ? a.nsplit - s0 : 32;
    for (int k0 = 0; k0 < n; k0 += kUnroll) {
      float wk[kUnroll];
      float4 v[kUnroll][2];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        wk[u] = __shfl_sync(0xffffffffu, wl, k0 + u);  // 0 past the last split
        if (wk[u] != 0.f) {
          const float4* src = reinterpret_cast<const float4*>(base + (int64_t)(s0 + k0 + u) * split_stride);
          v[u][0] = src[0];
          v[u][1] = src[1];
        } else {
          v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        acc[0] = fmaf(wk[u], v[u][0].x, acc[0]);
        acc[1] = fmaf(wk[u], v[u][0].y, acc[1]);
        acc[2] = fmaf(wk[u], v[u][0].z, acc[2]);
        acc[3] = fmaf(wk[u], v[u][0].w, acc[3]);
        acc[4] = fmaf(wk[u], v[u][1].x, acc[4]);
        acc[5] = fmaf(wk[u], v[u][1].y, acc[5]);
        acc[6] = fmaf(wk[u], v[u][1].z, acc[6]);
        acc[7] = fmaf(wk[u], v[u][1].w, acc[7]);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
  const float inv = 1.f / W;
  uint32_t packed[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * k] * inv, acc[2 * k + 1] * inv);
    packed[k] = *reinterpret_cast<uint32_t*>(&h2);
  }
  *o = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  if (half == 0 && lane == 0) a.lse[row] = M + logf(W);
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
