// Tree-mask builder: the packed visibility mask of a verify call, built on
// the device from the draft trees' parent arrays, so that the per-step mask
// build needs no host work and fits in the same CUDA graph as the verify
// call.  Building the tree and the mask on the host is a per-step cost the
// pages measured (small beside the kernel there) [Capture Safety to MoE
// Ceiling, §"Phase 2e: The Occupancy Epiphany and the 3-6x Speedup"]; the
// layout is the one the verify kernels read: request b's row-major
// [q_len, P_b + q_len] block of bits, LSB-first, starting at bit
// mask_indptr[b] [Custom sm_120 Verify Kernel, §"The Debugging Gauntlet"].
//
// Bit (i, j) of request b is 1 when j < P_b (every draft token sees the
// whole prefix) or when draft node j - P_b is node i or one of its
// ancestors.  Blocks of consecutive requests share bytes (a block is
// q_len * (P_b + q_len) bits), so each thread owns whole output bytes and no
// two threads write the same byte.
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kThreads = 256;

// First bit of request b's block: q_len * sum_{b' < b} (P_b' + q_len).
__device__ __forceinline__ int64_t block_start(const int32_t* kv_indptr, int b, int T) {
  return (int64_t)T * (((int64_t)kv_indptr[b] - kv_indptr[0]) + (int64_t)b * T);
}

// Request whose block holds bit g: the last b with block_start(b) <= g.
__device__ __forceinline__ int request_of(const int32_t* kv_indptr, int batch, int T, int64_t g) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (block_start(kv_indptr, mid, T) <= g)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

constexpr int kMaxStaged = 4;  // requests whose trees one block stages in shared memory

__global__ void __launch_bounds__(kThreads) tree_mask_kernel(const int32_t* __restrict__ parents,
                                                            const int32_t* __restrict__ kv_indptr, int batch,
                                                            int T, uint8_t* __restrict__ mask, int64_t mask_bytes,
                                                            int32_t* __restrict__ mask_indptr) {
  __shared__ int32_t s_par[kMaxStaged][kMaxQLen];
  const int64_t total_bits = block_start(kv_indptr, batch, T);
  int64_t nbytes = (total_bits + 7) / 8;
  if (nbytes > mask_bytes) nbytes = mask_bytes;
  // Every thread of a block runs the same iterations (the loop bound is per
  // block), so the block can stage the parent arrays of the requests its
  // bytes fall in; with more than kMaxStaged of them the walk reads global
  // memory.
  for (int64_t base = (int64_t)blockIdx.x * kThreads; base < nbytes; base += (int64_t)gridDim.x * kThreads) {
    const int64_t k = base + threadIdx.x;
    const int64_t last_byte = (base + kThreads < nbytes ? base + kThreads : nbytes) - 1;
    const int b_lo = request_of(kv_indptr, batch, T, 8 * base);
    const int64_t last_bit = (8 * last_byte + 7 < total_bits ? 8 * last_byte + 7 : total_bits - 1);
    const int b_hi = request_of(kv_indptr, batch, T, last_bit);
    const bool staged = b_hi - b_lo < kMaxStaged;
    __syncthreads();  // the previous iteration's walks are done with s_par
    if (staged)
      for (int x = threadIdx.x; x < (b_hi - b_lo + 1) * T; x += kThreads)
        s_par[x / T][x % T] = __ldg(parents + (int64_t)(b_lo + x / T) * T + x % T);
    __syncthreads();
    if (k >= nbytes) continue;

    int b = request_of(kv_indptr, batch, T, 8 * k);
    int64_t start = block_start(kv_indptr, b, T);
    int64_t next = block_start(kv_indptr, b + 1, T);
    uint32_t byte = 0;
    for (int e = 0; e < 8; ++e) {
      const int64_t g = 8 * k + e;
      if (g >= total_bits) break;
      while (g >= next && b < batch - 1) {  // a block can end inside this byte
        ++b;
        start = next;
        next = block_start(kv_indptr, b + 1, T);
      }
      // (the clamps only matter for a kv_indptr that decreases, which the
      // contract excludes; they keep every access in bounds)
      const int64_t P = (int64_t)kv_indptr[b + 1] - kv_indptr[b] > 0 ? (int64_t)kv_indptr[b + 1] - kv_indptr[b] : 0;
      const int64_t L = P + T;
      const int64_t off = g - start > 0 ? g - start : 0;
      int i = (int)(off / L);
      if (i > T - 1) i = T - 1;
      const int64_t j = off - (int64_t)i * L;
      uint32_t bit = 1;
      if (j >= P) {
        // Is draft node d = j - P the node i or an ancestor of it?  The walk
        // follows parent links (parent < node); an out-of-range link ends it.
        const int d = (int)(j - P);
        const bool in_smem = staged && b >= b_lo && b <= b_hi;
        const int32_t* gpar = parents + (int64_t)b * T;
        bit = 0;
        int n = i;
        for (int step = 0; step <= T && n >= 0; ++step) {
          if (n == d) {
            bit = 1;
            break;
          }
          const int p = in_smem ? s_par[b - b_lo][n] : __ldg(gpar + n);
          n = (p >= 0 && p < n) ? p : -1;
        }
      }
      byte |= bit << e;
    }
    mask[k] = (uint8_t)byte;
  }
  // Bit offsets of the requests' blocks.
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < batch; b += (int64_t)gridDim.x * blockDim.x)
    mask_indptr[b] = (int32_t)block_start(kv_indptr, (int)b, T);
}

}  // namespace

cudaError_t launch_tree_mask(const int32_t* parents, const int32_t* kv_indptr, int batch, int T, uint8_t* mask,
                             int64_t mask_bytes, int32_t* mask_indptr, int64_t max_bytes, cudaStream_t stream) {
  // Fixed grid (from the plan's bounds, not the lengths on the device); the
  // grid-stride loop covers any length up to mask_bytes.
  int64_t blocks = (max_bytes + kThreads - 1) / kThreads;
  if (blocks < 1) blocks = 1;
  if (blocks > 4 * 152) blocks = 4 * 152;
  tree_mask_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(parents, kv_indptr, batch, T, mask, mask_bytes,
                                                              mask_indptr);
  return cudaGetLastError();
}

}  // namespace mlav
