// Tree-mask builder: the packed visibility mask of a verify call, built on
// the device from the draft trees' parent arrays, so that the per-step mask
// build needs no host work and fits in the same CUDA graph as the verify
// call.  Building the tree and the mask on the host is a per-step cost the
// pages measured (small beside the kernel there) [Capture Safety to MoE
// Ceiling, §"Phase 2e: The Occupancy Epiphany and the 3-6x Speedup"]; the
// layout is the one the verify kernels read: request b's row-major
// [T_b, P_b + T_b] block of bits, LSB-first, starting at bit mask_indptr[b]
// [Custom sm_120 Verify Kernel, §"The Debugging Gauntlet"].  T_b is the
// plan's q_len, or in a varlen call qo_indptr[b+1] - qo_indptr[b], whose
// parents then sit at parents[qo_indptr[b] ..].
//
// Bit (i, j) of request b is 1 when j < P_b (every draft token sees the
// whole prefix) or when draft node j - P_b is node i or one of its
// ancestors.  Blocks of consecutive requests share bytes (a block is
// T_b * (P_b + T_b) bits), so each thread owns whole output bytes and no
// two threads write the same byte.
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxStaged = 4;  // requests whose trees one block stages in shared memory

// Where request b's block starts, its draft count and its parents: closed
// forms for a uniform q_len, a table in shared memory for a varlen call.
struct Layout {
  const int32_t* kv_indptr;
  const int32_t* qo_indptr;  // null: uniform
  const int64_t* s_start;    // varlen: first bit of each block, [batch+1]
  int T;                     // the plan's q_len
  __device__ __forceinline__ int64_t start(int b) const {
    if (qo_indptr) return s_start[b];
    return (int64_t)T * (((int64_t)kv_indptr[b] - kv_indptr[0]) + (int64_t)b * T);
  }
  __device__ __forceinline__ int count(int b) const {
    if (!qo_indptr) return T;
    const int t = qo_indptr[b + 1] - qo_indptr[b];
    return t < 0 ? 0 : (t > T ? T : t);  // the contract keeps 0 <= T_b <= q_len
  }
  __device__ __forceinline__ int64_t parent_base(int b) const {
    return qo_indptr ? (int64_t)qo_indptr[b] : (int64_t)b * T;
  }
  __device__ __forceinline__ int64_t prefix(int b) const {
    const int64_t P = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
    return P > 0 ? P : 0;  // (a decreasing kv_indptr is outside the contract)
  }
  // The request whose block holds bit g: the last b with start(b) <= g.
  __device__ __forceinline__ int request_of(int batch, int64_t g) const {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (start(mid) <= g)
        lo = mid;
      else
        hi = mid - 1;
    }
    return lo;
  }
};

__global__ void __launch_bounds__(kThreads) tree_mask_kernel(const int32_t* __restrict__ parents,
                                                            const int32_t* __restrict__ kv_indptr,
                                                            const int32_t* __restrict__ qo_indptr, int batch,
                                                            int T, uint8_t* __restrict__ mask, int64_t mask_bytes,
                                                            int32_t* __restrict__ mask_indptr) {
  __shared__ int32_t s_par[kMaxStaged][kMaxQLen];
  __shared__ int64_t s_start[kMaxTreeMaskVarlenBatch + 1];
  if (qo_indptr) {
    if (threadIdx.x == 0) {
      int64_t acc = 0;
      for (int b = 0; b < batch; ++b) {
        s_start[b] = acc;
        int t = qo_indptr[b + 1] - qo_indptr[b];
        t = t < 0 ? 0 : (t > T ? T : t);
        int64_t P = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
        P = P > 0 ? P : 0;
        acc += (int64_t)t * (P + t);
      }
      s_start[batch] = acc;
    }
    __syncthreads();
  }
  const Layout lay{kv_indptr, qo_indptr, s_start, T};
  const int64_t total_bits = lay.start(batch);
  int64_t nbytes = (total_bits + 7) / 8;
  if (nbytes > mask_bytes) nbytes = mask_bytes;
  // Every thread of a block runs the same iterations (the loop bound is per
  // block), so the block can stage the parent arrays of the requests its
  // bytes fall in; with more than kMaxStaged of them the walk reads global
  // memory.
  for (int64_t base = (int64_t)blockIdx.x * kThreads; base < nbytes; base += (int64_t)gridDim.x * kThreads) {
    const int64_t k = base + threadIdx.x;
    const int64_t last_byte = (base + kThreads < nbytes ? base + kThreads : nbytes) - 1;
    const int b_lo = lay.request_of(batch, 8 * base);
    const int64_t last_bit = (8 * last_byte + 7 < total_bits ? 8 * last_byte + 7 : total_bits - 1);
    const int b_hi = lay.request_of(batch, last_bit);
    const bool staged = b_hi - b_lo < kMaxStaged;
    __syncthreads();  // the previous iteration's walks are done with s_par
    if (staged)
      for (int x = threadIdx.x; x < (b_hi - b_lo + 1) * T; x += kThreads) {
        const int r = b_lo + x / T, n = x % T;
        if (n < lay.count(r)) s_par[x / T][n] = __ldg(parents + lay.parent_base(r) + n);
      }
    __syncthreads();
    if (k >= nbytes) continue;

    int b = lay.request_of(batch, 8 * k);
    int64_t start = lay.start(b);
    int64_t next = lay.start(b + 1);
    uint32_t byte = 0;
    for (int e = 0; e < 8; ++e) {
      const int64_t g = 8 * k + e;
      if (g >= total_bits) break;
      while (g >= next && b < batch - 1) {  // a block can end inside this byte
        ++b;
        start = next;
        next = lay.start(b + 1);
      }
      const int Tb = lay.count(b);
      if (Tb == 0) continue;  // (only a degenerate layout reaches here)
      const int64_t P = lay.prefix(b);
      const int64_t L = P + Tb;
      const int64_t off = g - start > 0 ? g - start : 0;
      int i = (int)(off / L);
      if (i > Tb - 1) i = Tb - 1;
      const int64_t j = off - (int64_t)i * L;
      uint32_t bit = 1;
      if (j >= P) {
        // Is draft node d = j - P the node i or an ancestor of it?  The walk
        // follows parent links (parent < node); an out-of-range link ends it.
        const int d = (int)(j - P);
        const bool in_smem = staged && b >= b_lo && b <= b_hi;
        const int32_t* gpar = parents + lay.parent_base(b);
        bit = 0;
        int n = i;
        for (int step = 0; step <= Tb && n >= 0; ++step) {
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
    mask_indptr[b] = (int32_t)lay.start((int)b);
}

}  // namespace

cudaError_t launch_tree_mask(const int32_t* parents, const int32_t* kv_indptr, const int32_t* qo_indptr, int batch,
                             int T, uint8_t* mask, int64_t mask_bytes, int32_t* mask_indptr, int64_t max_bytes,
                             cudaStream_t stream) {
  // Fixed grid (from the plan's bounds, not the lengths on the device); the
  // grid-stride loop covers any length up to mask_bytes.
  int64_t blocks = (max_bytes + kThreads - 1) / kThreads;
  if (blocks < 1) blocks = 1;
  if (blocks > 4 * 152) blocks = 4 * 152;
  tree_mask_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(parents, kv_indptr, qo_indptr, batch, T, mask,
                                                              mask_bytes, mask_indptr);
  return cudaGetLastError();
}

}  // namespace mlav
