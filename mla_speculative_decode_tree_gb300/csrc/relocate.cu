// KV relocation: each request's scattered prefix rows are copied into one
// contiguous block of free pool rows chosen by the caller, and kv_indices is
// rewritten to point at the copies.  This is the "live KV relocation" second
// tier of KV defragmentation the pages design and defer (move the rows,
// rewrite the indices) [The Art of Knowing When to Stop: Deferring Tier 1
// Defrag, §"The Decision: Why Tier 1 Defrag Gets Deferred"]; the first tier,
// a sorted free list, only shapes future allocations.
//
// Key k of the flat prefix index range [kv_indptr[0], kv_indptr[batch])
// belongs to the request b with kv_indptr[b] <= k < kv_indptr[b+1]; its row
// kv_indices[k] is copied whole (1152 bytes) to row dst_start[b] + (k -
// kv_indptr[b]), and kv_indices[k] becomes that row.  The destination rows
// must not be read by the same call (they are free rows): source and
// destination never overlap, so the copies may run in any order.
//
// The copy is a streaming gather/scatter bound by HBM: every source row is
// read once and every destination row written once, so loads and stores are
// marked streaming (evict-first) and each warp keeps kRows rows (4.5 KB) in
// flight; a row is 72 16-byte pieces, lane l moving pieces l, l+32 and (for
// l < 8) l+64.
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;                       // rows per warp per iteration
constexpr int kPieces = kRowBytes / 16;        // 16-byte pieces per row (72)
constexpr int kPerLane = (kPieces + 31) / 32;  // 3

// The request owning flat key k: the last b with kv_indptr[b] <= k.
__device__ __forceinline__ int owner_of(const int32_t* kv_indptr, int batch, int64_t k) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)kv_indptr[mid] <= k)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads) relocate_kernel(uint4* pool, const int32_t* kv_indptr,
                                                            int32_t* kv_indices, const int32_t* dst_start,
                                                            int batch, int64_t pool_rows, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int64_t k_begin = kv_indptr[0], k_end = kv_indptr[batch];
  constexpr int64_t kRowVec = kPieces;  // uint4 per row
  uint32_t bad = 0;
#pragma unroll 1
  for (int64_t base = k_begin + warp * kRows; base < k_end; base += nwarps * kRows) {
    // lane r < kRows resolves key base + r: source row, destination row
    int64_t src = -1, dst = -1;
    if (lane < kRows && base + lane < k_end) {
      const int64_t k = base + lane;
      const int b = owner_of(kv_indptr, batch, k);
      const int64_t s = kv_indices[k];
      const int64_t d = (int64_t)dst_start[b] + (k - kv_indptr[b]);
      if (s >= 0 && s < pool_rows && d >= 0 && d < pool_rows) {
        src = s;
        dst = d;
      } else {
        bad = 1;  // the key is left as it was
      }
    }
    int64_t s_r[kRows], d_r[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      s_r[r] = __shfl_sync(0xffffffffu, src, r);
      d_r[r] = __shfl_sync(0xffffffffu, dst, r);
    }
    uint4 v[kRows][kPerLane];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        const int p = lane + 32 * i;
        if (s_r[r] >= 0 && p < kPieces) v[r][i] = __ldcs(pool + s_r[r] * kRowVec + p);
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        const int p = lane + 32 * i;
        if (d_r[r] >= 0 && p < kPieces) __stcs(pool + d_r[r] * kRowVec + p, v[r][i]);
      }
    }
    if (lane < kRows && dst >= 0) kv_indices[base + lane] = (int32_t)dst;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && status) atomicOr(status, kStatusBadRow);
}

}  // namespace

cudaError_t launch_relocate(void* pool, const int32_t* kv_indptr, int32_t* kv_indices, const int32_t* dst_start,
                            int batch, int64_t pool_rows, int64_t max_keys, uint32_t* status, cudaStream_t stream) {
  if (batch <= 0 || max_keys <= 0) return cudaSuccess;
  int sms = 0, dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // enough warps for every key once, at most a full wave of 256-thread blocks
  const int64_t want = (max_keys + (int64_t)kRows * (kThreads / 32) - 1) / ((int64_t)kRows * (kThreads / 32));
  const int64_t cap = (int64_t)sms * (2048 / kThreads);
  const int grid = (int)(want < cap ? (want > 0 ? want : 1) : cap);
  relocate_kernel<<<grid, kThreads, 0, stream>>>(static_cast<uint4*>(pool), kv_indptr, kv_indices, dst_start, batch,
                                                   pool_rows, status);
  return cudaGetLastError();
}

}  // namespace mlav
