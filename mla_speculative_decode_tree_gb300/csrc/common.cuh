// Shared definitions of the MLA tree-verify kernels (device and host side).
#pragma once

#include <cuda.h>  // CUtensorMap (type only; encoding goes through the runtime's driver entry point)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mlav {

constexpr int kDLatent = 512;
constexpr int kDRope = 64;
constexpr int kDRow = kDLatent + kDRope;  // 576 bf16 = 1152 bytes per pool row
constexpr int kRowBytes = kDRow * 2;
constexpr int kKeysPerTile = 128;         // keys per pipeline tile
constexpr int kHalfTile = 64;             // finest chunk granule: a chunk may end in a half tile
constexpr int kMinChunk = 128;
constexpr int kMaxQLen = 64;
constexpr int kWsHeader = 256;            // bytes: [0] status accumulated by split, [1] status of the last merge

// Status bits (mirror MLA_VERIFY_DEV_* in mla_verify.h).
constexpr uint32_t kStatusBadRow = 0x1u;
constexpr uint32_t kStatusTimeout = 0x2u;

struct SplitArgs {
  const __nv_bfloat16* q_nope;   // [B*T, H, 512]
  const __nv_bfloat16* q_rope;   // [B*T, H, 64]
  const __nv_bfloat16* kv_pool;  // [pool_rows, 576]
  const int32_t* kv_indptr;      // [B+1]
  const int32_t* kv_indices;
  const int32_t* out_cache_loc;  // [B*T]
  const uint8_t* mask;           // packed bits LSB-first
  const int32_t* mask_indptr;    // [B] bit offsets
  const int32_t* qo_indptr;      // [B+1] first token row of each request, or null: request b owns
                                 // token rows b*T .. b*T+T-1 (T = the plan's q_len, the maximum)
  int32_t batch, H, T, nsplit;
  int32_t min_chunk;             // shortest chunk (keys, a multiple of chunk_granule) for any request
  int32_t chunk_granule;         // chunk lengths are multiples of it: kKeysPerTile or kHalfTile
  int32_t test_stall;            // test only: the gather never signals block 0 (waits time out)
  int64_t pool_rows;
  int64_t rows_max;              // max_batch*T*H: row stride of one split's partials
  float scale_log2;              // sm_scale * log2(e): scores are kept in base 2
  float* part_lse;               // [nsplit, rows_max]   natural log, -inf when nothing visible
  float* part_o;                 // [nsplit, rows_max, 512] normalised partial output
  uint32_t* status;              // workspace header word 0
  // Fused merge (tensor-core kernel only; null when the merge kernel runs):
  // one arrival counter per (request, row group), zero between calls, and the
  // final outputs the last CTA of a group writes.
  uint32_t* merge_count;         // [max_batch, groups]
  __nv_bfloat16* o;              // [rows, 512]
  float* lse;                    // [rows]
};

// TMA descriptors of one call: the pool for row gathers (box 64 columns x 1
// row, 128-byte swizzle) and the two query tensors (box 64 columns x NQ rows).
struct TcMaps {  // CUtensorMap carries its own (64-byte or larger) alignment
  CUtensorMap kv, qn, qr;
};

struct MergeArgs {
  int32_t rows;      // batch*T*H rows (the most a call can have)
  const int32_t* qo_indptr;  // null, or [batch+1]: only rows below qo_indptr[batch]*H exist
  int32_t batch, H;
  int32_t nsplit;
  int64_t rows_max;
  const float* part_lse;
  const float* part_o;
  __nv_bfloat16* o;  // [rows, 512]
  float* lse;        // [rows]
  uint32_t* status;  // header words 0 (accumulated) and 1 (last call)
  int32_t quarter;      // four warps per row (few rows) instead of two
  int32_t speculative;  // quarter layout: load the first 16 splits' partials before their LSEs
};

// Key range of split s for a request with L keys: [s*chunk, min(L,(s+1)*chunk)),
// with chunk = ceil(L/nsplit) rounded up to the plan's granule and at least
// min_chunk (a multiple of the granule fixed by the plan, at least kMinChunk).
// The granule is a power of two.
__host__ __device__ inline int64_t chunk_len(int64_t L, int nsplit, int64_t min_chunk, int granule = kKeysPerTile) {
  int64_t per = (L + nsplit - 1) / nsplit;
  int64_t c = (per + granule - 1) & ~(int64_t)(granule - 1);
  return c < min_chunk ? min_chunk : c;
}

#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar`.  Gives up after ~kWaitLimitNs of
// wall time or 2^30 polls, whichever comes first, or as soon as another
// thread of the CTA has raised *abort.  On giving up it raises *abort and the
// timeout status bit and returns false; callers then skip the rest of their
// work so every thread reaches the teardown.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) break;
    }
  }
  *abort = 1;
  atomicOr(status, kStatusTimeout);
  return false;
}

// Non-blocking test of phase `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait for a single latency-critical thread: polls without suspending
// (a suspended waiter wakes up later than a polling one), same limits and
// abort behaviour.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               uint32_t* status) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) break;
    }
  }
  *abort = 1;
  atomicOr(status, kStatusTimeout);
  return false;
}

// ---- cp.async (16-byte, L2-only), zero-filled when src_bytes == 0 ----------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival is counted in the barrier's initial count).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- index helpers --------------------------------------------------------
// Token rows of request b: the first one (q0) and how many (at most T).
struct RequestTokens {
  int64_t q0;
  int n;
};
__device__ __forceinline__ RequestTokens request_tokens(const SplitArgs& a, int b) {
  if (!a.qo_indptr) return {(int64_t)b * a.T, a.T};
  const int64_t q0 = a.qo_indptr[b];
  int64_t n = (int64_t)a.qo_indptr[b + 1] - q0;
  n = n < 0 ? 0 : (n > a.T ? a.T : n);  // the contract bounds T_b by q_len
  return {q0, (int)n};
}

// Pool row of key position j of a request (prefix from kv_indices, drafts
// from out_cache_loc at the request's token rows q0..); -1 when it lies
// outside [0, pool_rows).
__device__ __forceinline__ int64_t resolve_row(const SplitArgs& a, int64_t q0, int64_t P, int64_t kv_base,
                                               int64_t j) {
  int64_t r = (j < P) ? (int64_t)__ldg(a.kv_indices + kv_base + j)
                      : (int64_t)__ldg(a.out_cache_loc + q0 + (j - P));
  return (r >= 0 && r < a.pool_rows) ? r : -1;
}

// The raw index entry of key position j (no range check): lets a caller issue
// the load early and check it when the value is used.
__device__ __forceinline__ int32_t load_row_id(const SplitArgs& a, int64_t q0, int64_t P, int64_t kv_base,
                                               int64_t j) {
  return (j < P) ? __ldg(a.kv_indices + kv_base + j) : __ldg(a.out_cache_loc + q0 + (j - P));
}

__device__ __forceinline__ uint32_t mask_bit(const uint8_t* mask, int64_t bit) {
  return (__ldg(mask + (bit >> 3)) >> (bit & 7)) & 1u;
}

#endif  // __CUDACC__

// Host launchers (defined in the kernel translation units).
cudaError_t launch_split_simt(const SplitArgs& a, dim3 grid, cudaStream_t stream);
// resident: whole-tile mode (NQ <= 64; the 96-row launcher refuses it).
#define MLAV_DECLARE_TC(NQ)                                                                            \
  cudaError_t launch_split_tc_##NQ(const SplitArgs& a, const TcMaps& m, dim3 grid, cudaStream_t stream, \
                                   bool resident);                                                     \
  int split_tc_smem_##NQ(bool resident);
MLAV_DECLARE_TC(16)
MLAV_DECLARE_TC(32)
MLAV_DECLARE_TC(48)
MLAV_DECLARE_TC(64)
MLAV_DECLARE_TC(96)
#undef MLAV_DECLARE_TC
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);
constexpr int kMaxTreeMaskVarlenBatch = 1024;  // requests of a varlen mask build
cudaError_t launch_tree_mask(const int32_t* parents, const int32_t* kv_indptr, const int32_t* qo_indptr, int batch,
                             int T, uint8_t* mask, int64_t mask_bytes, int32_t* mask_indptr, int64_t max_bytes,
                             cudaStream_t stream);
cudaError_t launch_relocate(void* pool, const int32_t* kv_indptr, int32_t* kv_indices, const int32_t* dst_start,
                            int batch, int64_t pool_rows, int64_t max_keys, uint32_t* status, cudaStream_t stream);
int merge_blocks(int rows, bool quarter);
bool merge_quarter_fits(int64_t rows, int sms);

constexpr int kSimtRowsPerCta = 8;  // one warp per query row

}  // namespace mlav
