// mla_verify_run_noalloc: the verify call for callers that cannot allocate
// device memory.  The split partials live in a fixed scratch array compiled
// into the library instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mla_verify.h"
#include "common.cuh"

namespace mlav {
int record_cuda_error(cudaError_t e);  // api.cu: keeps the text for mla_verify_strerror
size_t plan_zero_bytes(const mla_verify_plan_s* pl);  // api.cu: header + merge counters
}

namespace {

// Every device that loads the library reserves this much global memory for
// as long as the process lives.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array, looked up once per device.  In host code the
// array's name is only a host-side stand-in, never a usable device pointer.
std::mutex g_mu;
void* g_scratch_ptr[64];

int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mlav::record_cuda_error(e);
  if (dev < 0 || dev >= 64) return MLA_VERIFY_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // with `dev` current
    if (e != cudaSuccess) return mlav::record_cuda_error(e);
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MLA_VERIFY_OK;
}

}  // namespace

extern "C" int mla_verify_run_noalloc(mla_verify_plan_t plan, const void* q_nope_absorbed, const void* q_rope,
                                      const void* kv_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                                      const int32_t* out_cache_loc, const uint8_t* custom_mask,
                                      const int32_t* mask_indptr, int32_t batch, float sm_scale, int32_t nsplit,
                                      void* o, float* lse, void* stream) {
  mla_verify_plan_info info;
  int rc = mla_verify_plan_describe(plan, &info);
  if (rc != MLA_VERIFY_OK) return rc;
  if (info.workspace_bytes > kNoAllocScratchBytes) return MLA_VERIFY_EWORKSPACE;
  void* scratch = nullptr;
  if ((rc = scratch_for_current_device(&scratch)) != MLA_VERIFY_OK) return rc;
  // The array keeps the previous call's contents; its status header (and a
  // fused merge's counters) must start at zero for this call (the partials
  // are rewritten in full).
  cudaError_t e = cudaMemsetAsync(scratch, 0, mlav::plan_zero_bytes(plan), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return mlav::record_cuda_error(e);
  return mla_verify_run(plan, q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, out_cache_loc, custom_mask,
                        mask_indptr, batch, sm_scale, nsplit, scratch, kNoAllocScratchBytes, o, lse, stream);
}
