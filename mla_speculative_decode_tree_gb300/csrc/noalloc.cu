// mla_verify_run_noalloc: the verify call for callers that cannot allocate
// device memory.  The split partials live in a fixed scratch array compiled
// into the library instead of a caller-provided workspace.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mla_verify.h"
#include "common.cuh"

namespace mlav {
int record_cuda_error(cudaError_t e);                 // api.cu: keeps the text for mla_verify_strerror
size_t plan_zero_bytes(const mla_verify_plan_s* pl);  // api.cu: header + merge counters
size_t plan_workspace_bytes(const mla_verify_plan_s* pl);
int check_run_args(const mla_verify_plan_s* pl, const void* q_nope_absorbed, const void* q_rope,
                   const void* kv_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                   const int32_t* out_cache_loc, const uint8_t* custom_mask, const int32_t* mask_indptr,
                   int32_t batch, float sm_scale, int32_t nsplit, const void* o, const float* lse);
}  // namespace mlav

namespace {

// Every device that loads the library reserves this much global memory for
// as long as the process lives.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address belongs to the CUDA context that loaded the
// library's module, so it is looked up once per context (keyed by the
// context's unique ID: a context created later -- by another host plugin,
// or after cudaDeviceReset -- gets its own lookup).  In host code the array's
// name is only a host-side stand-in, never a usable device pointer.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
constexpr int kMaxContexts = 64;
std::mutex g_mu;
CtxGetCurrentFn g_get_current = nullptr;
CtxGetIdFn g_get_id = nullptr;
unsigned long long g_ctx_id[kMaxContexts];
void* g_ctx_ptr[kMaxContexts];
int g_nctx = 0;

int driver_fn(const char* name, void** fn) {
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess) return mlav::record_cuda_error(e);
  return (q == cudaDriverEntryPointSuccess && *fn) ? MLA_VERIFY_OK : MLA_VERIFY_EUNSUPPORTED;
}

int scratch_for_current_context(void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  int rc;
  if (!g_get_current) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    if ((rc = driver_fn("cuCtxGetCurrent", &f1)) != MLA_VERIFY_OK) return rc;
    if ((rc = driver_fn("cuCtxGetId", &f2)) != MLA_VERIFY_OK) return rc;
    g_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    g_get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  // The context current to this thread (a caller's own driver context, or
  // the device's primary context).  With none current yet, the symbol lookup
  // below makes the runtime bind the device's primary context first.
  CUcontext ctx = nullptr;
  void* p = nullptr;
  if (g_get_current(&ctx) != CUDA_SUCCESS) return MLA_VERIFY_ECUDA;
  if (!ctx) {
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return mlav::record_cuda_error(e);
    if (g_get_current(&ctx) != CUDA_SUCCESS || !ctx) return MLA_VERIFY_ECUDA;
  }
  unsigned long long id = 0;
  if (g_get_id(ctx, &id) != CUDA_SUCCESS) return MLA_VERIFY_ECUDA;
  for (int i = 0; i < g_nctx; ++i)
    if (g_ctx_id[i] == id) {
      *out = g_ctx_ptr[i];
      return MLA_VERIFY_OK;
    }
  if (g_nctx == kMaxContexts) return MLA_VERIFY_EUNSUPPORTED;
  if (!p) {
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // in the current context
    if (e != cudaSuccess) return mlav::record_cuda_error(e);
  }
  g_ctx_id[g_nctx] = id;
  g_ctx_ptr[g_nctx] = p;
  ++g_nctx;
  *out = p;
  return MLA_VERIFY_OK;
}

}  // namespace

extern "C" int mla_verify_run_noalloc(mla_verify_plan_t plan, const void* q_nope_absorbed, const void* q_rope,
                                      const void* kv_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                                      const int32_t* out_cache_loc, const uint8_t* custom_mask,
                                      const int32_t* mask_indptr, int32_t batch, float sm_scale, int32_t nsplit,
                                      void* o, float* lse, void* stream) {
  // The same checks as mla_verify_run, before the shared array is touched: a
  // rejected call must not disturb a call still running on another stream.
  int rc = mlav::check_run_args(plan, q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, out_cache_loc,
                                custom_mask, mask_indptr, batch, sm_scale, nsplit, o, lse);
  if (rc != MLA_VERIFY_OK || batch == 0) return rc;
  if (mlav::plan_workspace_bytes(plan) > kNoAllocScratchBytes) return MLA_VERIFY_EWORKSPACE;
  void* scratch = nullptr;
  if ((rc = scratch_for_current_context(&scratch)) != MLA_VERIFY_OK) return rc;
  // The array keeps the previous call's contents; its status header (and a
  // fused merge's counters) must start at zero for this call (the partials
  // are rewritten in full).
  cudaError_t e = cudaMemsetAsync(scratch, 0, mlav::plan_zero_bytes(plan), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return mlav::record_cuda_error(e);
  return mla_verify_run(plan, q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, out_cache_loc, custom_mask,
                        mask_indptr, batch, sm_scale, nsplit, scratch, kNoAllocScratchBytes, o, lse, stream);
}
