// C ABI of libmlaverify.so (declared in include/mla_verify.h): argument
// checks, plan choices, workspace sizing and the two launches per call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/mla_verify.h"
#include "common.cuh"

using namespace mlav;

struct mla_verify_plan_s {
  mla_verify_params p;
  int kernel;  // 1 = tcgen05, 0 = CUDA cores
  int nq;      // query rows per split CTA
  bool resident;  // tensor-core kernel in resident-tile mode (each key lands once per CTA)
  int groups;  // row groups per request
  int64_t rows_max;
  bool fused;  // the split kernel merges (MLA_VERIFY_FUSED_MERGE on the tensor-core kernel)
  int splits;  // KV chunks per request = grid dimension = partials per row (nsplit, or the plan's count)
  int min_chunk;  // shortest chunk of any request (keys)
  int chunk_granule;  // chunk lengths are multiples of it (keys)
  size_t off_cnt, off_lse, off_o, ws_bytes;  // [0, off_lse) must be zero between calls
  int merge_blocks;
  bool merge_quarter;  // merge with four warps per row (at most one wave of rows)
  int smem;
};

namespace {

thread_local char g_cuda_msg[256] = "CUDA error";

int cuda_fail(cudaError_t e) {
  std::snprintf(g_cuda_msg, sizeof g_cuda_msg, "CUDA error %d (%s): %s", (int)e, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return MLA_VERIFY_ECUDA;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Row-group sizes of the tensor-core kernel (resident mode: at most 64).
const int kNqChoices[] = {16, 32, 48, 64, 96};
constexpr int kMaxResidentNq = 64;

// SMs of the current device (152 on GB300, also when no device can be asked).
int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0) {
    (void)cudaGetLastError();
    return 152;
  }
  return n;
}

// Time model of a split launch, from measurements on GB300 (clocks at
// 2070 MHz).  A CTA is bound by landing its gathered blocks, not by its MMAs:
// a 128-key tile takes ~5.1 us when it stays resident (one landing per key,
// but each tile waits out its own landing), and ~5.3-5.9 us when the value
// blocks are fetched a second time through the ring (17 blocks at ~0.34 us;
// larger row groups leave fewer ring slots beside Q).  A CTA adds ~5 us of
// start-up, first landing and epilogue; the merge reads each written partial
// (2 KB per row) at ~3 TB/s after a ~2 us launch.  One request: CTAs of equal
// length run in waves of one per SM.  Several requests (lengths unknown at
// plan time, taken as half of max_kv_len on average): the CTAs are
// list-scheduled, so the time is about the work per SM plus one chunk of the
// longest request.
double tile_us(bool resident, int nq) { return resident ? 5.1 : nq >= 96 ? 5.9 : nq >= 64 ? 5.6 : 5.3; }

double est_us(int64_t rows_b, int64_t max_kv_len, int max_batch, int nsplit, int nq, bool resident, double sms) {
  constexpr double kCtaUs = 5.0, kMergeUs = 2.0, kMergeBytesPerUs = 3.0e6;
  const double groups = (double)((rows_b + nq - 1) / nq);
  const int64_t chunk = chunk_len(max_kv_len, nsplit, kMinChunk);
  const double per = (double)(chunk / kKeysPerTile);                 // tiles in a chunk of the longest request
  const double splits = (double)((max_kv_len + chunk - 1) / chunk);  // its non-empty chunks
  const double tiles_max = (double)((max_kv_len + kKeysPerTile - 1) / kKeysPerTile);
  const double tu = tile_us(resident, nq);
  double t;
  if (max_batch == 1) {
    t = std::ceil(groups * splits / sms) * (per * tu + kCtaUs);
  } else {
    const double work = groups * max_batch * tiles_max / 2.0;
    t = (work / sms + per) * tu + groups * max_batch * splits * kCtaUs / sms;
  }
  return t + kMergeUs + splits * rows_b * max_batch * 2048.0 / kMergeBytesPerUs;
}

// Mode and row-group size for a given split count (and, nsplit = 0, the
// split count too): the least modelled time; among choices within 2 % of it,
// the least per-key cost ceil(rows/NQ) * (128 + NQ) -- each row group lands
// every key and reads its 4 KB key operand per k-step, each query row adds
// 32 bytes of operand -- then the fewest splits (fewest partials), then the
// resident mode.
struct Choice {
  bool resident;
  int nq, splits;
};
Choice choose(int64_t rows_b, int64_t max_kv_len, int max_batch, int nsplit, bool allow_resident) {
  const double sms = (double)device_sm_count();
  const int64_t tiles_max = (max_kv_len + kKeysPerTile - 1) / kKeysPerTile;
  const int64_t n_lo = nsplit > 0 ? nsplit : 1;
  const int64_t n_hi = nsplit > 0 ? nsplit : std::min<int64_t>(tiles_max, 4096);
  auto for_each = [&](auto&& fn) {
    for (int res = allow_resident ? 1 : 0; res >= 0; --res)  // resident first: it wins exact ties
      for (int nq : kNqChoices) {
        if (res && nq > kMaxResidentNq) continue;
        for (int64_t n = n_lo; n <= n_hi; ++n) {
          if (nsplit == 0 && n > 1 && (tiles_max + n - 2) / (n - 1) == (tiles_max + n - 1) / n)
            continue;  // same chunks as n - 1 splits, only more partials
          fn(res != 0, nq, (int)n, est_us(rows_b, max_kv_len, max_batch, (int)n, nq, res != 0, sms));
        }
      }
  };
  double t_min = -1.0;
  for_each([&](bool, int, int, double t) {
    if (t_min < 0 || t < t_min) t_min = t;
  });
  Choice best{false, 96, (int)n_lo};
  int64_t best_work = -1;
  int best_n = 0;
  for_each([&](bool res, int nq, int n, double t) {
    if (t > t_min * 1.02) return;
    const int64_t work = (rows_b + nq - 1) / nq * (128 + nq);
    if (best_work < 0 || work < best_work || (work == best_work && n < best_n)) {
      best_work = work;
      best_n = n;
      best = {res, nq, n};
    }
  });
  return best;
}

int tc_smem(int nq, bool res) {
  switch (nq) {
    case 16: return split_tc_smem_16(res);
    case 32: return split_tc_smem_32(res);
    case 48: return split_tc_smem_48(res);
    case 64: return split_tc_smem_64(res);
    default: return split_tc_smem_96(res);
  }
}

cudaError_t tc_launch(int nq, bool res, const SplitArgs& a, const TcMaps& m, dim3 grid, cudaStream_t st) {
  switch (nq) {
    case 16: return launch_split_tc_16(a, m, grid, st, res);
    case 32: return launch_split_tc_32(a, m, grid, st, res);
    case 48: return launch_split_tc_48(a, m, grid, st, res);
    case 64: return launch_split_tc_64(a, m, grid, st, res);
    default: return launch_split_tc_96(a, m, grid, st, res);
  }
}

// ---- TMA descriptors --------------------------------------------------------
// cuTensorMapEncodeTiled is a driver entry point; it is fetched through the
// runtime so the library needs no link-time dependency on libcuda.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::mutex g_enc_mu;
EncodeTiledFn g_encode = nullptr;

int get_encode(EncodeTiledFn* out) {
  std::lock_guard<std::mutex> lk(g_enc_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return cuda_fail(e);
    if (q != cudaDriverEntryPointSuccess || !fn) {
      std::snprintf(g_cuda_msg, sizeof g_cuda_msg, "cuTensorMapEncodeTiled is not available from the driver");
      return MLA_VERIFY_ECUDA;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = g_encode;
  return MLA_VERIFY_OK;
}

// 2-D bf16 tensor [rows, inner] with a row pitch of inner*2 bytes; boxes of
// box_inner x box_rows elements, 128-byte swizzle, out-of-range reads as 0.
int encode_bf16_2d(EncodeTiledFn enc, CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                   uint32_t box_inner, uint32_t box_rows) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_cuda_msg, sizeof g_cuda_msg, "cuTensorMapEncodeTiled failed with CUresult %d", (int)r);
    return MLA_VERIFY_ECUDA;
  }
  return MLA_VERIFY_OK;
}

// Per-device capability check, cached.  The library carries sm_103a code only.
std::mutex g_dev_mu;
int g_dev_state[64];  // 0 unknown, 1 ok, 2 unsupported

int check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return MLA_VERIFY_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_state[dev] == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    g_dev_state[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return g_dev_state[dev] == 1 ? MLA_VERIFY_OK : MLA_VERIFY_EUNSUPPORTED;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The input arrays of a split launch (everything but the workspace).
int check_inputs(const void* q_nope_absorbed, const void* q_rope, const void* kv_pool, const int32_t* kv_indptr,
                 const int32_t* kv_indices, const int32_t* out_cache_loc, const uint8_t* custom_mask,
                 const int32_t* mask_indptr, float sm_scale) {
  if (!q_nope_absorbed || !q_rope || !kv_pool || !kv_indptr || !out_cache_loc || !custom_mask || !mask_indptr)
    return MLA_VERIFY_EINVAL;
  // kv_indices may be NULL only when every prefix is empty; the device never
  // reads it then.
  if (!aligned(q_nope_absorbed, 16) || !aligned(q_rope, 16) || !aligned(kv_pool, 16) || !aligned(kv_indptr, 4) ||
      (kv_indices && !aligned(kv_indices, 4)) || !aligned(out_cache_loc, 4) || !aligned(mask_indptr, 4))
    return MLA_VERIFY_EINVAL;
  if (!std::isfinite(sm_scale)) return MLA_VERIFY_EINVAL;
  return MLA_VERIFY_OK;
}


int check_common(const mla_verify_plan_s* pl, int32_t batch, int32_t nsplit, void* ws, size_t ws_bytes) {
  if (!pl) return MLA_VERIFY_EINVAL;
  if (batch < 0 || batch > pl->p.max_batch) return MLA_VERIFY_EINVAL;
  if (nsplit != pl->p.nsplit) return MLA_VERIFY_EINVAL;
  if (batch == 0) return MLA_VERIFY_OK;
  if (!ws || ws_bytes < pl->ws_bytes) return MLA_VERIFY_EWORKSPACE;
  if (!aligned(ws, 256)) return MLA_VERIFY_EINVAL;
  return MLA_VERIFY_OK;
}

}  // namespace

namespace mlav {
// Records the text of a CUDA error for mla_verify_strerror (used by other
// translation units of the library) and returns MLA_VERIFY_ECUDA.
int record_cuda_error(cudaError_t e) { return cuda_fail(e); }
// Bytes at the start of a plan's workspace that must be zero between calls
// (status header and, for a fused merge, the arrival counters).
size_t plan_zero_bytes(const mla_verify_plan_s* pl) { return pl->off_lse; }
size_t plan_workspace_bytes(const mla_verify_plan_s* pl) { return pl->ws_bytes; }
// Every check mla_verify_run makes before it enqueues work, except the
// workspace ones: plan, batch range, nsplit, inputs, outputs, device.  The
// no-allocation entry point runs it before it touches its scratch array.
int check_run_args(const mla_verify_plan_s* pl, const void* q_nope_absorbed, const void* q_rope,
                   const void* kv_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                   const int32_t* out_cache_loc, const uint8_t* custom_mask, const int32_t* mask_indptr,
                   int32_t batch, float sm_scale, int32_t nsplit, const void* o, const float* lse) {
  if (!pl) return MLA_VERIFY_EINVAL;
  if (batch < 0 || batch > pl->p.max_batch || nsplit != pl->p.nsplit) return MLA_VERIFY_EINVAL;
  if (batch == 0) return MLA_VERIFY_OK;
  if (!o || !lse || !aligned(o, 16) || !aligned(lse, 4)) return MLA_VERIFY_EINVAL;
  int rc = check_inputs(q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, out_cache_loc, custom_mask,
                        mask_indptr, sm_scale);
  if (rc != MLA_VERIFY_OK) return rc;
  return check_device();
}
}  // namespace mlav

extern "C" {

int mla_verify_plan(const mla_verify_params* params, size_t* workspace_bytes, mla_verify_plan_t* out) {
  if (!params || !workspace_bytes || !out) return MLA_VERIFY_EINVAL;
  const mla_verify_params& p = *params;
  if (p.max_batch < 1 || p.num_heads < 1 || p.q_len < 1 || p.q_len > kMaxQLen || p.nsplit < 0 ||
      p.pool_rows < 1 || p.max_kv_len < p.q_len)
    return MLA_VERIFY_EINVAL;
  if (p.d_latent != kDLatent || p.d_rope != kDRope) return MLA_VERIFY_EUNSUPPORTED;
  if ((p.flags & ~(MLA_VERIFY_FORCE_SIMT | MLA_VERIFY_FUSED_MERGE | MLA_VERIFY_REFETCH_VALUES |
                   MLA_VERIFY_TEST_STALL_GATHER)) != 0)
    return MLA_VERIFY_EINVAL;
  const int64_t rows_b = (int64_t)p.q_len * p.num_heads;
  const int64_t rows_max = rows_b * p.max_batch;
  if (rows_max > (int64_t)1 << 30 || p.pool_rows > ((int64_t)1 << 31) - 1) return MLA_VERIFY_EINVAL;

  mla_verify_plan_s* pl = new (std::nothrow) mla_verify_plan_s();
  if (!pl) return MLA_VERIFY_EINVAL;
  pl->p = p;
  pl->rows_max = rows_max;
  // Tensor cores for every shape unless MLA_VERIFY_FORCE_SIMT.  Even where
  // the 16-column tile is mostly padding (1 to 8 query rows) the kernel is
  // bound by gathering the rows, not by the MMAs, and measured 6-8x faster
  // than the CUDA-core kernel (16 requests x 8 heads x 1 token over 1k-33k
  // keys: 146 against 1064 us per call).
  pl->kernel = (p.flags & MLA_VERIFY_FORCE_SIMT) ? 0 : 1;
  if (pl->kernel) {
    // The mode (resident tile, unless MLA_VERIFY_REFETCH_VALUES), the row-group
    // size and, for nsplit = 0, the split count, from the time model.
    const Choice c = choose(rows_b, p.max_kv_len, p.max_batch, p.nsplit, !(p.flags & MLA_VERIFY_REFETCH_VALUES));
    pl->resident = c.resident;
    pl->nq = c.nq;
    pl->splits = c.splits;
  } else {
    // CUDA-core kernel (8 query rows per CTA); nsplit = 0 aims at about four
    // CTAs per SM in all.
    pl->resident = false;
    pl->nq = kSimtRowsPerCta;
    const int64_t rows = ((rows_b + kSimtRowsPerCta - 1) / kSimtRowsPerCta) * p.max_batch;
    const int64_t tiles = (p.max_kv_len + kKeysPerTile - 1) / kKeysPerTile;
    const int64_t want = std::max<int64_t>(1, (int64_t)device_sm_count() * 4 / std::max<int64_t>(rows, 1));
    pl->splits = p.nsplit > 0 ? p.nsplit : (int)std::min<int64_t>(want, tiles);
  }
  // Chunk granule: half a tile for one request in resident mode, where a
  // closing half tile lands half the rows and a chunk of ceil(L/nsplit) keys
  // then needs up to half a tile less (GB300, 64 heads x 9 tokens over 4,105
  // keys at nsplit 16: 35.1 -> 34.3 us per call); whole tiles otherwise, where
  // the extra chunks measured slower (value refetch over 65,545 keys at
  // nsplit 64: 204.5 -> 207.5 us; 16 ragged decode requests +0.5 %).
  pl->chunk_granule = (pl->kernel == 1 && pl->resident && p.max_batch == 1) ? kHalfTile : kKeysPerTile;
  // Chunks are never shorter than half the longest request's chunk: a
  // request much shorter than max_kv_len then takes fewer, longer chunks and
  // writes fewer partials, while the longest request -- the launch's
  // critical path -- keeps its chunks.
  {
    const int64_t longest = chunk_len(p.max_kv_len, pl->splits, kMinChunk, pl->chunk_granule);
    const int64_t half = longest / 2 / pl->chunk_granule * pl->chunk_granule;
    pl->min_chunk = (int)(half < kMinChunk ? kMinChunk : half);
  }
  pl->groups = (int)((rows_b + pl->nq - 1) / pl->nq);
  pl->smem = pl->kernel ? tc_smem(pl->nq, pl->resident) : 0;

  pl->fused = pl->kernel == 1 && (p.flags & MLA_VERIFY_FUSED_MERGE);
  pl->off_cnt = kWsHeader;
  pl->off_lse = pl->fused ? round_up(pl->off_cnt + sizeof(uint32_t) * (size_t)p.max_batch * pl->groups, 256)
                          : kWsHeader;
  pl->off_o = round_up(pl->off_lse + sizeof(float) * (size_t)pl->splits * (size_t)rows_max, 256);
  pl->ws_bytes = pl->off_o + sizeof(float) * (size_t)pl->splits * (size_t)rows_max * kDLatent;
  pl->merge_quarter = merge_quarter_fits(rows_max, device_sm_count());
  pl->merge_blocks = pl->fused ? 0 : merge_blocks((int)rows_max, pl->merge_quarter);
  *workspace_bytes = pl->ws_bytes;
  *out = pl;
  return MLA_VERIFY_OK;
}

int mla_verify_plan_describe(mla_verify_plan_t pl, mla_verify_plan_info* info) {
  if (!pl || !info) return MLA_VERIFY_EINVAL;
  info->kernel = pl->kernel;
  info->rows_per_cta = pl->nq;
  info->resident_tile = pl->resident ? 1 : 0;
  info->keys_per_tile = kKeysPerTile;
  info->grid_x = pl->groups;
  info->grid_y = pl->splits;
  info->grid_z = pl->p.max_batch;
  info->merge_blocks = pl->merge_blocks;
  info->smem_bytes = pl->smem;
  info->min_chunk = pl->min_chunk;
  info->chunk_granule = pl->chunk_granule;
  info->workspace_bytes = pl->ws_bytes;
  return MLA_VERIFY_OK;
}

}  // extern "C"

namespace {

int split_impl(mla_verify_plan_t pl, const void* q_nope_absorbed, const void* q_rope, const void* kv_pool,
               const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* qo_indptr,
               const int32_t* out_cache_loc, const uint8_t* custom_mask, const int32_t* mask_indptr, int32_t batch,
               float sm_scale, int32_t nsplit, void* workspace, size_t workspace_bytes, void* o, float* lse,
               void* stream) {
  int rc = check_common(pl, batch, nsplit, workspace, workspace_bytes);
  if (rc != MLA_VERIFY_OK || batch == 0) return rc;
  if (pl->fused && (!o || !lse)) return MLA_VERIFY_EINVAL;  // a fused plan has no split-only call
  if ((rc = check_inputs(q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, out_cache_loc, custom_mask,
                         mask_indptr, sm_scale)) != MLA_VERIFY_OK)
    return rc;
  if ((rc = check_device()) != MLA_VERIFY_OK) return rc;

  SplitArgs a = {};
  a.q_nope = static_cast<const __nv_bfloat16*>(q_nope_absorbed);
  a.q_rope = static_cast<const __nv_bfloat16*>(q_rope);
  a.kv_pool = static_cast<const __nv_bfloat16*>(kv_pool);
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.out_cache_loc = out_cache_loc;
  a.mask = custom_mask;
  a.mask_indptr = mask_indptr;
  a.qo_indptr = qo_indptr;
  a.test_stall = (pl->p.flags & MLA_VERIFY_TEST_STALL_GATHER) ? 1 : 0;
  a.batch = batch;
  a.H = pl->p.num_heads;
  a.T = pl->p.q_len;
  a.nsplit = pl->splits;
  a.min_chunk = pl->min_chunk;
  a.chunk_granule = pl->chunk_granule;
  a.pool_rows = pl->p.pool_rows;
  a.rows_max = pl->rows_max;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.part_lse = reinterpret_cast<float*>(ws + pl->off_lse);
  a.part_o = reinterpret_cast<float*>(ws + pl->off_o);
  a.merge_count = pl->fused ? reinterpret_cast<uint32_t*>(ws + pl->off_cnt) : nullptr;
  a.o = pl->fused ? static_cast<__nv_bfloat16*>(o) : nullptr;
  a.lse = pl->fused ? lse : nullptr;

  const dim3 grid(pl->groups, pl->splits, pl->p.max_batch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (pl->kernel) {
    // Descriptors are plain host structs passed by value with the launch: no
    // device work, so this stays capture-safe.
    EncodeTiledFn enc;
    if ((rc = get_encode(&enc)) != MLA_VERIFY_OK) return rc;
    TcMaps maps;
    const uint64_t rows_total = (uint64_t)batch * pl->p.q_len * pl->p.num_heads;
    if ((rc = encode_bf16_2d(enc, &maps.kv, kv_pool, kDRow, (uint64_t)pl->p.pool_rows, 64, 1)) != MLA_VERIFY_OK ||
        (rc = encode_bf16_2d(enc, &maps.qn, q_nope_absorbed, kDLatent, rows_total, 64, pl->nq)) != MLA_VERIFY_OK ||
        (rc = encode_bf16_2d(enc, &maps.qr, q_rope, kDRope, rows_total, 64, pl->nq)) != MLA_VERIFY_OK)
      return rc;
    e = tc_launch(pl->nq, pl->resident, a, maps, grid, st);
  } else {
    e = launch_split_simt(a, grid, st);
  }
  return e == cudaSuccess ? MLA_VERIFY_OK : cuda_fail(e);
}

int merge_impl(mla_verify_plan_t pl, int32_t batch, int32_t nsplit, const int32_t* qo_indptr, void* workspace,
               size_t workspace_bytes, void* o, float* lse, void* stream) {
  int rc = check_common(pl, batch, nsplit, workspace, workspace_bytes);
  if (rc != MLA_VERIFY_OK || batch == 0) return rc;
  if (!o || !lse || !aligned(o, 16) || !aligned(lse, 4)) return MLA_VERIFY_EINVAL;
  if ((rc = check_device()) != MLA_VERIFY_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  MergeArgs m = {};
  m.rows = batch * pl->p.q_len * pl->p.num_heads;
  m.qo_indptr = qo_indptr;
  m.batch = batch;
  m.H = pl->p.num_heads;
  m.nsplit = pl->splits;
  m.rows_max = pl->rows_max;
  m.part_lse = reinterpret_cast<const float*>(ws + pl->off_lse);
  m.part_o = reinterpret_cast<const float*>(ws + pl->off_o);
  m.o = static_cast<__nv_bfloat16*>(o);
  m.lse = lse;
  m.status = reinterpret_cast<uint32_t*>(ws);
  // Few rows: four warps per row.  When the partials also total at most
  // ~48 MB (still in L2 after the split kernel), the merge loads them before
  // their LSEs (an empty split's partial is read and dropped), one round trip
  // fewer.
  m.quarter = pl->merge_quarter ? 1 : 0;
  m.speculative =
      m.quarter && (uint64_t)pl->splits * (uint64_t)pl->rows_max * kDLatent * sizeof(float) <= (48ull << 20) ? 1 : 0;
  cudaError_t e = launch_merge(m, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_VERIFY_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int mla_verify_split(mla_verify_plan_t pl, const void* q_nope_absorbed, const void* q_rope, const void* kv_pool,
                     const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* out_cache_loc,
                     const uint8_t* custom_mask, const int32_t* mask_indptr, int32_t batch, float sm_scale,
                     int32_t nsplit, void* workspace, size_t workspace_bytes, void* stream) {
  return split_impl(pl, q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, nullptr, out_cache_loc, custom_mask,
                    mask_indptr, batch, sm_scale, nsplit, workspace, workspace_bytes, nullptr, nullptr, stream);
}

int mla_verify_merge(mla_verify_plan_t pl, int32_t batch, int32_t nsplit, void* workspace, size_t workspace_bytes,
                     void* o, float* lse, void* stream) {
  return merge_impl(pl, batch, nsplit, nullptr, workspace, workspace_bytes, o, lse, stream);
}

int mla_verify_run(mla_verify_plan_t pl, const void* q_nope_absorbed, const void* q_rope, const void* kv_pool,
                   const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* out_cache_loc,
                   const uint8_t* custom_mask, const int32_t* mask_indptr, int32_t batch, float sm_scale,
                   int32_t nsplit, void* workspace, size_t workspace_bytes, void* o, float* lse, void* stream) {
  int rc = check_common(pl, batch, nsplit, workspace, workspace_bytes);
  if (rc != MLA_VERIFY_OK || batch == 0) return rc;
  if (!o || !lse || !aligned(o, 16) || !aligned(lse, 4)) return MLA_VERIFY_EINVAL;
  rc = split_impl(pl, q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, nullptr, out_cache_loc, custom_mask,
                  mask_indptr, batch, sm_scale, nsplit, workspace, workspace_bytes, o, lse, stream);
  if (rc != MLA_VERIFY_OK || pl->fused) return rc;
  return merge_impl(pl, batch, nsplit, nullptr, workspace, workspace_bytes, o, lse, stream);
}

int mla_verify_run_varlen(mla_verify_plan_t pl, const void* q_nope_absorbed, const void* q_rope,
                          const void* kv_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                          const int32_t* qo_indptr, const int32_t* out_cache_loc, const uint8_t* custom_mask,
                          const int32_t* mask_indptr, int32_t batch, float sm_scale, int32_t nsplit,
                          void* workspace, size_t workspace_bytes, void* o, float* lse, void* stream) {
  int rc = check_common(pl, batch, nsplit, workspace, workspace_bytes);
  if (rc != MLA_VERIFY_OK || batch == 0) return rc;
  if (!qo_indptr || !aligned(qo_indptr, 4)) return MLA_VERIFY_EINVAL;
  if (!o || !lse || !aligned(o, 16) || !aligned(lse, 4)) return MLA_VERIFY_EINVAL;
  rc = split_impl(pl, q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, qo_indptr, out_cache_loc,
                  custom_mask, mask_indptr, batch, sm_scale, nsplit, workspace, workspace_bytes, o, lse, stream);
  if (rc != MLA_VERIFY_OK || pl->fused) return rc;
  return merge_impl(pl, batch, nsplit, qo_indptr, workspace, workspace_bytes, o, lse, stream);
}

int mla_verify_build_tree_mask(mla_verify_plan_t pl, const int32_t* parents, const int32_t* kv_indptr,
                               int32_t batch, uint8_t* custom_mask, size_t mask_bytes, int32_t* mask_indptr,
                               void* stream) {
  if (!pl || batch < 0 || batch > pl->p.max_batch) return MLA_VERIFY_EINVAL;
  if (batch == 0) return MLA_VERIFY_OK;
  if (!parents || !kv_indptr || !custom_mask || !mask_indptr || !aligned(parents, 4) || !aligned(kv_indptr, 4) ||
      !aligned(mask_indptr, 4))
    return MLA_VERIFY_EINVAL;
  int rc;
  if ((rc = check_device()) != MLA_VERIFY_OK) return rc;
  const int64_t max_bytes = ((int64_t)pl->p.max_batch * pl->p.q_len * pl->p.max_kv_len + 7) / 8;
  cudaError_t e = launch_tree_mask(parents, kv_indptr, nullptr, batch, pl->p.q_len, custom_mask, (int64_t)mask_bytes,
                                   mask_indptr, max_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_VERIFY_OK : cuda_fail(e);
}

int mla_verify_build_tree_mask_varlen(mla_verify_plan_t pl, const int32_t* parents, const int32_t* kv_indptr,
                                      const int32_t* qo_indptr, int32_t batch, uint8_t* custom_mask,
                                      size_t mask_bytes, int32_t* mask_indptr, void* stream) {
  if (!pl || batch < 0 || batch > pl->p.max_batch || batch > kMaxTreeMaskVarlenBatch) return MLA_VERIFY_EINVAL;
  if (batch == 0) return MLA_VERIFY_OK;
  if (!parents || !kv_indptr || !qo_indptr || !custom_mask || !mask_indptr || !aligned(parents, 4) ||
      !aligned(kv_indptr, 4) || !aligned(qo_indptr, 4) || !aligned(mask_indptr, 4))
    return MLA_VERIFY_EINVAL;
  int rc;
  if ((rc = check_device()) != MLA_VERIFY_OK) return rc;
  const int64_t max_bytes = ((int64_t)pl->p.max_batch * pl->p.q_len * pl->p.max_kv_len + 7) / 8;
  cudaError_t e = launch_tree_mask(parents, kv_indptr, qo_indptr, batch, pl->p.q_len, custom_mask,
                                   (int64_t)mask_bytes, mask_indptr, max_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_VERIFY_OK : cuda_fail(e);
}

int mla_verify_relocate_kv(mla_verify_plan_t pl, void* kv_pool, const int32_t* kv_indptr, int32_t* kv_indices,
                           const int32_t* dst_start, int32_t batch, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (!pl || batch < 0 || batch > pl->p.max_batch) return MLA_VERIFY_EINVAL;
  if (batch == 0) return MLA_VERIFY_OK;
  if (!kv_pool || !kv_indptr || !kv_indices || !dst_start || !aligned(kv_pool, 16) || !aligned(kv_indptr, 4) ||
      !aligned(kv_indices, 4) || !aligned(dst_start, 4))
    return MLA_VERIFY_EINVAL;
  if (!workspace || workspace_bytes < pl->ws_bytes) return MLA_VERIFY_EWORKSPACE;
  if (!aligned(workspace, 256)) return MLA_VERIFY_EINVAL;
  int rc;
  if ((rc = check_device()) != MLA_VERIFY_OK) return rc;
  const int64_t max_keys = (int64_t)pl->p.max_batch * pl->p.max_kv_len;
  cudaError_t e = mlav::launch_relocate(kv_pool, kv_indptr, kv_indices, dst_start, batch, pl->p.pool_rows, max_keys,
                                        reinterpret_cast<uint32_t*>(workspace), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_VERIFY_OK : cuda_fail(e);
}

int mla_verify_workspace_init(mla_verify_plan_t pl, void* workspace, size_t workspace_bytes, void* stream) {
  if (!pl || !workspace || workspace_bytes < pl->ws_bytes || !aligned(workspace, 256)) return MLA_VERIFY_EINVAL;
  cudaError_t e = cudaMemsetAsync(workspace, 0, pl->off_lse, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_VERIFY_OK : cuda_fail(e);
}

int mla_verify_read_status(mla_verify_plan_t pl, void* workspace, void* stream, uint32_t* device_status) {
  if (!pl || !workspace || !device_status) return MLA_VERIFY_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t w[2] = {0, 0};
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(w, workspace, sizeof w, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof w, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  *device_status = w[0] | w[1];
  return MLA_VERIFY_OK;
}

int mla_verify_destroy(mla_verify_plan_t pl) {
  delete pl;
  return MLA_VERIFY_OK;
}

const char* mla_verify_strerror(int code) {
  switch (code) {
    case MLA_VERIFY_OK: return "ok";
    case MLA_VERIFY_EINVAL: return "invalid argument (NULL, misaligned, out-of-range size or batch, nsplit mismatch)";
    case MLA_VERIFY_EUNSUPPORTED: return "unsupported: dims must be 512/64 and the device sm_103";
    case MLA_VERIFY_EWORKSPACE: return "workspace missing or smaller than the plan requires";
    case MLA_VERIFY_ECUDA: return g_cuda_msg;
    default: return "unknown error code";
  }
}

}  // extern "C"
