/*
 * mla_verify.h -- C ABI of the GB300 (sm_103a) MLA tree-verify attention library
 * (libmlaverify.so).
 *
 * The operation.  Speculative decoding verifies a tree of T draft tokens per
 * request in one attention call: every draft token i of request b attends,
 * for each of H heads, over that request's whole paged latent KV cache under
 * a tree-visibility mask [Custom sm_120 Verify Kernel, §"The Bottleneck:
 * Triton's Scattered KV Access at 14 GB/s"; Capture Safety to MoE Ceiling,
 * §"The Architecture of Capture Safety"].  The cache has page_size = 1, so
 * each pool row is one token: 512 bf16 latent values followed by 64 bf16
 * RoPE key values (576 values, 1152 bytes).  With P_b prefix tokens and
 * L_b = P_b + T keys per request:
 *
 *   row(j)   = kv_indices[kv_indptr[b] + j]           for j <  P_b
 *            = out_cache_loc[b*T + (j - P_b)]         for j >= P_b
 *   vis(i,j) = bit (mask_indptr[b] + i*L_b + j) of custom_mask, LSB-first
 *   s_j      = sm_scale * (q_nope[b*T+i, h, :] . kv[row(j), 0:512]
 *                        + q_rope[b*T+i, h, :] . kv[row(j), 512:576])
 *   O        = sum_{vis j} softmax(s)_j * kv[row(j), 0:512]
 *   LSE      = ln sum_{vis j} exp(s_j)
 *
 * Prefix rows come from kv_indices and draft rows from out_cache_loc (two
 * arrays, selected by position), and the mask row stride is P_b + T, not P_b
 * [Custom sm_120 Verify Kernel, §"The Debugging Gauntlet: Three Real Bugs
 * Against Live Tensors", bug 2]; mask_indptr holds B entries, one per
 * request [same section, bug 3].  A token whose visible set is empty gets
 * O = 0 and LSE = -inf.
 *
 * The computation is split-K: each request's key range is cut into `nsplit`
 * chunks (or as many as the plan picked, nsplit = 0), one CTA per (chunk,
 * group of query rows, request) writes a partial
 * (normalised O, LSE) into the workspace, and a second kernel merges the
 * partials by log-sum-exp [Custom sm_120 Verify Kernel, §"Building the
 * Custom Kernel: From Occupancy Starvation to Flash-Decode"].  The grid is
 * fixed at plan time and chunk bounds are computed on the device from the
 * actual lengths; chunks past a request's end exit at once [Capture Safety
 * to MoE Ceiling, §"The Architecture of Capture Safety"].
 *
 * Conventions.
 *  - All device pointers are borrowed: the caller owns every device buffer,
 *    the workspace included.  The library owns only the host-side plan.
 *  - mla_verify_run (and split/merge) allocate nothing, never synchronise
 *    with the host and only enqueue work on `stream`, so a call can be
 *    captured into a CUDA graph and replayed with new device contents.
 *  - Calls return MLA_VERIFY_OK (0) or a positive error code; no exception
 *    or signal crosses the ABI.  mla_verify_strerror() describes a code.
 *  - Errors detected on the device (a pool row index outside [0, pool_rows),
 *    a pipeline wait that timed out) do not abort the call: a key whose
 *    row is out of range is left out (as if masked) and a bit is set in a
 *    status word inside the workspace, read with mla_verify_read_status().
 *  - One plan may serve concurrent calls on different streams when each
 *    call has its own workspace.
 */
#ifndef MLA_VERIFY_H_
#define MLA_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define MLA_VERIFY_OK 0
#define MLA_VERIFY_EINVAL 1       /* bad / NULL / misaligned argument, batch > max_batch */
#define MLA_VERIFY_EUNSUPPORTED 2 /* d_latent != 512, d_rope != 64, or a device other than sm_103 (the only code the library carries) */
#define MLA_VERIFY_EWORKSPACE 3   /* workspace missing or smaller than the plan requires */
#define MLA_VERIFY_ECUDA 4        /* a CUDA runtime call failed (launch, attribute query) */

/* Device status bits (see mla_verify_read_status). */
#define MLA_VERIFY_DEV_BAD_ROW 0x1u /* some resolved pool row was outside [0, pool_rows) */
#define MLA_VERIFY_DEV_TIMEOUT 0x2u /* a pipeline wait gave up; that CTA's partial is invalid */

/* Plan flags. */
#define MLA_VERIFY_FORCE_SIMT 0x1 /* use the CUDA-core (warp-shuffle) split kernel for every shape */
/* Merge inside the tensor-core split kernel: the last CTA of each (request,
 * row group) to finish merges that group's rows from the other CTAs'
 * partials, so a run is one kernel launch (describe() then reports
 * merge_blocks = 0).  Results are bit-identical to the separate merge.  The
 * workspace gains one counter per (request, row group) between the header
 * and the partials; mla_verify_split is refused (EINVAL) for such a plan.
 * Ignored with MLA_VERIFY_FORCE_SIMT (the CUDA-core kernel keeps the separate merge). */
#define MLA_VERIFY_FUSED_MERGE 0x2
/* Run the tensor-core split kernel in its value-refetch mode: each 128-key
 * tile's 8 value blocks are gathered a second time for the PV product, which
 * allows row groups of up to 96 query rows.  Without this flag the kernel
 * keeps each tile resident in shared memory (row groups of at most 64 rows,
 * each key gathered once per row group).  Results agree within rounding;
 * the flag exists to compare the two modes. */
#define MLA_VERIFY_REFETCH_VALUES 0x4
/* Test only: the tensor-core split kernel's gather never signals its first
 * block, so every CTA's bounded pipeline waits run out (about 2 s), the CTAs
 * drain and return, and the call reports MLA_VERIFY_DEV_TIMEOUT; its outputs
 * are not valid.  It exercises failure detection without faulting the GPU. */
#define MLA_VERIFY_TEST_STALL_GATHER 0x100

typedef struct mla_verify_plan_s* mla_verify_plan_t; /* opaque, host-only, immutable after plan */

typedef struct {
  int32_t max_batch;  /* B_max >= 1: largest batch a run may pass; sizes the grid and workspace */
  int32_t num_heads;  /* H >= 1 */
  int32_t q_len;      /* T in [1, 64]: draft tokens per request (uniform) */
  int32_t max_kv_len; /* >= max_b (P_b + T); documents the longest request (chunk size is per request) */
  int64_t pool_rows;  /* rows in kv_pool; keys resolving outside [0, pool_rows) are left out and flagged */
  int32_t nsplit;     /* >= 1: KV chunks per request = partials per output row (fixed grid
                       *       dimension); request b's chunk is ceil(L_b/nsplit) rounded up to
                       *       describe().chunk_granule keys, and at least describe().min_chunk (half the chunk of a
                       *       max_kv_len request), so a much shorter request fills fewer chunks
                       *       and its other chunks are empty;
                       * 0: the plan picks the number of chunks (describe().grid_y) and the
                       *    row-group size for this GPU from max_batch and max_kv_len; runs then
                       *    pass nsplit = 0 as well */
  int32_t d_latent;   /* must be 512 */
  int32_t d_rope;     /* must be 64 */
  int32_t flags;      /* OR of MLA_VERIFY_FORCE_SIMT, MLA_VERIFY_FUSED_MERGE, MLA_VERIFY_REFETCH_VALUES,
                       * MLA_VERIFY_TEST_STALL_GATHER */
} mla_verify_params;

/* What a plan chose (for tests, benchmarks and logs). */
typedef struct {
  int32_t kernel;        /* 1 = tcgen05 tensor-core split kernel, 0 = CUDA-core split kernel */
  int32_t rows_per_cta;  /* query rows (token x head pairs) one split CTA covers */
  int32_t keys_per_tile; /* keys per pipeline tile (128) */
  int32_t grid_x, grid_y, grid_z; /* split grid: row groups x KV chunks per request x max_batch */
  int32_t merge_blocks;  /* merge grid size; 0 when the split kernel merges (MLA_VERIFY_FUSED_MERGE) */
  int32_t smem_bytes;    /* dynamic shared memory of the split kernel */
  size_t workspace_bytes;
  int32_t resident_tile; /* 1: tensor-core kernel keeps each key tile resident (one gather per key and
                          * row group); 0: value blocks gathered twice, or the CUDA-core kernel */
  int32_t min_chunk;     /* shortest chunk of any request, in keys (see nsplit) */
  int32_t chunk_granule; /* chunk lengths are multiples of it: 64 keys (resident tiles, one request) or 128 */
} mla_verify_plan_info;

/*
 * Validate `params` and build a plan.  Host only: touches no device state.
 * On success *out receives the plan and *workspace_bytes the size of the
 * device workspace every run with this plan needs (fp32 partial O and LSE
 * for grid_y x max_batch*q_len*num_heads rows -- grid_y = nsplit, or the
 * plan's count when nsplit = 0 -- plus a 256-byte header, and
 * for MLA_VERIFY_FUSED_MERGE one 32-bit counter per request and row group).
 * The workspace must be 256-byte aligned and zero-filled once before its
 * first use (e.g. torch.zeros, or mla_verify_workspace_init); the library
 * keeps the header and the counters consistent afterwards (after a call that
 * reported MLA_VERIFY_DEV_TIMEOUT, initialise it again).
 * Errors: EINVAL (NULL pointer, non-positive sizes, q_len > 64),
 * EUNSUPPORTED (d_latent != 512 or d_rope != 64).
 */
int mla_verify_plan(const mla_verify_params* params, size_t* workspace_bytes,
                    mla_verify_plan_t* out);

/* Fill *info with the choices of `plan`.  Errors: EINVAL. */
int mla_verify_plan_describe(mla_verify_plan_t plan, mla_verify_plan_info* info);

/*
 * One verify call: split kernel then merge kernel, both enqueued on `stream`.
 *
 *  q_nope_absorbed  bf16 [batch*q_len, num_heads, 512], contiguous, 16-byte aligned
 *  q_rope           bf16 [batch*q_len, num_heads, 64],  contiguous, 16-byte aligned
 *  kv_pool          bf16 [pool_rows, 576], contiguous, 16-byte aligned (rows of 1152 bytes)
 *  kv_indptr        int32 [batch+1], kv_indptr[0] = 0, non-decreasing; prefix rows only
 *  kv_indices       int32 [kv_indptr[batch]] pool rows of the prefixes
 *  out_cache_loc    int32 [batch*q_len] pool rows holding the draft tokens' KV
 *                   (already written before the call)
 *  custom_mask      uint8 packed bits, LSB-first; request b's [q_len, P_b+q_len]
 *                   row-major block starts at bit mask_indptr[b]
 *  mask_indptr      int32 [batch] bit offsets (B entries, not B+1)
 *  batch            0 <= batch <= max_batch (0 enqueues nothing)
 *  sm_scale         score scale (1/sqrt(192) for the K2-class MLA geometry)
 *  nsplit           must equal the plan's nsplit (0 for a plan that picked its own count)
 *  workspace        device buffer of >= the plan's workspace_bytes (see mla_verify_plan)
 *  o                bf16 [batch*q_len, num_heads, 512] output (round-to-nearest-even)
 *  lse              fp32 [batch*q_len, num_heads] output, natural log
 *  stream           cudaStream_t (NULL = legacy default stream)
 *
 * The device arrays must stay valid until the enqueued work completes.
 * Every row the call references, visible or masked, must hold finite values
 * (a masked key still enters the value product with weight 0).
 * Errors: EINVAL (NULL or misaligned pointer, batch outside [0, max_batch],
 * nsplit mismatch), EWORKSPACE, EUNSUPPORTED (device is not sm_103),
 * ECUDA (launch failure; see mla_verify_strerror).
 */
int mla_verify_run(mla_verify_plan_t plan, const void* q_nope_absorbed, const void* q_rope,
                   const void* kv_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                   const int32_t* out_cache_loc, const uint8_t* custom_mask,
                   const int32_t* mask_indptr, int32_t batch, float sm_scale, int32_t nsplit,
                   void* workspace, size_t workspace_bytes, void* o, float* lse, void* stream);

/*
 * mla_verify_run for requests with their own numbers of draft tokens,
 * T_b = qo_indptr[b+1] - qo_indptr[b] with 0 <= T_b <= the plan's q_len
 * (T_b = 1 everywhere is plain decode on the same kernels).  Request b owns
 * token rows qo_indptr[b] .. qo_indptr[b+1]-1 of q_nope_absorbed, q_rope, o
 * and lse (output row (qo_indptr[b] + i)*num_heads + h); its draft rows are
 * out_cache_loc[qo_indptr[b] + t]; its mask block is [T_b, P_b + T_b]
 * row-major at bit mask_indptr[b] -- the layout of mla_verify_run with T
 * replaced by T_b [Custom sm_120 Verify Kernel, §"The Debugging Gauntlet",
 * bugs 2 and 3].
 *
 *  qo_indptr  int32 [batch+1], qo_indptr[0] = 0, non-decreasing
 *  q_nope_absorbed, q_rope, o, lse: allocated for batch*q_len token rows (the
 *             fixed-size buffers a captured call uses); rows from
 *             qo_indptr[batch] on may be read but are never written
 *  everything else as mla_verify_run.
 *
 * Errors as mla_verify_run, plus EINVAL for a NULL or misaligned qo_indptr.
 */
int mla_verify_run_varlen(mla_verify_plan_t plan, const void* q_nope_absorbed, const void* q_rope,
                          const void* kv_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                          const int32_t* qo_indptr, const int32_t* out_cache_loc,
                          const uint8_t* custom_mask, const int32_t* mask_indptr, int32_t batch,
                          float sm_scale, int32_t nsplit, void* workspace, size_t workspace_bytes,
                          void* o, float* lse, void* stream);

/*
 * The two launches of mla_verify_run, separately: the split kernel (writes
 * the partials into the workspace) and the merge kernel (reads them, writes
 * o and lse).  Same arguments and errors as mla_verify_run; merge ignores
 * the input arrays.  A merge must follow the split of the same call on the
 * same stream (or be ordered after it).  A plan with MLA_VERIFY_FUSED_MERGE
 * on the tensor-core kernel has no split-only call (EINVAL); merge still
 * works on the partials its run left in the workspace.
 */
int mla_verify_split(mla_verify_plan_t plan, const void* q_nope_absorbed, const void* q_rope,
                     const void* kv_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                     const int32_t* out_cache_loc, const uint8_t* custom_mask,
                     const int32_t* mask_indptr, int32_t batch, float sm_scale, int32_t nsplit,
                     void* workspace, size_t workspace_bytes, void* stream);
int mla_verify_merge(mla_verify_plan_t plan, int32_t batch, int32_t nsplit, void* workspace,
                     size_t workspace_bytes, void* o, float* lse, void* stream);

/* Zero the workspace header (and a fused merge's counters) on `stream` (one
 * cudaMemsetAsync).  Errors: EINVAL, ECUDA. */
int mla_verify_workspace_init(mla_verify_plan_t plan, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Synchronise `stream`, then report in *device_status the OR of the
 * MLA_VERIFY_DEV_* bits raised since the previous read (and clear them).
 * Test and diagnostics only: it blocks the host, so never call it inside
 * stream capture.  Errors: EINVAL, ECUDA.
 */
int mla_verify_read_status(mla_verify_plan_t plan, void* workspace, void* stream,
                           uint32_t* device_status);

/*
 * Build the packed visibility mask of a verify call on the device from the
 * draft trees' parent arrays (one kernel on `stream`; no allocation, no host
 * synchronisation, so it can be captured in the same CUDA graph as
 * mla_verify_run).  The pages build the tree and the mask on the host every
 * step and measured that cost [Capture Safety to MoE Ceiling, §"Phase 2e:
 * The Occupancy Epiphany and the 3-6x Speedup"]; the layout written is the
 * one mla_verify_run reads [Custom sm_120 Verify Kernel, §"The Debugging
 * Gauntlet"].
 *
 *  parents      int32 [batch*q_len]: parents[b*q_len + i] is the parent node of
 *               draft token i of request b, -1 for a root; a parent precedes its
 *               child (-1 <= parent < i).  A link outside that range ends the
 *               ancestor walk (the token then sees only the nodes walked).
 *  kv_indptr    int32 [batch+1], non-decreasing: P_b = kv_indptr[b+1] - kv_indptr[b]
 *  batch        0 <= batch <= max_batch (0 enqueues nothing)
 *  custom_mask  uint8 output: bit mask_indptr[b] + i*(P_b+q_len) + j (LSB-first) is 1
 *               when j < P_b, or when draft node j - P_b is i or an ancestor of i
 *  mask_bytes   capacity of custom_mask; bits past it are not written
 *  mask_indptr  int32 [batch] output: q_len * sum_{b'<b} (P_b' + q_len)
 *  stream       cudaStream_t (NULL = legacy default stream)
 *
 * Bits past the last request's block, within the last byte, are written 0.
 * The plan supplies q_len and the grid (sized for max_batch requests of
 * max_kv_len keys).  Errors: EINVAL (NULL or misaligned pointer, batch outside
 * [0, max_batch]), ECUDA.
 */
int mla_verify_build_tree_mask(mla_verify_plan_t plan, const int32_t* parents, const int32_t* kv_indptr,
                               int32_t batch, uint8_t* custom_mask, size_t mask_bytes,
                               int32_t* mask_indptr, void* stream);

/*
 * mla_verify_build_tree_mask for a varlen call (see mla_verify_run_varlen):
 * request b has T_b = qo_indptr[b+1] - qo_indptr[b] draft tokens
 * (0 <= T_b <= q_len), its parent array is parents[qo_indptr[b] ..
 * qo_indptr[b] + T_b) (node indices local to the request, -1 for a root),
 * its block is [T_b, P_b + T_b] and mask_indptr[b] =
 * sum_{b'<b} T_b' * (P_b' + T_b').  Other arguments and the bit rule as
 * mla_verify_build_tree_mask.  Errors: EINVAL (also batch > 1024), ECUDA.
 */
int mla_verify_build_tree_mask_varlen(mla_verify_plan_t plan, const int32_t* parents, const int32_t* kv_indptr,
                                      const int32_t* qo_indptr, int32_t batch, uint8_t* custom_mask,
                                      size_t mask_bytes, int32_t* mask_indptr, void* stream);

/*
 * KV relocation (the second, "live" tier of KV defragmentation: move each
 * request's scattered rows into contiguous rows and rewrite its indices
 * [The Art of Knowing When to Stop: Deferring Tier 1 Defrag, §"The Decision:
 * Why Tier 1 Defrag Gets Deferred"]).  One kernel on `stream`, no
 * allocation, no host synchronisation.
 *
 *  kv_pool      bf16 [pool_rows, 576], 16-byte aligned; read and written
 *  kv_indptr    int32 [batch+1], non-decreasing: request b's prefix keys are
 *               kv_indices[kv_indptr[b] .. kv_indptr[b+1])
 *  kv_indices   int32, read and rewritten in place
 *  dst_start    int32 [batch]: first destination row of request b
 *  batch        0 <= batch <= max_batch (0 enqueues nothing)
 *  workspace    the plan's workspace (only its status word is used)
 *
 * For every prefix key k of request b (j = k - kv_indptr[b]), pool row
 * kv_indices[k] is copied whole to row dst_start[b] + j and kv_indices[k]
 * becomes dst_start[b] + j.  The destination rows must be free: no source
 * row of the call may lie in any request's destination block (the copies run
 * in no particular order).  Draft rows (out_cache_loc) are not moved.  A key
 * whose source or destination row is outside [0, pool_rows) is left as it was
 * and raises MLA_VERIFY_DEV_BAD_ROW in the workspace status word.  A verify
 * call on the relocated pool and indices gives bit-identical results (row
 * ids do not enter the arithmetic).  The plan supplies pool_rows and the grid
 * (max_batch x max_kv_len keys at most).  Errors: EINVAL (NULL or misaligned
 * pointer, batch outside [0, max_batch]), EWORKSPACE, ECUDA.
 */
int mla_verify_relocate_kv(mla_verify_plan_t plan, void* kv_pool, const int32_t* kv_indptr, int32_t* kv_indices,
                           const int32_t* dst_start, int32_t batch, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * mla_verify_run without a workspace argument, for callers that have no way
 * to obtain device memory of their own: for example a plugin host that hands
 * a kernel only its input and output buffers, or a latency-critical path that
 * must not call cudaMalloc (it can synchronise the device and fail under
 * memory pressure).  The pages describe nothing like it; it exists for such
 * integrations.
 *
 * The split partials go to a scratch array of 32 MiB compiled into the
 * library, which every GPU that loads the library keeps reserved until the
 * process exits.  A plan whose workspace_bytes exceeds 32 MiB is rejected
 * with MLA_VERIFY_EWORKSPACE (e.g. 64 heads x 9 draft tokens fit up to
 * nsplit = 28 at batch 1).  Nothing is allocated: the first call in each CUDA
 * context (the device's primary context, or a context the caller made
 * current) looks up the array's device address in that context
 * (cudaGetSymbolAddress), so make that first call outside any stream capture;
 * a process may use up to 64 contexts this way (then EUNSUPPORTED).  Each
 * call first makes every check of mla_verify_run (a rejected call touches
 * nothing on the device), then zeroes the array's 256-byte status header and,
 * for a MLA_VERIFY_FUSED_MERGE plan, its arrival counters, on `stream`, and
 * runs exactly mla_verify_run on the array.  All calls in the process share
 * the one array: calls whose work overlaps on the GPU (other streams, other
 * threads) race and corrupt each other's results; serialise them.
 * Device-detected conditions are not reported (there is no workspace to read
 * a status word from).  Arguments and errors otherwise as mla_verify_run.
 */
int mla_verify_run_noalloc(mla_verify_plan_t plan, const void* q_nope_absorbed, const void* q_rope,
                           const void* kv_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                           const int32_t* out_cache_loc, const uint8_t* custom_mask,
                           const int32_t* mask_indptr, int32_t batch, float sm_scale, int32_t nsplit,
                           void* o, float* lse, void* stream);

/* Free the plan (NULL is accepted).  Returns MLA_VERIFY_OK. */
int mla_verify_destroy(mla_verify_plan_t plan);

/* Static description of a return code, or of the last CUDA error for ECUDA. */
const char* mla_verify_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* MLA_VERIFY_H_ */
