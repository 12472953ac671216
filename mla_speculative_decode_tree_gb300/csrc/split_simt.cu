// CUDA-core split kernel: one warp per query row (token, head), warp-shuffle
// dot products and an online softmax over the keys of one split.
//
// This is the shape-agnostic path, taken with MLA_VERIFY_FORCE_SIMT: the
// independent second implementation the tensor-core kernel is compared with
// (the planner uses the tensor cores for every shape, also for one to eight
// query rows per request, where this kernel measured 6-8x slower).
// Each lane owns 16 of the 512 latent columns (16-byte chunks l and l+32 of a
// row) and lanes 0-7 also own one 16-byte chunk of the 64 RoPE columns, so a
// key row is fetched with 128-bit loads [Capture Safety to MoE Ceiling,
// §"Vectorized Loads: The Final Push"; Custom sm_120 Verify Kernel, §"The
// Float4 Vectorization"].
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kKeysPerStep = 4;

__device__ __forceinline__ void bf16x8_to_f32(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(32 * kSimtRowsPerCta) split_simt_kernel(SplitArgs a) {
  const int b = blockIdx.z;
  if (b >= a.batch) return;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int s = blockIdx.y;
  const int64_t kv_base = a.kv_indptr[b];
  const int64_t P = (int64_t)a.kv_indptr[b + 1] - kv_base;
  const RequestTokens rq = request_tokens(a, b);
  const int64_t L = P + rq.n;
  const int64_t chunk = chunk_len(L, a.nsplit, a.min_chunk, a.chunk_granule);
  const int64_t j0 = (int64_t)s * chunk;
  const int64_t j1 = (j0 + chunk < L) ? j0 + chunk : L;
  const int rows_b = rq.n * a.H;
  const int r = blockIdx.x * kSimtRowsPerCta + warp;
  if (r >= rows_b) return;
  const int i = r / a.H;
  const int64_t grow = rq.q0 * a.H + r;  // == (q0 + i)*H + h
  float* lse_out = a.part_lse + (int64_t)s * a.rows_max + grow;
  if (j0 >= j1) {
    if (lane == 0) *lse_out = -INFINITY;
    return;
  }

  // Query row in registers (fp32).
  float qa[8], qb[8], qr[8];
  {
    const uint4* qn = reinterpret_cast<const uint4*>(a.q_nope + grow * kDLatent);
    bf16x8_to_f32(__ldg(qn + lane), qa);
    bf16x8_to_f32(__ldg(qn + 32 + lane), qb);
    const uint4* qp = reinterpret_cast<const uint4*>(a.q_rope + grow * kDRope);
    uint4 z = make_uint4(0, 0, 0, 0);
    bf16x8_to_f32(lane < 8 ? __ldg(qp + lane) : z, qr);
  }

  const int64_t mask_row = (int64_t)a.mask_indptr[b] + (int64_t)i * L;
  float m = -INFINITY, lsum = 0.f;
  float acc_a[8], acc_b[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc_a[k] = acc_b[k] = 0.f;

  for (int64_t jb = j0; jb < j1; jb += kKeysPerStep) {
    uint4 va[kKeysPerStep], vb[kKeysPerStep], vr[kKeysPerStep];
    bool vis[kKeysPerStep];
#pragma unroll
    for (int u = 0; u < kKeysPerStep; ++u) {
      const int64_t j = jb + u;
      vis[u] = (j < j1) && mask_bit(a.mask, mask_row + j);
      va[u] = vb[u] = vr[u] = make_uint4(0, 0, 0, 0);
      if (vis[u]) {
        const int64_t row = resolve_row(a, rq.q0, P, kv_base, j);
        if (row >= 0) {
          const uint4* kv = reinterpret_cast<const uint4*>(a.kv_pool + row * kDRow);
          va[u] = __ldg(kv + lane);
          vb[u] = __ldg(kv + 32 + lane);
          if (lane < 8) vr[u] = __ldg(kv + 64 + lane);
        } else {  // a row outside the pool excludes the key
          vis[u] = false;
          if (lane == 0) atomicOr(a.status, kStatusBadRow);
        }
      }
    }
    float sc[kKeysPerStep];
#pragma unroll
    for (int u = 0; u < kKeysPerStep; ++u) {
      float fa[8], fb[8], fr[8];
      bf16x8_to_f32(va[u], fa);
      bf16x8_to_f32(vb[u], fb);
      bf16x8_to_f32(vr[u], fr);
      float d = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) d = fmaf(qa[k], fa[k], fmaf(qb[k], fb[k], fmaf(qr[k], fr[k], d)));
      sc[u] = d;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int u = 0; u < kKeysPerStep; ++u) sc[u] += __shfl_xor_sync(0xffffffffu, sc[u], off);
#pragma unroll
    for (int u = 0; u < kKeysPerStep; ++u) {
      if (!vis[u]) continue;
      const float sv = sc[u] * a.scale_log2;
      if (sv > m) {
        const float alpha = ex2_approx(m - sv);  // m = -inf gives 0
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          acc_a[k] *= alpha;
          acc_b[k] *= alpha;
        }
        lsum *= alpha;
        m = sv;
      }
      const float p = ex2_approx(sv - m);
      float fa[8], fb[8];
      bf16x8_to_f32(va[u], fa);
      bf16x8_to_f32(vb[u], fb);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc_a[k] = fmaf(p, fa[k], acc_a[k]);
        acc_b[k] = fmaf(p, fb[k], acc_b[k]);
      }
      lsum += p;
    }
  }

  if (lsum == 0.f) {
    if (lane == 0) *lse_out = -INFINITY;
    return;
  }
  const float inv = 1.f / lsum;
  float4* o = reinterpret_cast<float4*>(a.part_o + ((int64_t)s * a.rows_max + grow) * kDLatent);
  o[2 * lane] = make_float4(acc_a[0] * inv, acc_a[1] * inv, acc_a[2] * inv, acc_a[3] * inv);
  o[2 * lane + 1] = make_float4(acc_a[4] * inv, acc_a[5] * inv, acc_a[6] * inv, acc_a[7] * inv);
  o[64 + 2 * lane] = make_float4(acc_b[0] * inv, acc_b[1] * inv, acc_b[2] * inv, acc_b[3] * inv);
  o[64 + 2 * lane + 1] = make_float4(acc_b[4] * inv, acc_b[5] * inv, acc_b[6] * inv, acc_b[7] * inv);
  if (lane == 0) *lse_out = (m + __log2f(lsum)) * 0.69314718055994530942f;
}

}  // namespace

cudaError_t launch_split_simt(const SplitArgs& a, dim3 grid, cudaStream_t stream) {
  split_simt_kernel<<<grid, 32 * kSimtRowsPerCta, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlav
