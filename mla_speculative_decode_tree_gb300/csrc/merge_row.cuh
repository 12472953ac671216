// Log-sum-exp merge of one query row's split partials -- the second
// reduction of the split-K verify [Custom sm_120 Verify Kernel, §"Building
// the Custom Kernel: From Occupancy Starvation to Flash-Decode"] -- shared by
// the merge kernel and the split kernel's fused merge, so both give the same
// bits.
//
//   M = max_s lse_s,  w_s = exp(lse_s - M),
//   O = sum_s w_s O_s / sum_s w_s  (bf16, round-to-nearest-even),
//   LSE = M + ln sum_s w_s;        M = -inf  ->  O = 0, LSE = -inf.
//
// One warp merges one half (256 latent columns) of the row; lane l owns 8
// columns of it.  The lanes first take one split each (lse, weight), then
// the warp walks the splits kMergeUnroll at a time with all their loads in flight,
// the weights broadcast by shuffle.  Splits with lse_s = -inf (empty chunk or
// nothing visible) are skipped without touching their O_s, which the split
// kernel does not write.  kL2Only reads the partials from L2 (ld.global.cg),
// as the fused merge must: other CTAs of the same launch wrote them.  The
// arithmetic does not depend on it.
#pragma once

#include "common.cuh"

namespace mlav {

constexpr int kMergeUnroll = 8;  // divides 32

template <bool kL2Only>
__device__ __forceinline__ float merge_ld(const float* p) {
  if constexpr (kL2Only) return __ldcg(p);
  return *p;
}
template <bool kL2Only>
__device__ __forceinline__ float4 merge_ld4(const float4* p) {
  if constexpr (kL2Only) return __ldcg(p);
  return *p;
}

// nsplit: the splits to read (0..nsplit-1); rows_max: the partials' row stride.
template <bool kL2Only>
__device__ __forceinline__ void merge_row_half(const float* part_lse, const float* part_o, int64_t rows_max,
                                               int nsplit, int64_t row, int half, int lane, __nv_bfloat16* o_out,
                                               float* lse_out) {
  float M = -INFINITY;
  for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, merge_ld<kL2Only>(part_lse + (int64_t)s * rows_max + row));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  const int col = half * (kDLatent / 2) + 8 * lane;
  uint4* o = reinterpret_cast<uint4*>(o_out + row * kDLatent + col);
  if (M == -INFINITY) {
    *o = make_uint4(0, 0, 0, 0);
    if (half == 0 && lane == 0) lse_out[row] = -INFINITY;
    return;
  }

  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
  float W = 0.f;
  const int64_t split_stride = rows_max * kDLatent;
  const float* base = part_o + row * kDLatent + col;
  for (int s0 = 0; s0 < nsplit; s0 += 32) {
    const int s = s0 + lane;
    const float ls = s < nsplit ? merge_ld<kL2Only>(part_lse + (int64_t)s * rows_max + row) : -INFINITY;
    const float wl = ls == -INFINITY ? 0.f : expf(ls - M);
    W += wl;
    const int n = (nsplit - s0 < 32) ? nsplit - s0 : 32;
    for (int k0 = 0; k0 < n; k0 += kMergeUnroll) {
      float wk[kMergeUnroll];
      float4 v[kMergeUnroll][2];
#pragma unroll
      for (int u = 0; u < kMergeUnroll; ++u) {
        wk[u] = __shfl_sync(0xffffffffu, wl, k0 + u);  // 0 past the last split
        if (wk[u] != 0.f) {
          const float4* src = reinterpret_cast<const float4*>(base + (int64_t)(s0 + k0 + u) * split_stride);
          v[u][0] = merge_ld4<kL2Only>(src);
          v[u][1] = merge_ld4<kL2Only>(src + 1);
        } else {
          v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kMergeUnroll; ++u) {
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
  if (half == 0 && lane == 0) lse_out[row] = M + logf(W);
}

// The same merge with one warp per quarter (128 latent columns) of the row,
// lane l owning 4 columns, and the same arithmetic in the same order, so the
// bits equal merge_row_half's.  Splits are taken 16 at a time; with kSpec the
// first 16 splits' partials are loaded before their LSEs are known (one L2
// round trip fewer), and a split with weight 0 -- an empty chunk whose partial
// was never written -- has its loaded values replaced by 0 before use.  The
// loads stay inside the workspace's nsplit partials.
template <bool kSpec>
__device__ __forceinline__ void merge_row_quarter(const float* part_lse, const float* part_o, int64_t rows_max,
                                                  int nsplit, int64_t row, int quarter, int lane,
                                                  __nv_bfloat16* o_out, float* lse_out) {
  constexpr int G = 16;  // splits loaded ahead with kSpec
  constexpr int U = 8;   // splits in flight per step otherwise; both divide 32
  const int col = quarter * (kDLatent / 4) + 4 * lane;
  const int64_t split_stride = rows_max * kDLatent;
  const float* base = part_o + row * kDLatent + col;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 pre[kSpec ? G : 1];
  if constexpr (kSpec) {
#pragma unroll
    for (int u = 0; u < G; ++u)
      pre[u] = u < nsplit ? *reinterpret_cast<const float4*>(base + (int64_t)u * split_stride) : zero;
  }
  float M = -INFINITY;
  for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, part_lse[(int64_t)s * rows_max + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  uint2* o = reinterpret_cast<uint2*>(o_out + row * kDLatent + col);
  if (M == -INFINITY) {
    *o = make_uint2(0, 0);
    if (quarter == 0 && lane == 0) lse_out[row] = -INFINITY;
    return;
  }

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  auto fma4 = [&](float w, const float4& x) {
    acc[0] = fmaf(w, x.x, acc[0]);
    acc[1] = fmaf(w, x.y, acc[1]);
    acc[2] = fmaf(w, x.z, acc[2]);
    acc[3] = fmaf(w, x.w, acc[3]);
  };
  float W = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += 32) {
    const int s = s0 + lane;
    const float ls = s < nsplit ? part_lse[(int64_t)s * rows_max + row] : -INFINITY;
    const float wl = ls == -INFINITY ? 0.f : expf(ls - M);
    W += wl;
    const int n = (nsplit - s0 < 32) ? nsplit - s0 : 32;
    int k0 = 0;
    if (kSpec && s0 == 0) {
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const float w = __shfl_sync(0xffffffffu, wl, u);  // 0 past the last split
        fma4(w, w != 0.f ? pre[u < G ? u : 0] : zero);
      }
      k0 = G;
    }
    for (; k0 < n; k0 += U) {
      float wk[U];
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        wk[u] = __shfl_sync(0xffffffffu, wl, k0 + u);  // 0 past the last split
        v[u] = wk[u] != 0.f ? *reinterpret_cast<const float4*>(base + (int64_t)(s0 + k0 + u) * split_stride) : zero;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) fma4(wk[u], v[u]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
  const float inv = 1.f / W;
  const __nv_bfloat162 h01 = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  const __nv_bfloat162 h23 = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  *o = make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
  if (quarter == 0 && lane == 0) lse_out[row] = M + logf(W);
}

}  // namespace mlav
