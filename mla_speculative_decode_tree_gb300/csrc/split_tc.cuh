// Tensor-core (tcgen05) split kernel for MLA tree-verify attention.
//
// One CTA computes, for one request b, one chunk s of its keys and one group
// of NQ query rows (token, head pairs; row r = i*H + h), the partial softmax
// statistics the merge kernel combines [Custom sm_120 Verify Kernel,
// §"Building the Custom Kernel: From Occupancy Starvation to Flash-Decode"].
//
// Orientation.  An fp32 O accumulator for 128 query rows x 512 latent columns
// would fill all of tensor memory (128 lanes x 512 columns), so the kernel
// keeps the transposed problem: keys (128 per tile) sit on the MMA's M
// dimension and the NQ query rows on N.
//   S^T[128 x NQ]       = K_tile[128 x 576] . Q^T        (36 MMAs, K = 16)
//   O^T[4 x 128 x NQ]  += V^T_tile[512 x 128] . P^T      (4 M-blocks x 8 MMAs)
// TMEM columns: O^T block m at [m*S_o, m*S_o + NQ) with S_o = NQ rounded up
// to 32, then one or two S^T buffers of NQ columns (two when they fit, so the
// next tile's scores can be computed while the softmax reads this tile's).
//
// Shared memory holds Q (9 blocks of NQ rows x 64 columns, 128-byte
// swizzled, K-major), P^T (NQ rows x 128 keys, K-major) and a ring of 16 KB
// slots, each 128 keys x 64 columns of the gathered pool rows in the
// 128-byte-swizzle atom (8 keys x 128 bytes).  That atom is at once the
// K-major layout of the key operand and the MN-major layout of the value
// operand, so the value blocks need no transposition.  The value blocks of a
// tile are fetched a second time (after the next tile's key blocks) rather
// than kept resident: a whole 128-key tile (144 KB) does not fit next to Q.
//
// Warp roles (224 threads):
//   warps 0-3  softmax: TMEM lane quadrant w holds keys 32w..32w+31 of S^T.
//              The scores stay in TMEM and are read in 32-column groups by
//              short loops (a straight-line pass over all columns would not
//              stay in the instruction cache): pass 1 masks and checks them
//              against the running max, which is raised only when a score
//              exceeds it by more than kTau in base 2 (then the exact column
//              max is reduced and O^T rescaled in TMEM); pass 2 writes
//              P = exp2(s - m) as bf16 into P^T.  Epilogue: O = O^T / l, LSE.
//   warp 4     TMEM allocation and the single MMA-issuing thread.
//   warps 5-6  gather: cp.async 16-byte copies of the rows the split needs,
//              resolved from kv_indices (prefix) or out_cache_loc (drafts)
//              [Capture Safety to MoE Ceiling, §"The Architecture of Capture
//              Safety"] into shared memory, each row's 64-column block placed
//              in swizzled order.
// Block sequence through the ring: K(0), K(1), V(0), K(2), V(1), ...,
// K(nt-1), V(nt-2), V(nt-1), where K(t) is the 9 column blocks of tile t and
// V(t) its first 8 in pairs (one M=128 block of latent columns per pair).  A
// pair must occupy adjacent slots, so an empty slot is inserted whenever a
// pair would start in the last slot; producer and consumer apply the same rule.
//
// Every wait is bounded (mbar_wait); on a timeout the CTA raises the status
// bit, all roles drain, the in-flight MMAs are awaited and TMEM is freed.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace mlav {

constexpr int kTcThreads = 224;
constexpr int kSoftmaxThreads = 128;
constexpr int kMmaWarp = 4;
constexpr int kProducerWarp0 = 5;
constexpr int kProducerThreads = 64;
constexpr float kTau = 8.0f;  // base-2 headroom before the running max is raised

template <int NQ>
struct TcCfg {
  static_assert(NQ % 16 == 0 && NQ >= 16 && NQ <= 96, "NQ must be a multiple of 16 in [16, 96]");
  static constexpr int kQBlock = NQ * 128;  // one 64-column block of Q
  static constexpr int kQBytes = 9 * kQBlock;
  static constexpr int kPRegion = NQ * 128;  // P^T keys 0..63 or 64..127
  static constexpr int kPBytes = 2 * kPRegion;
  static constexpr int kSlotBytes = 128 * 128;
  static constexpr int kStages = NQ >= 96 ? 5 : NQ >= 80 ? 6 : NQ >= 64 ? 8 : NQ >= 48 ? 9 : NQ >= 32 ? 10 : 12;
  static constexpr int kOffP = kQBytes;
  static constexpr int kOffRing = kQBytes + kPBytes;
  static constexpr int kOffCtl = kOffRing + kStages * kSlotBytes;
  static constexpr int kOStride = (NQ + 31) / 32 * 32;  // TMEM columns per O^T block (32-aligned)
  static constexpr int kColS = 4 * kOStride;
  static constexpr int kSBuf = (kColS + 2 * NQ <= 512) ? 2 : 1;  // S^T buffers
  static constexpr int kGroups = (NQ + 31) / 32;                 // 32-column groups
};

template <int NQ>
struct TcCtl {
  uint64_t full[TcCfg<NQ>::kStages];
  uint64_t empty[TcCfg<NQ>::kStages];
  uint64_t s_full[2], s_free[2];
  uint64_t q_full, p_full, pv_done, mma_idle;
  uint32_t tmem_base;
  int abort;
  int flag[2][4];
  int rflag[2];
  alignas(16) float mtau[NQ];   // running max + kTau (base 2); -inf before any visible key
  alignas(16) float muse[NQ];   // running max, 0 while it is -inf (all P of the column are 0 then)
  alignas(16) float alpha[NQ];  // rescale factor of the current tile; 1/l in the epilogue
  alignas(16) float red[4][NQ];
  int rowid[2][kKeysPerTile];   // pool rows of the current / previous tile (-1: zero fill)
  uint32_t colmask[kMaxQLen][TcCfg<NQ>::kGroups];  // columns owned by each token of the group
};

template <int NQ>
constexpr int tc_smem_bytes() {
  return TcCfg<NQ>::kOffCtl + (int)sizeof(TcCtl<NQ>) + 1024;  // + alignment slack
}

// Bounded wait that ignores the abort flag (teardown only).
__device__ __forceinline__ void mbar_wait_teardown(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Sum (or max) of v[0..31] over the 32 lanes of the warp, column by column,
// by recursive halving: at offset o each lane keeps the half of its values
// whose index bit o matches its own lane bit and combines it with the
// partner's copy.  Lane L returns the result for index L.
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int m = 0; m < o; ++m) {
      const float send = upper ? v[m] : v[m + o];
      const float keep = upper ? v[m + o] : v[m];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[m] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

// Scores of one 32-column group from TMEM (columns past NQ are not read).
template <int NQ>
__device__ __forceinline__ void load_group(uint32_t taddr, int g, float (&v)[32]) {
  tc::tmem_ld16(taddr, *reinterpret_cast<float(*)[16]>(&v[0]));
  if (32 * g + 16 < NQ) {
    tc::tmem_ld16(taddr + 16, *reinterpret_cast<float(*)[16]>(&v[16]));
  } else {
#pragma unroll
    for (int k = 16; k < 32; ++k) v[k] = 0.f;
  }
  tc::tmem_wait_ld();
}

template <int NQ>
__global__ void __launch_bounds__(kTcThreads, 1) split_tc_kernel(SplitArgs a) {
  using Cfg = TcCfg<NQ>;
  constexpr int S = Cfg::kStages;
  constexpr int SB = Cfg::kSBuf;
  const int b = blockIdx.z;
  if (b >= a.batch) return;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int s_idx = blockIdx.y;
  const int g = blockIdx.x;

  const int64_t kv_base = a.kv_indptr[b];
  const int64_t P = (int64_t)a.kv_indptr[b + 1] - kv_base;
  const int64_t L = P + a.T;
  const int64_t chunk = chunk_len(L, a.nsplit);
  const int64_t j0 = (int64_t)s_idx * chunk;
  const int64_t j1 = (j0 + chunk < L) ? j0 + chunk : L;
  const int rows_b = a.T * a.H;
  const int r0 = g * NQ;
  if (r0 >= rows_b) return;
  const int nrows = (rows_b - r0 < NQ) ? rows_b - r0 : NQ;
  const int64_t grow0 = (int64_t)b * rows_b + r0;
  float* lse_out = a.part_lse + (int64_t)s_idx * a.rows_max + grow0;
  if (j0 >= j1) {
    for (int n = tid; n < nrows; n += kTcThreads) lse_out[n] = -INFINITY;
    return;
  }
  const int nt = (int)((j1 - j0 + kKeysPerTile - 1) / kKeysPerTile);
  const int i0 = r0 / a.H;
  const int ntok = (r0 + nrows - 1) / a.H - i0 + 1;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  const uint32_t sQ = sbase, sP = sbase + Cfg::kOffP, sRing = sbase + Cfg::kOffRing;
  TcCtl<NQ>& ctl = *reinterpret_cast<TcCtl<NQ>*>(smem + Cfg::kOffCtl);

  // ---- set-up ---------------------------------------------------------------
  if (tid == 0) {
    for (int k = 0; k < S; ++k) {
      mbar_init(&ctl.full[k], kProducerThreads);
      mbar_init(&ctl.empty[k], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&ctl.s_full[k], 1);
      mbar_init(&ctl.s_free[k], 4);
    }
    mbar_init(&ctl.q_full, kProducerThreads);
    mbar_init(&ctl.p_full, 4);
    mbar_init(&ctl.pv_done, 1);
    mbar_init(&ctl.mma_idle, 1);
    ctl.abort = 0;
    ctl.rflag[0] = ctl.rflag[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&ctl.tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (tid < kSoftmaxThreads) {
    for (int n = tid; n < NQ; n += kSoftmaxThreads) {
      ctl.mtau[n] = -INFINITY;
      ctl.muse[n] = 0.f;
    }
    for (int t = tid; t < ntok * Cfg::kGroups; t += kSoftmaxThreads) {
      const int tok = t / Cfg::kGroups, w = t % Cfg::kGroups;
      uint32_t bits = 0;
      for (int c = 0; c < 32; ++c) {
        const int n = 32 * w + c;
        if (n < nrows && (r0 + n) / a.H == i0 + tok) bits |= 1u << c;
      }
      ctl.colmask[tok][w] = bits;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;

  if (warp >= kProducerWarp0) {
    // =========================== gather ======================================
    const int pw = warp - kProducerWarp0;
    const int ptid = tid - kProducerWarp0 * 32;
    // Q rows of the group (zero-filled past the last row): 72 chunks of 16
    // bytes per row, 64 from q_nope and 8 from q_rope.
#pragma unroll 2
    for (int idx = ptid; idx < NQ * 72; idx += kProducerThreads) {
      const int n = idx / 72, c = idx - n * 72;
      const bool ok = n < nrows;
      const __nv_bfloat16* src =
          !ok ? a.q_nope : (c < 64 ? a.q_nope + (grow0 + n) * kDLatent + c * 8 : a.q_rope + (grow0 + n) * kDRope + (c - 64) * 8);
      cp_async16(sQ + (c >> 3) * Cfg::kQBlock + n * 128 + (((c & 7) ^ (n & 7)) << 4), src, ok ? 16u : 0u);
    }
    cp_async_arrive(&ctl.q_full);

    int seq = 0;
    bool stop = false;
    uint32_t bad = 0;
    const int c8 = lane & 7;
    const int jl = 4 * pw + (lane >> 3);  // key index mod 8 this lane copies
    const uint32_t lane_off = jl * 128 + ((c8 ^ jl) << 4);
    // Row ids of the keys this warp copies (keys with bit 2 == pw), two per lane.
    auto resolve = [&](int t) {
      const int it = lane >> 1;
      const int q0 = 2 * (lane & 1);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int jj = 8 * it + 4 * pw + q0 + q;
        const int64_t j = j0 + (int64_t)t * kKeysPerTile + jj;
        int row = -1;
        if (j < j1) {
          const int64_t rr = resolve_row(a, b, P, kv_base, j);
          if (rr < 0) bad = 1;
          row = (int)rr;
        }
        ctl.rowid[t & 1][jj] = row;
      }
      __syncwarp();
    };
    // Fill one ring slot (blk < 0: the empty filler slot).  Each thread's
    // copies are published by an asynchronous arrival on full[slot] that
    // fires when they have landed, so this warp never waits for memory, only
    // for a free slot.
    auto produce = [&](int blk, int t) {
      if (stop) return;
      const int slot = seq % S;
      if (!mbar_wait(&ctl.empty[slot], ((seq / S) & 1) ^ 1, &ctl.abort, a.status)) {
        stop = true;
        return;
      }
      if (blk >= 0) {
        const uint32_t dst0 = sRing + slot * Cfg::kSlotBytes + lane_off;
        const __nv_bfloat16* base = a.kv_pool + blk * 64 + c8 * 8;
        const int* rid = &ctl.rowid[t & 1][jl];
#pragma unroll 4
        for (int it = 0; it < 16; ++it) {
          const int row = rid[8 * it];
          cp_async16(dst0 + it * 1024, row >= 0 ? base + (int64_t)row * kDRow : a.kv_pool, row >= 0 ? 16u : 0u);
        }
        cp_async_arrive(&ctl.full[slot]);
      } else {
        mbar_arrive(&ctl.full[slot]);
      }
      ++seq;
    };
    for (int t = 0; t <= nt && !stop; ++t) {
      if (t < nt) {
        resolve(t);
#pragma unroll 1
        for (int blk = 0; blk < 9; ++blk) produce(blk, t);
      }
      if (t >= 1) {
#pragma unroll 1
        for (int pr = 0; pr < 4; ++pr) {
          if (seq % S == S - 1) produce(-1, t - 1);
          produce(2 * pr, t - 1);
          produce(2 * pr + 1, t - 1);
        }
      }
    }
    cp_async_wait_all();  // nothing in flight when the CTA exits
    if (bad) atomicOr(a.status, kStatusBadRow);
  } else if (warp == kMmaWarp) {
    // ============================ MMA issue ==================================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, NQ, false, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(128, NQ, true, false);
      int seq = 0;
      // cp.async writes shared memory through the generic proxy and the MMA
      // reads it through the async proxy: a proxy fence follows each acquire.
      bool ok = mbar_wait(&ctl.q_full, 0, &ctl.abort, a.status);
      fence_proxy_async_smem();
      auto take = [&](int& slot) -> bool {
        slot = seq % S;
        const bool r = mbar_wait(&ctl.full[slot], (seq / S) & 1, &ctl.abort, a.status);
        fence_proxy_async_smem();
        tc::fence_after_sync();
        return r;
      };
      for (int t = 0; t <= nt && ok; ++t) {
        if (t < nt) {
          // S^T(t) into buffer t % SB once the softmax released it (tile t - SB).
          const int sb = t % SB;
          if (t >= SB) {
            ok = mbar_wait(&ctl.s_free[sb], ((t / SB) & 1) ^ 1, &ctl.abort, a.status);
            tc::fence_after_sync();
            if (!ok) break;
          }
          const uint32_t d_s = tmem + Cfg::kColS + sb * NQ;
#pragma unroll 1
          for (int blk = 0; blk < 9 && ok; ++blk) {
            int slot;
            if (!(ok = take(slot))) break;
            ++seq;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t adesc = tc::smem_desc(sRing + slot * Cfg::kSlotBytes + k * 32, 16, 1024, tc::kSwizzle128B);
              const uint64_t bdesc = tc::smem_desc(sQ + blk * Cfg::kQBlock + k * 32, 16, 1024, tc::kSwizzle128B);
              tc::mma_bf16_ss(d_s, adesc, bdesc, idesc_qk, (blk | k) ? 1u : 0u);
            }
            tc::mma_commit(&ctl.empty[slot]);
          }
          if (!ok) break;
          tc::mma_commit(&ctl.s_full[sb]);
        }
        if (t >= 1) {
          // O^T += V^T(t-1) . P^T(t-1)
          const int u = t - 1;
          ok = mbar_wait(&ctl.p_full, u & 1, &ctl.abort, a.status);
          tc::fence_after_sync();
#pragma unroll 1
          for (int m = 0; m < 4 && ok; ++m) {
            int sa, sb2;
            if (seq % S == S - 1) {
              if (!(ok = take(sa))) break;
              mbar_arrive(&ctl.empty[sa]);
              ++seq;
            }
            if (!(ok = take(sa))) break;
            ++seq;
            if (!(ok = take(sb2))) break;
            ++seq;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t adesc =
                  tc::smem_desc(sRing + sa * Cfg::kSlotBytes + kk * 2048, Cfg::kSlotBytes, 1024, tc::kSwizzle128B);
              const uint64_t bdesc =
                  tc::smem_desc(sP + (kk >> 2) * Cfg::kPRegion + (kk & 3) * 32, 16, 1024, tc::kSwizzle128B);
              tc::mma_bf16_ss(tmem + m * Cfg::kOStride, adesc, bdesc, idesc_pv, (u > 0 || kk > 0) ? 1u : 0u);
            }
            tc::mma_commit(&ctl.empty[sa]);
            tc::mma_commit(&ctl.empty[sb2]);
          }
          if (ok) tc::mma_commit(&ctl.pv_done);
        }
      }
      // Drain: every MMA this thread issued has completed before TMEM is freed.
      tc::mma_commit(&ctl.mma_idle);
      mbar_wait_teardown(&ctl.mma_idle, 0);
    }
    __syncwarp();
  } else {
    // ============================ softmax ====================================
    const int j = tid;  // key within the tile == TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(32 * warp) << 16);
    const int64_t mask_base = (int64_t)a.mask_indptr[b] + (int64_t)i0 * L;
    const float scale = a.scale_log2;
    // Thread n < NQ owns the running sum of query column n over the bf16 P
    // values fed to the MMA; it normalises O, so the weights of a split sum to
    // one exactly.  LSE needs the sum of the unrounded P: lane L of each warp
    // also keeps, for columns L, L+32, L+64, the sum over its warp's keys of
    // the rounding residuals p - bf16(p).
    float l_col = 0.f;
    float l_res0 = 0.f, l_res1 = 0.f, l_res2 = 0.f;
    // P^T is the K-major B operand [NQ rows x 128 keys]: key j lives in region
    // j/64, 16-byte chunk (j%64)/8 (swizzled by row), element j%8.
    const uint32_t pbase = sP + (j >> 6) * Cfg::kPRegion + (j & 7) * 2;
    const uint32_t jc = (j >> 3) & 7;
    bool my_abort = false;
#pragma unroll 1
    for (int t = 0; t < nt; ++t) {
      const int sb = t % SB;
      const uint32_t s_addr = t_lane + Cfg::kColS + sb * NQ;
      const int64_t key = j0 + (int64_t)t * kKeysPerTile + j;
      uint32_t vis0 = 0, vis1 = 0, vis2 = 0;
      if (key < j1) {
        for (int tl = 0; tl < ntok; ++tl) {
          if (mask_bit(a.mask, mask_base + (int64_t)tl * L + key)) {
            vis0 |= ctl.colmask[tl][0];
            if (Cfg::kGroups > 1) vis1 |= ctl.colmask[tl][Cfg::kGroups > 1 ? 1 : 0];
            if (Cfg::kGroups > 2) vis2 |= ctl.colmask[tl][Cfg::kGroups > 2 ? 2 : 0];
          }
        }
      }
      if (!my_abort) my_abort = !mbar_wait(&ctl.s_full[sb], (t / SB) & 1, &ctl.abort, a.status);
      tc::fence_after_sync();

      // ---- pass 1: does any score pass the running max by more than kTau?
      bool need = false;
      if (!my_abort) {
#pragma unroll 1
        for (int gq = 0; gq < Cfg::kGroups; ++gq) {
          float v[32];
          load_group<NQ>(s_addr + 32 * gq, gq, v);
          const uint32_t vw = gq == 0 ? vis0 : (gq == 1 ? vis1 : vis2);
          const float* mt = &ctl.mtau[32 * gq];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            if (32 * gq + k < NQ) need |= ((vw >> k) & 1u) && (v[k] * scale > mt[k]);
          }
        }
      }
      const bool warp_need = __any_sync(0xffffffffu, need);
      const bool warp_abort = __any_sync(0xffffffffu, my_abort) || ctl.abort;
      if (lane == 0) ctl.flag[t & 1][warp] = (warp_need ? 1 : 0) | (warp_abort ? 2 : 0);
      named_bar_sync(1, kSoftmaxThreads);
      const int f = ctl.flag[t & 1][0] | ctl.flag[t & 1][1] | ctl.flag[t & 1][2] | ctl.flag[t & 1][3];
      if (tid == 0) ctl.rflag[(t + 1) & 1] = 0;
      if (f & 2) {
        my_abort = true;
        break;
      }
      bool rescale = false;
      if (f & 1) {
        // Exact column max over the tile's 128 keys; raise the running max
        // where it passed by more than kTau.
#pragma unroll 1
        for (int gq = 0; gq < Cfg::kGroups; ++gq) {
          float v[32];
          load_group<NQ>(s_addr + 32 * gq, gq, v);
          const uint32_t vw = gq == 0 ? vis0 : (gq == 1 ? vis1 : vis2);
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = ((vw >> k) & 1u) ? v[k] * scale : -INFINITY;
          const float cm = warp_transpose_reduce<true>(v, lane);
          if (32 * gq + lane < NQ) ctl.red[warp][32 * gq + lane] = cm;
        }
        named_bar_sync(1, kSoftmaxThreads);
        if (tid < NQ) {
          const float cm = fmaxf(fmaxf(ctl.red[0][tid], ctl.red[1][tid]), fmaxf(ctl.red[2][tid], ctl.red[3][tid]));
          const float old = ctl.mtau[tid];  // -inf or max + kTau
          float al = 1.f;
          if (cm > old) {
            al = (old == -INFINITY) ? 0.f : ex2_approx(old - kTau - cm);
            ctl.mtau[tid] = cm + kTau;
            ctl.muse[tid] = cm;
            ctl.rflag[t & 1] = 1;
          }
          ctl.alpha[tid] = al;
          l_col *= al;
        }
        named_bar_sync(1, kSoftmaxThreads);
        if (lane < NQ) l_res0 *= ctl.alpha[lane];
        if (32 + lane < NQ) l_res1 *= ctl.alpha[32 + lane];
        if (64 + lane < NQ) l_res2 *= ctl.alpha[64 + lane];
        rescale = (t > 0) && ctl.rflag[t & 1];
      }
      // PV of the previous tile must be done before P^T and O^T are touched.
      if (t >= 1 && !my_abort) my_abort = !mbar_wait(&ctl.pv_done, (t - 1) & 1, &ctl.abort, a.status);
      tc::fence_after_sync();
      if (!my_abort && rescale) {
#pragma unroll 1
        for (int c = 0; c < NQ / 16; ++c) {
          bool any = false;
#pragma unroll
          for (int k = 0; k < 16; ++k) any |= ctl.alpha[16 * c + k] != 1.f;
          if (!any) continue;
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
            float v[16];
            tc::tmem_ld16(t_lane + m * Cfg::kOStride + 16 * c, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] *= ctl.alpha[16 * c + k];
            tc::tmem_st16(t_lane + m * Cfg::kOStride + 16 * c, v);
          }
        }
        tc::tmem_wait_st();
      }

      // ---- pass 2: P = exp2(s - m) -> bf16 into P^T; residual sums for LSE.
      if (!my_abort) {
#pragma unroll 1
        for (int gq = 0; gq < Cfg::kGroups; ++gq) {
          float v[32];
          load_group<NQ>(s_addr + 32 * gq, gq, v);
          const uint32_t vw = gq == 0 ? vis0 : (gq == 1 ? vis1 : vis2);
          const float* mu = &ctl.muse[32 * gq];
          const uint32_t prow = pbase + 32 * gq * 128;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            float r = 0.f;
            if (32 * gq + k < NQ) {
              const float x = ((vw >> k) & 1u) ? fmaf(v[k], scale, -mu[k]) : -INFINITY;
              const float p = ex2_approx(x);
              const __nv_bfloat16 hb = __float2bfloat16_rn(p);
              const uint16_t hv = *reinterpret_cast<const uint16_t*>(&hb);
              asm volatile("st.shared.u16 [%0], %1;" ::"r"(prow + k * 128 + ((jc ^ (uint32_t)(k & 7)) << 4)), "h"(hv)
                           : "memory");
              r = p - __bfloat162float(hb);
            }
            v[k] = r;
          }
          const float rs = warp_transpose_reduce<false>(v, lane);
          if (gq == 0) l_res0 += rs;
          else if (gq == 1) l_res1 += rs;
          else l_res2 += rs;
        }
      }
      // The scores of this tile are no longer needed, nor (after the MMA reads
      // it) P^T; hand the S^T buffer back and P^T to the MMA.
      tc::fence_before_sync();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && !my_abort) {
        mbar_arrive(&ctl.s_free[sb]);
        mbar_arrive(&ctl.p_full);
      }
      // Column sums of this tile's bf16 P (the MMA reads P^T concurrently).
      named_bar_sync(1, kSoftmaxThreads);
      if (tid < NQ && !my_abort) {
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
        for (int k = 0; k < 16; ++k) {
          const int c = (k + tid) & 7;  // staggered: 8 neighbouring rows hit 8 different chunks
          const uint32_t addr = sP + (k >> 3) * Cfg::kPRegion + tid * 128 + c * 16;
          uint32_t w0, w1, w2, w3;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3) : "r"(addr));
          acc0 += __uint_as_float(w0 << 16) + __uint_as_float(w1 << 16) + __uint_as_float(w2 << 16) +
                  __uint_as_float(w3 << 16);
          acc1 += __uint_as_float(w0 & 0xFFFF0000u) + __uint_as_float(w1 & 0xFFFF0000u) +
                  __uint_as_float(w2 & 0xFFFF0000u) + __uint_as_float(w3 & 0xFFFF0000u);
        }
        l_col += acc0 + acc1;
      }
    }

    // ---- epilogue: O = O^T / l, LSE -------------------------------------------
    if (!my_abort) my_abort = !mbar_wait(&ctl.pv_done, (nt - 1) & 1, &ctl.abort, a.status);
    tc::fence_after_sync();
    const bool wa = __any_sync(0xffffffffu, my_abort) || ctl.abort;
    if (lane == 0) ctl.flag[nt & 1][warp] = wa ? 2 : 0;
    if (lane < NQ) ctl.red[warp][lane] = l_res0;
    if (32 + lane < NQ) ctl.red[warp][32 + lane] = l_res1;
    if (64 + lane < NQ) ctl.red[warp][64 + lane] = l_res2;
    named_bar_sync(1, kSoftmaxThreads);
    const int f = ctl.flag[nt & 1][0] | ctl.flag[nt & 1][1] | ctl.flag[nt & 1][2] | ctl.flag[nt & 1][3];
    if (tid < NQ) {
      const float lfull = l_col + ((ctl.red[0][tid] + ctl.red[1][tid]) + (ctl.red[2][tid] + ctl.red[3][tid]));
      ctl.alpha[tid] = l_col > 0.f ? 1.f / l_col : 0.f;
      if (!(f & 2) && tid < nrows)
        lse_out[tid] = l_col > 0.f ? (ctl.muse[tid] + __log2f(lfull)) * 0.69314718055994530942f : -INFINITY;
    }
    named_bar_sync(1, kSoftmaxThreads);
    if (!(f & 2)) {
      float* po = a.part_o + ((int64_t)s_idx * a.rows_max + grow0) * kDLatent + j;
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
#pragma unroll 1
        for (int c = 0; c < NQ / 16; ++c) {
          float v[16];
          tc::tmem_ld16(t_lane + m * Cfg::kOStride + 16 * c, v);
          tc::tmem_wait_ld();
          const float* inv = &ctl.alpha[16 * c];
          float* dst = po + (int64_t)(16 * c) * kDLatent + 128 * m;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            if (16 * c + k < nrows && inv[k] > 0.f) dst[(int64_t)k * kDLatent] = v[k] * inv[k];
          }
        }
      }
    }
    tc::fence_before_sync();
  }

  // ---- teardown ---------------------------------------------------------------
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int NQ>
cudaError_t launch_split_tc_nq(const SplitArgs& a, dim3 grid, cudaStream_t stream) {
  constexpr int smem = tc_smem_bytes<NQ>();
  static_assert(smem <= 232448, "shared memory budget exceeded");
  cudaError_t e = cudaFuncSetAttribute(split_tc_kernel<NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  split_tc_kernel<NQ><<<grid, kTcThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlav
