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
// to 32, S^T at [4*S_o, 4*S_o + NQ).
//
// Shared memory holds Q (9 blocks of NQ rows x 64 columns, 128-byte
// swizzled, K-major), P^T (NQ rows x 128 keys, K-major) and 16 KB slots, each
// 128 keys x 64 columns of the gathered pool rows in the 128-byte-swizzle
// atom (8 keys x 128 bytes).  That atom is at once the K-major layout of the
// key operand and the MN-major layout of the value operand, so the value
// blocks need no transposition.  A whole 128-key tile (144 KB) fits next to
// Q only for NQ <= 64 (resident mode below); otherwise the slots form a ring
// and a tile's value blocks are fetched a second time, after the next tile's
// key blocks (value-refetch mode).
//
// Warp roles (512 threads; CG = 3 column groups for NQ = 96, else 2):
//   warps 0..4CG-1  softmax.  Warp w reads TMEM lane quadrant w%4 (keys
//              32(w%4)..+31 of the tile) and owns query columns
//              [(w/4)*NQ/CG, (w/4+1)*NQ/CG).  It loads its scores once (the S^T
//              buffer is handed back to the MMA right away), masks them,
//              checks them against the running max -- raised only when a
//              score exceeds it by more than kTau in base 2, after which the
//              exact column max is reduced and O^T rescaled in TMEM -- and
//              writes P = exp2(s - m) as bf16 into P^T.  Per thread and
//              column it accumulates the bf16 P (normalises O) and the fp32
//              rounding residual p - bf16(p) (completes LSE).  Epilogue: O^T
//              scaled by 1/l and stored from TMEM straight to global memory.
//   warp 4CG   TMEM allocation and the single MMA-issuing thread.
//   warps 4CG+1..  gather (at most one per ring slot), taking turns block by
//              block with 16-byte cp.async copies (several warps: one cannot
//              issue them fast enough); rows resolved from kv_indices (prefix)
//              or out_cache_loc (drafts, at the request's token rows)
//              [Capture Safety to MoE Ceiling, §"The Architecture of Capture
//              Safety"]; Q arrives once by 2-D TMA.
// Two ways to feed the tiles (kMode):
//
// kRefetch (up to 96 query rows).  Block sequence through the ring: K(0),
// K(1), V(0), K(2), V(1), ..., K(nt-1), V(nt-2), V(nt-1), where K(t) is the
// 9 column blocks of tile t and V(t) its first 8 in pairs (one M=128 block of
// latent columns per pair).  A pair must occupy adjacent slots, so an empty
// slot is inserted whenever a pair would start in the last slot; producer
// and consumer apply the same rule.
//
// kResident (at most 64 query rows).  Q then takes at most 72 KB, so a whole
// tile fits beside it: nine fixed slots, slot b holding column block b of the
// current tile.  Each key lands once per CTA and feeds both products: QK(t)
// reads all nine blocks; P^T(t) is written into slot 8 (the RoPE block,
// which only QK reads) once QK(t) is complete; PV(t) reads slots 0..7 and
// P^T, releasing the value pair (2m, 2m+1) after M-block m, and slot 8 last.
// The gather refills each slot with the next tile's block as soon as it is
// released.  The MMA thread issues QK(t), PV(t), QK(t+1), ..., so the commit
// that completes S^T(t) also covers PV(t-1): the softmax may rescale O^T and
// write P^T right after it, with no other wait.  The next tile's blocks land
// only after PV(t), so every tile waits out one landing.
//
// Every wait is bounded (mbar_wait, mbar_wait_spin for the MMA thread); on a
// timeout the CTA raises the status bit, all roles drain, the in-flight MMAs
// are awaited and TMEM is freed.
#pragma once

#include "common.cuh"
#include "merge_row.cuh"
#include "tc_ptx.cuh"

namespace mlav {

constexpr float kTau = 8.0f;  // base-2 headroom before the running max is raised

enum TcMode : int { kRefetch = 0, kResident = 1 };

template <int NQ, int kMode>
struct TcCfg {
  static_assert(NQ % 16 == 0 && NQ >= 16 && NQ <= 96, "NQ must be a multiple of 16 in [16, 96]");
  static constexpr bool kLandOnce = kMode != kRefetch;  // each key lands once per CTA
  static_assert(!kLandOnce || NQ <= 64, "resident tiles fit beside Q for at most 64 query rows");
  static constexpr int kKeys = kKeysPerTile;  // keys per tile = M of the QK MMA
  static constexpr int kCG = NQ == 96 ? 3 : 2;  // softmax warps per TMEM lane quadrant
  static constexpr int kHC = NQ / kCG;          // query columns per softmax thread
  static constexpr int kSoftmaxWarps = 4 * kCG;
  static constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps;
  static_assert(kHC % 8 == 0, "columns per softmax thread must be a multiple of 8");
  static constexpr int kQBlock = NQ * 128;  // one 64-column block of Q
  static constexpr int kQBytes = 9 * kQBlock;
  static constexpr int kPRegion = NQ * 128;  // P^T for 64 keys (keys 0..63 or 64..127 of a tile)
  static constexpr int kPBytes = (kKeys / 64) * kPRegion;
  static constexpr int kSlotBytes = kKeys * 128;  // one 64-column block of a tile
  static_assert(!kLandOnce || kPBytes <= kSlotBytes, "P^T must fit in the RoPE block's slot");
  static constexpr int kStages =
      kLandOnce ? 9 : NQ >= 96 ? 5 : NQ >= 64 ? 8 : NQ >= 48 ? 9 : NQ >= 32 ? 11 : 12;
  static constexpr int kOffRing = kLandOnce ? kQBytes : kQBytes + kPBytes;
  // P^T: its own buffer, or (resident) the RoPE block's slot 8
  static constexpr int kOffP = kLandOnce ? kOffRing + 8 * kSlotBytes : kQBytes;
  static constexpr int kOffCtl = kOffRing + kStages * kSlotBytes;
  static constexpr int kOStride = (NQ + 31) / 32 * 32;  // TMEM columns per O^T block (32-aligned)
  static constexpr int kColS = 4 * kOStride;            // S^T
  static_assert(kColS + kOStride <= 512, "TMEM budget");
  // Column sums: thread tid < 2*NQ sums half a row of P^T (64 keys) per
  // tile.  In resident mode these warps release slot 8 together with the MMA.
  static constexpr int kPSumWarps = 2 * NQ / 32;
  // Gather warps: up to 16 warps in all.  kRefetch: no more than ring slots;
  // a warp fills every kProducerWarps-th block, and with more warps than slots
  // it could reach a slot whose empty barrier is two phases behind, where the
  // parity wait cannot tell the phases apart.  kResident: warp w owns slots
  // w, w + kProducerWarps, ... of every tile, so it always waits on a slot it
  // filled itself one tile earlier.
  static constexpr int kProducerWarp = kSoftmaxWarps + 1;
  static constexpr int kProducerWarps = (15 - kSoftmaxWarps) < kStages ? (15 - kSoftmaxWarps) : kStages;
  static_assert(kProducerWarps >= 1 && kProducerWarps <= kStages, "gather warps must not outnumber ring slots");
  static constexpr int kThreads = 32 * (kProducerWarp + kProducerWarps);
};

template <int NQ, int kMode>
struct TcCtl {
  uint64_t full[TcCfg<NQ, kMode>::kStages];
  uint64_t empty[TcCfg<NQ, kMode>::kStages];
  uint64_t q_full, s_full, s_free, p_full, pv_done[2], pv_last, mma_idle;
  uint32_t tmem_base;
  int abort;
  int merge_last;  // fused merge: this CTA is the last of its row group to finish
  int flag[2][12];
  int rflag[2];
  alignas(16) float mtau[NQ];   // running max + kTau (base 2); -inf before any visible key
  alignas(16) float muse[NQ];   // running max, 0 while it is -inf (all P of the column are 0 then)
  alignas(16) float alpha[NQ];  // rescale factor of the current tile; 1/l in the epilogue
  alignas(16) float red[4][NQ];
  alignas(16) float red2[4][NQ];
  uint64_t colmask[kMaxQLen][3];  // per token: which of a column group's columns belong to it
};

template <int NQ, int kMode>
constexpr int tc_smem_bytes() {
  return TcCfg<NQ, kMode>::kOffCtl + (int)sizeof(TcCtl<NQ, kMode>) + 1024;  // + alignment slack
}

// Bounded wait that ignores the abort flag (teardown only).
__device__ __forceinline__ void mbar_wait_teardown(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Sum (or max) of v[0..31] over the 32 lanes of the warp, index by index,
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

// Reduce per-thread column values x[0..HC) over the warp's 32 lanes and store
// the result for column c at dst[c] (lane c%32 of group c/32 writes it).
template <int HC, bool kMax>
__device__ __forceinline__ void warp_columns_to_smem(const float (&x)[HC], float* dst, int lane) {
#pragma unroll
  for (int g = 0; g < (HC + 31) / 32; ++g) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int c = 32 * g + k;
      v[k] = (c < HC) ? x[c < HC ? c : 0] : (kMax ? -INFINITY : 0.f);
    }
    const float r = warp_transpose_reduce<kMax>(v, lane);
    if (32 * g + lane < HC) dst[32 * g + lane] = r;
  }
}

// kFused: the CTA that finishes a row group last also merges it (a separate
// instantiation, so the plain kernel carries none of that code).  kMode:
// how the tiles are fed (see above).
template <int NQ, bool kFused, int kMode>
__global__ void __launch_bounds__(TcCfg<NQ, kMode>::kThreads, 1)
    split_tc_kernel(const __grid_constant__ SplitArgs a, const __grid_constant__ TcMaps maps) {
  using Cfg = TcCfg<NQ, kMode>;
  constexpr bool kLandOnce = Cfg::kLandOnce;
  constexpr int kKeys = Cfg::kKeys;
  constexpr int kM = kKeys / 32;  // row ids per gather lane and tile
  constexpr int S = Cfg::kStages;
  constexpr int HC = Cfg::kHC;
  constexpr int CG = Cfg::kCG;
  constexpr int kSoftmaxWarps = Cfg::kSoftmaxWarps;
  constexpr int kSoftmaxThreads = Cfg::kSoftmaxThreads;
  constexpr int kMmaWarp = Cfg::kMmaWarp;
  constexpr int kProducerWarp = Cfg::kProducerWarp;
  constexpr int kTcThreads = Cfg::kThreads;
  const int b = blockIdx.z;
  if (b >= a.batch) return;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int s_idx = blockIdx.y;
  const int g = blockIdx.x;

  const int64_t kv_base = a.kv_indptr[b];
  const int64_t P = (int64_t)a.kv_indptr[b + 1] - kv_base;
  const RequestTokens rq = request_tokens(a, b);
  const int64_t L = P + rq.n;
  const int64_t chunk = chunk_len(L, a.nsplit, a.min_chunk, a.chunk_granule);
  const int64_t j0 = (int64_t)s_idx * chunk;
  const int64_t j1 = (j0 + chunk < L) ? j0 + chunk : L;
  const int rows_b = rq.n * a.H;
  const int r0 = g * NQ;
  if (r0 >= rows_b) return;
  const int nrows = (rows_b - r0 < NQ) ? rows_b - r0 : NQ;
  const int64_t grow0 = rq.q0 * a.H + r0;  // global row of the group's first row
  float* lse_out = a.part_lse + (int64_t)s_idx * a.rows_max + grow0;
  if (j0 >= j1) {
    for (int n = tid; n < nrows; n += kTcThreads) lse_out[n] = -INFINITY;
    return;
  }
  const int nt = (int)((j1 - j0 + kKeys - 1) / kKeys);
  const int i0 = r0 / a.H;
  const int ntok = (r0 + nrows - 1) / a.H - i0 + 1;
  // The row groups of a split read the same keys; group g starts g tiles
  // into the split (a rotation of the tile order), so the highest group
  // fetches each tile from HBM and the others read it from L2 one or more
  // tiles later, while it is still resident even when the keys of all splits
  // together exceed L2.  The order of the tiles does not change the result
  // beyond rounding, and it is fixed for a given grid.
  const int rot = g % nt;
  auto tile_at = [&](int t) -> int { return t + rot < nt ? t + rot : t + rot - nt; };

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  const uint32_t sQ = sbase, sP = sbase + Cfg::kOffP, sRing = sbase + Cfg::kOffRing;
  TcCtl<NQ, kMode>& ctl = *reinterpret_cast<TcCtl<NQ, kMode>*>(smem + Cfg::kOffCtl);

  // ---- set-up ---------------------------------------------------------------
  if (tid == 0) {
    for (int k = 0; k < S; ++k) {
      mbar_init(&ctl.full[k], 32);  // every lane of the filling warp
      // resident mode: slot 8 (P^T) is free once PV has read it and the
      // column-sum warps are done with it
      mbar_init(&ctl.empty[k], (kLandOnce && k == 8) ? 1 + Cfg::kPSumWarps : 1);
    }
    mbar_init(&ctl.q_full, 1);
    mbar_init(&ctl.s_full, 1);
    mbar_init(&ctl.s_free, kSoftmaxWarps);
    mbar_init(&ctl.p_full, kSoftmaxWarps);
    mbar_init(&ctl.pv_done[0], 1);
    mbar_init(&ctl.pv_done[1], 1);
    mbar_init(&ctl.pv_last, 1);
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
    for (int t = tid; t < ntok * CG; t += kSoftmaxThreads) {
      const int tok = t / CG, h = t % CG;
      uint64_t bits = 0;
      for (int c = 0; c < HC; ++c) {
        const int n = h * HC + c;
        if (n < nrows && (r0 + n) / a.H == i0 + tok) bits |= 1ull << c;
      }
      ctl.colmask[tok][h] = bits;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;

  if (warp >= kProducerWarp) {
    // =========================== gather ======================================
    // Value-refetch mode: the gather warps walk the same block sequence and
    // take turns, warp pw filling the blocks with seq % kProducerWarps == pw.
    // Resident mode: warp pw owns fixed slots.  A block is 128 keys x 64
    // columns: lane (jl = lane/8, c = lane%8) copies 16-byte chunk c of
    // keys 4*it + jl, it = 0..31, into its swizzled place (cp.async, L2 only);
    // the copies of a lane signal full[slot] when they land.
    const int pw = warp - kProducerWarp;
    const int jl = lane >> 3, c8 = lane & 7;
    if (pw == 0 && lane == 0) {
      tma::arrive_expect_tx(&ctl.q_full, 9 * Cfg::kQBlock);
#pragma unroll 1
      for (int blk = 0; blk < 8; ++blk) tma::load_2d(sQ + blk * Cfg::kQBlock, &maps.qn, blk * 64, (int)grow0, &ctl.q_full);
      tma::load_2d(sQ + 8 * Cfg::kQBlock, &maps.qr, 0, (int)grow0, &ctl.q_full);
    }
    // Row ids: lane (jl, c8) resolves keys 4*(c8 + 8m) + jl, m = 0..3, which
    // are exactly the keys lanes 8*jl.. copy at iterations it = c8 + 8m; a
    // shuffle of own[it/8] from lane 8*jl + it%8 hands each copier its row.
    // Keys resolving outside the pool are fetched from the split's first row
    // (finite by contract); keys past the split's end (a closing half tile)
    // are not fetched: their slots are zero-filled.  The softmax masks both.
    // The index loads run a tile ahead of their use (ids of tile t+1 are
    // loaded while tile t is fetched), so no gather warp waits on an index
    // load between tiles.
    auto key_of = [&](int tile, int m) -> int64_t {
      return j0 + (int64_t)tile * kKeys + 4 * (c8 + 8 * m) + jl;
    };
    auto load_ids = [&](int t, int (&raw)[kM]) {
      const int tile = tile_at(t < nt ? t : 0);
#pragma unroll
      for (int m = 0; m < kM; ++m) {
        const int64_t j = key_of(tile, m);
        raw[m] = (t < nt && j < j1) ? load_row_id(a, rq.q0, P, kv_base, j) : -1;
      }
    };
    int64_t rsub = resolve_row(a, rq.q0, P, kv_base, j0);
    int raw_cur[kM], raw_nxt[kM];
    load_ids(0, raw_cur);
    load_ids(1, raw_nxt);
    if (rsub < 0) rsub = 0;
    int own[kM], prev[kM];
#pragma unroll
    for (int m = 0; m < kM; ++m) own[m] = prev[m] = 0;
    uint32_t bad = 0;
    // Rows of tile t (tile_at(t)) into own[], the previous tile's into prev[];
    // then the index loads of tile t+2 are issued.
    auto next_rows = [&](int t) {
      const int tile = tile_at(t);
#pragma unroll
      for (int m = 0; m < kM; ++m) {
        prev[m] = own[m];
        int64_t rr = -1;  // past the split's end
        if (key_of(tile, m) < j1) {
          if (raw_cur[m] >= 0 && raw_cur[m] < a.pool_rows) {
            rr = raw_cur[m];
          } else {
            rr = rsub;
            bad = 1;
          }
        }
        own[m] = (int)rr;
        raw_cur[m] = raw_nxt[m];
      }
      load_ids(t + 2, raw_nxt);
    };
    // Column block blk of the keys whose rows r[] holds, into `slot`; the
    // copies of every lane signal full[slot] when they land.
    auto copy_block = [&](int slot, int blk, const int (&r)[kM]) {
      const uint32_t base = sRing + slot * Cfg::kSlotBytes + jl * 128;
      const __nv_bfloat16* src0 = a.kv_pool + blk * 64 + c8 * 8;
#pragma unroll
      for (int it = 0; it < kKeys / 4; ++it) {
        const int row = __shfl_sync(0xffffffffu, r[it >> 3], 8 * jl + (it & 7));
        const int swz = (c8 ^ (4 * (it & 1) + jl)) << 4;  // key (4*it + jl) mod 8 = 4*(it%2) + jl
        // row < 0: zero-fill, nothing read (the address stays inside the pool)
        cp_async16(base + it * 512 + swz, src0 + (int64_t)(row < 0 ? 0 : row) * kDRow, row < 0 ? 0u : 16u);
      }
      cp_async_arrive(&ctl.full[slot]);
    };
    bool stop = false;
    if constexpr (kLandOnce) {
      // Warp pw fills slots pw, pw + kProducerWarps, ... of every tile, each
      // once the previous tile has released it.
#pragma unroll 1
      for (int t = 0; t < nt && !stop; ++t) {
        next_rows(t);
#pragma unroll 1
        for (int blk = pw; blk < 9; blk += Cfg::kProducerWarps) {
          const bool got = mbar_wait(&ctl.empty[blk], (t & 1) ^ 1, &ctl.abort, a.status);
          if (!__all_sync(0xffffffffu, got)) {
            stop = true;
            break;
          }
          if (!(a.test_stall && t == 0 && blk == 0)) copy_block(blk, blk, own);  // test only: block 0 never lands
        }
      }
    } else {
      int seq = 0;
      auto produce = [&](int blk, const int (&r)[kM]) {
        if (stop) return;
        if (seq % Cfg::kProducerWarps != pw) {
          ++seq;
          return;
        }
        const int slot = seq % S;
        // every lane acquires the slot; the warp stops together if any gave up
        const bool got = mbar_wait(&ctl.empty[slot], ((seq / S) & 1) ^ 1, &ctl.abort, a.status);
        if (!__all_sync(0xffffffffu, got)) {
          stop = true;
          return;
        }
        if (a.test_stall && seq == 0) {
          // test only: block 0 is never filled nor signalled
        } else if (blk >= 0) {
          copy_block(slot, blk, r);
        } else {
          mbar_arrive(&ctl.full[slot]);
        }
        ++seq;
      };
#pragma unroll 1
      for (int t = 0; t <= nt && !stop; ++t) {
        if (t < nt) {
          next_rows(t);
#pragma unroll 1
          for (int blk = 0; blk < 9; ++blk) produce(blk, own);
        }
        if (t >= 1) {
          // value blocks of tile t-1: its rows are in prev[] (or still in own[]
          // after the last tile)
          const bool last = (t == nt);
#pragma unroll 1
          for (int pr = 0; pr < 4; ++pr) {
            if (seq % S == S - 1) produce(-1, own);
            produce(2 * pr, last ? own : prev);
            produce(2 * pr + 1, last ? own : prev);
          }
        }
      }
    }
    cp_async_wait_all();  // nothing in flight when the CTA exits
    if (bad) atomicOr(a.status, kStatusBadRow);
  } else if (warp == kMmaWarp) {
    // ============================ MMA issue ==================================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kKeys, NQ, false, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(128, NQ, true, false);
      bool ok = mbar_wait_spin(&ctl.q_full, 0, &ctl.abort, a.status);
      // cp.async writes shared memory through the generic proxy and the MMA
      // reads it through the async proxy: a proxy fence follows each acquire.
      auto fences = [&]() {
        fence_proxy_async_smem();
        tc::fence_after_sync();
      };
      // S^T (+)= K block (slot) . Q block blk^T
      auto qk_block = [&](int slot, int blk, bool first) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t adesc = tc::smem_desc(sRing + slot * Cfg::kSlotBytes + k * 32, 16, 1024, tc::kSwizzle128B);
          const uint64_t bdesc = tc::smem_desc(sQ + blk * Cfg::kQBlock + k * 32, 16, 1024, tc::kSwizzle128B);
          tc::mma_bf16_ss(tmem + Cfg::kColS, adesc, bdesc, idesc_qk, (first && k == 0) ? 0u : 1u);
        }
      };
      // O^T block m (+)= V^T (slots sa, sa+1) . P^T
      auto pv_block = [&](int m, int sa, bool first) {
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t adesc =
              tc::smem_desc(sRing + sa * Cfg::kSlotBytes + kk * 2048, Cfg::kSlotBytes, 1024, tc::kSwizzle128B);
          const uint64_t bdesc =
              tc::smem_desc(sP + (kk >> 2) * Cfg::kPRegion + (kk & 3) * 32, 16, 1024, tc::kSwizzle128B);
          tc::mma_bf16_ss(tmem + m * Cfg::kOStride, adesc, bdesc, idesc_pv, (first && kk == 0) ? 0u : 1u);
        }
      };
      // A slot is free again once the MMAs reading it are done.
      auto release = [&](int slot) { tc::mma_commit(&ctl.empty[slot]); };
      if constexpr (kLandOnce) {
#pragma unroll 1
        for (int t = 0; t < nt && ok; ++t) {
          // QK(t): block b from slot b, in the order PV(t-1) released them
#pragma unroll 1
          for (int blk = 0; blk < 9; ++blk) {
            if (!(ok = mbar_wait_spin(&ctl.full[blk], t & 1, &ctl.abort, a.status))) break;
            fences();
            qk_block(blk, blk, blk == 0);
          }
          if (!ok) break;
          tc::mma_commit(&ctl.s_full);  // also covers PV(t-1): O^T and slot 8 are the softmax's now
          ok = mbar_wait_spin(&ctl.p_full, t & 1, &ctl.abort, a.status);
          tc::fence_after_sync();
          if (!ok) break;
          // PV(t), releasing each value pair after its M-block and slot 8 last
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
            pv_block(m, 2 * m, t == 0);
            release(2 * m);
            release(2 * m + 1);
          }
          release(8);
        }
        if (ok) tc::mma_commit(&ctl.pv_last);
      } else {
        int seq = 0;
        auto wait_full = [&](int& slot) -> bool {
          slot = seq % S;
          return mbar_wait_spin(&ctl.full[slot], (seq / S) & 1, &ctl.abort, a.status);
        };
#pragma unroll 1
        for (int t = 0; t <= nt && ok; ++t) {
          if (t < nt) {
            // S^T(t) once the softmax has read S^T(t-1) out of TMEM.
            if (t >= 1) {
              ok = mbar_wait_spin(&ctl.s_free, (t - 1) & 1, &ctl.abort, a.status);
              tc::fence_after_sync();
              if (!ok) break;
            }
#pragma unroll 1
            for (int blk = 0; blk < 9 && ok; ++blk) {
              int slot;
              if (!(ok = wait_full(slot))) break;
              fences();
              ++seq;
              qk_block(slot, blk, blk == 0);
              release(slot);
            }
            if (!ok) break;
            tc::mma_commit(&ctl.s_full);
          }
          if (t >= 1) {
            // O^T += V^T(t-1) . P^T(t-1)
            const int u = t - 1;
            ok = mbar_wait_spin(&ctl.p_full, u & 1, &ctl.abort, a.status);
            tc::fence_after_sync();
#pragma unroll 1
            for (int m = 0; m < 4 && ok; ++m) {
              int sa, sb;
              if (seq % S == S - 1) {  // filler slot: nothing to read
                if (!(ok = wait_full(sa))) break;
                release(sa);
                ++seq;
              }
              // one fence after both halves of the pair have landed
              if (!(ok = wait_full(sa))) break;
              ++seq;
              if (!(ok = wait_full(sb))) break;
              ++seq;
              fences();
              pv_block(m, sa, u == 0);
              release(sa);
              release(sb);
            }
            if (ok) tc::mma_commit(&ctl.pv_done[u & 1]);
          }
        }
      }
      // Drain: every MMA this thread issued has completed before TMEM is freed.
      tc::mma_commit(&ctl.mma_idle);
      mbar_wait_teardown(&ctl.mma_idle, 0);
    }
    __syncwarp();
  } else {
    // ============================ softmax ====================================
    const int quad = warp & 3;
    const int half = warp >> 2;  // column group
    const int j = 32 * quad + lane;  // key within the tile == TMEM lane
    const int c0 = half * HC;        // first query column of this thread
    const uint32_t t_lane = tmem + ((uint32_t)(32 * quad) << 16);
    const int64_t mask_base = (int64_t)a.mask_indptr[b] + (int64_t)i0 * L;
    const float scale = a.scale_log2;
    // Column sums.  Thread tid < 2*NQ sums half-row tid of P^T (column tid/2,
    // keys 64*(tid%2)..+63) over the tiles: the bf16 P fed to the MMA, which
    // normalises O so a split's weights sum to one exactly.  Each thread also
    // keeps, per own column, the fp32 residuals p - bf16(p) of its key, for
    // LSE from the unrounded sum.
    float l_half = 0.f;
    float acc_r[HC];
#pragma unroll
    for (int k = 0; k < HC; ++k) acc_r[k] = 0.f;
    // P^T is the K-major B operand [NQ rows x 128 keys]: key j lives in region
    // j/64, 16-byte chunk (j%64)/8 (swizzled by row), element j%8.
    const uint32_t pbase = sP + (j >> 6) * Cfg::kPRegion + (j & 7) * 2 + c0 * 128;
    const uint32_t jc = (j >> 3) & 7;
    bool my_abort = false;
#pragma unroll 1
    for (int t = 0; t < nt; ++t) {
      const int64_t key = j0 + (int64_t)tile_at(t) * kKeys + j;
      uint64_t vis = 0;
      if (key < j1 && resolve_row(a, rq.q0, P, kv_base, key) >= 0) {  // rows outside the pool are excluded
        for (int tl = 0; tl < ntok; ++tl)
          if (mask_bit(a.mask, mask_base + (int64_t)tl * L + key)) vis |= ctl.colmask[tl][half];
      }
      float s[HC];
      if (!my_abort) my_abort = !mbar_wait(&ctl.s_full, t & 1, &ctl.abort, a.status);
      my_abort = __any_sync(0xffffffffu, my_abort);  // tcgen05.ld below is warp-collective
      tc::fence_after_sync();
      if (!my_abort) {
#pragma unroll
        for (int c = 0; c < HC / 8; ++c) tc::tmem_ld8(t_lane + Cfg::kColS + c0 + 8 * c, &s[8 * c]);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < HC; ++k) s[k] = 0.f;
      }
      tc::fence_before_sync();
      __syncwarp();
      // S^T may be overwritten now (resident mode: QK(t+1) follows PV(t), which
      // waits for P^T(t), so no separate signal is needed)
      if (!kLandOnce && lane == 0 && !my_abort) mbar_arrive(&ctl.s_free);

      bool need = false;
      const float4* mt4 = reinterpret_cast<const float4*>(&ctl.mtau[c0]);
#pragma unroll
      for (int k4 = 0; k4 < HC / 4; ++k4) {
        const float4 mt = mt4[k4];
        const float mtk[4] = {mt.x, mt.y, mt.z, mt.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int k = 4 * k4 + q;
          s[k] = ((vis >> k) & 1ull) ? s[k] * scale : -INFINITY;
          need |= s[k] > mtk[q];
        }
      }
      const bool warp_need = __any_sync(0xffffffffu, need);
      const bool warp_abort = __any_sync(0xffffffffu, my_abort) || ctl.abort;
      if (lane == 0) ctl.flag[t & 1][warp] = (warp_need ? 1 : 0) | (warp_abort ? 2 : 0);
      named_bar_sync(1, kSoftmaxThreads);
      int f = 0;
#pragma unroll
      for (int w = 0; w < kSoftmaxWarps; ++w) f |= ctl.flag[t & 1][w];
      if (tid == 0) ctl.rflag[(t + 1) & 1] = 0;
      if (f & 2) {
        my_abort = true;
        break;
      }
      bool rescale = false;
      if (f & 1) {
        // Exact column max over the tile's 128 keys; raise the running max
        // where it passed by more than kTau.
        warp_columns_to_smem<HC, true>(s, &ctl.red[quad][c0], lane);
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
        }
        named_bar_sync(1, kSoftmaxThreads);
#pragma unroll
        for (int k = 0; k < HC; ++k) acc_r[k] *= ctl.alpha[c0 + k];
        if (tid < 2 * NQ) l_half *= ctl.alpha[tid >> 1];
        rescale = (t > 0) && ctl.rflag[t & 1];
      }
      // P^T(t) overwrites what PV(t-1) reads, and a rescale of O^T needs
      // PV(t-1) complete as well (resident mode: S^T(t) completing implies it).
      if (!kLandOnce && t >= 1 && !my_abort)
        my_abort = !mbar_wait(&ctl.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, &ctl.abort, a.status);
      my_abort = __any_sync(0xffffffffu, my_abort);
      tc::fence_after_sync();
      if (!my_abort && rescale) {
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int c = 0; c < HC / 8; ++c) {
            float v[8];
            tc::tmem_ld8(t_lane + m * Cfg::kOStride + c0 + 8 * c, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] *= ctl.alpha[c0 + 8 * c + k];
            tc::tmem_st8(t_lane + m * Cfg::kOStride + c0 + 8 * c, v);
          }
        }
        tc::tmem_wait_st();
      }
      if (!my_abort) {
        const uint32_t pb_t = pbase;
        const float4* mu4 = reinterpret_cast<const float4*>(&ctl.muse[c0]);
#pragma unroll
        for (int k4 = 0; k4 < HC / 4; ++k4) {
          const float4 mu = mu4[k4];
          const float p0 = ex2_approx(s[4 * k4 + 0] - mu.x);  // s = -inf (masked) gives 0
          const float p1 = ex2_approx(s[4 * k4 + 1] - mu.y);
          const float p2 = ex2_approx(s[4 * k4 + 2] - mu.z);
          const float p3 = ex2_approx(s[4 * k4 + 3] - mu.w);
          const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1);
          const __nv_bfloat162 h23 = __floats2bfloat162_rn(p2, p3);
          const uint32_t w01 = *reinterpret_cast<const uint32_t*>(&h01);
          const uint32_t w23 = *reinterpret_cast<const uint32_t*>(&h23);
          acc_r[4 * k4 + 0] += p0 - __uint_as_float(w01 << 16);
          acc_r[4 * k4 + 1] += p1 - __uint_as_float(w01 & 0xFFFF0000u);
          acc_r[4 * k4 + 2] += p2 - __uint_as_float(w23 << 16);
          acc_r[4 * k4 + 3] += p3 - __uint_as_float(w23 & 0xFFFF0000u);
          const int k = 4 * k4;
          asm volatile(
              "st.shared.u16 [%0], %4;\n\tst.shared.u16 [%1], %5;\n\tst.shared.u16 [%2], %6;\n\tst.shared.u16 [%3], %7;" ::"r"(
                  pb_t + (k + 0) * 128 + ((jc ^ (uint32_t)((k + 0) & 7)) << 4)),
              "r"(pb_t + (k + 1) * 128 + ((jc ^ (uint32_t)((k + 1) & 7)) << 4)),
              "r"(pb_t + (k + 2) * 128 + ((jc ^ (uint32_t)((k + 2) & 7)) << 4)),
              "r"(pb_t + (k + 3) * 128 + ((jc ^ (uint32_t)((k + 3) & 7)) << 4)), "h"((uint16_t)(w01 & 0xFFFFu)),
              "h"((uint16_t)(w01 >> 16)), "h"((uint16_t)(w23 & 0xFFFFu)), "h"((uint16_t)(w23 >> 16))
              : "memory");
        }
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0 && !my_abort) mbar_arrive(&ctl.p_full);
      // bf16 column sums of this tile (the MMA reads P^T concurrently).  The
      // chunk order is staggered by column so the 8 threads of a bank group
      // read 8 different 16-byte chunks.
      named_bar_sync(1, kSoftmaxThreads);
      if (tid < 2 * NQ && !my_abort) {
        const int col = tid >> 1;
        const uint32_t row = sP + (tid & 1) * Cfg::kPRegion + col * 128;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t w0, w1, w2, w3;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                       : "r"(row + (((k + col) & 7) << 4)));
          a0 += (__uint_as_float(w0 << 16) + __uint_as_float(w1 << 16)) +
                (__uint_as_float(w2 << 16) + __uint_as_float(w3 << 16));
          a1 += (__uint_as_float(w0 & 0xFFFF0000u) + __uint_as_float(w1 & 0xFFFF0000u)) +
                (__uint_as_float(w2 & 0xFFFF0000u) + __uint_as_float(w3 & 0xFFFF0000u));
        }
        l_half += a0 + a1;
      }
      if constexpr (kLandOnce) {
        // slot 8 may take the next tile's RoPE block once PV and these reads are done
        if (tid < 2 * NQ && !my_abort) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.empty[8]);
        }
      }
    }

    // ---- epilogue: l, LSE, O = O^T / l ----------------------------------------
    // The sums need no MMA: reduce them while the last PV runs.
    if (tid < 2 * NQ) ctl.red[tid & 1][tid >> 1] = l_half;
    warp_columns_to_smem<HC, false>(acc_r, &ctl.red2[quad][c0], lane);
    if (!my_abort) {
      if constexpr (kLandOnce)
        my_abort = !mbar_wait(&ctl.pv_last, 0, &ctl.abort, a.status);
      else
        my_abort = !mbar_wait(&ctl.pv_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, &ctl.abort, a.status);
    }
    tc::fence_after_sync();
    const bool wa = __any_sync(0xffffffffu, my_abort) || ctl.abort;
    if (lane == 0) ctl.flag[nt & 1][warp] = wa ? 2 : 0;
    named_bar_sync(1, kSoftmaxThreads);
    int f = 0;
#pragma unroll
    for (int w = 0; w < kSoftmaxWarps; ++w) f |= ctl.flag[nt & 1][w];
    if (tid < NQ) {
      const float lp = ctl.red[0][tid] + ctl.red[1][tid];
      const float lr = (ctl.red2[0][tid] + ctl.red2[1][tid]) + (ctl.red2[2][tid] + ctl.red2[3][tid]);
      ctl.alpha[tid] = lp > 0.f ? 1.f / lp : 0.f;
      if (!(f & 2) && tid < nrows)
        lse_out[tid] = lp > 0.f ? (ctl.muse[tid] + __log2f(lp + lr)) * 0.69314718055994530942f : -INFINITY;
    }
    named_bar_sync(1, kSoftmaxThreads);
    if (!(f & 2)) {
      // O straight from TMEM to global memory: thread (quad, lane) holds
      // latent column 128m + j of query rows c0..c0+HC, so each warp store
      // writes 32 consecutive columns (128 bytes) of one row.  Rows with
      // nothing visible are not written (their LSE is -inf).
      float* ocol = a.part_o + ((int64_t)s_idx * a.rows_max + grow0) * kDLatent + j;
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        float v[HC];
#pragma unroll
        for (int c = 0; c < HC / 8; ++c) tc::tmem_ld8(t_lane + m * Cfg::kOStride + c0 + 8 * c, &v[8 * c]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < HC; ++k) {
          const int n = c0 + k;
          const float inv_l = ctl.alpha[n];
          if (n < nrows && inv_l > 0.f) ocol[(int64_t)n * kDLatent + 128 * m] = v[k] * inv_l;
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

  // ---- fused merge ------------------------------------------------------------
  // Every CTA of a (request, row group) takes a ticket once its partials are
  // visible device-wide; the one that takes the last ticket (of the
  // request's non-empty splits) merges the group's rows and resets the
  // counter for the next call.  Nobody waits on another CTA.
  if constexpr (kFused) {
    const int n_split = (int)((L + chunk - 1) / chunk);  // splits with keys: 0..n_split-1
    uint32_t* cnt = a.merge_count + (int64_t)b * gridDim.x + g;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const bool last = atomicAdd(cnt, 1u) + 1u == (uint32_t)n_split;
      if (last) *cnt = 0u;
      ctl.merge_last = last ? 1 : 0;
    }
    __syncthreads();
    if (ctl.merge_last) {
      __threadfence();
      // warp w merges half w%2 of row w/2, then of row (w + warps)/2, ...
      for (int w = warp; w < 2 * nrows; w += kTcThreads / 32)
        merge_row_half<true>(a.part_lse, a.part_o, a.rows_max, n_split, grow0 + (w >> 1), w & 1, lane, a.o, a.lse);
    }
  }
}

template <int NQ, int kMode>
cudaError_t launch_split_tc_nq(const SplitArgs& a, const TcMaps& maps, dim3 grid, cudaStream_t stream) {
  constexpr int smem = tc_smem_bytes<NQ, kMode>();
  static_assert(smem <= 232448, "shared memory budget exceeded");
  void (*kernel)(SplitArgs, TcMaps) =
      a.merge_count ? split_tc_kernel<NQ, true, kMode> : split_tc_kernel<NQ, false, kMode>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(TcCfg<NQ, kMode>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  e = cudaLaunchKernelEx(&cfg, kernel, a, maps);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mlav
