/*
 * CPU oracle for MLA tree-verify attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline leg may load this library.  The product path (the CUDA library
 * and its Python binding) never calls it and shares no code with it.
 *
 * What it computes (plain definition, fp64, no blocking or fusion):
 * for every request b, draft token i < T_b and head h, over the
 * L_b = P_b + T_b keys of that request, where request b's tokens are the
 * token rows q0_b .. q0_b + T_b - 1 (q0_b = qo_indptr[b] and
 * T_b = qo_indptr[b+1] - qo_indptr[b]; without qo_indptr every request has
 * T tokens and q0_b = b*T),
 *
 *   visible(j)  = bit (mask_indptr[b] + i*L_b + j) of custom_mask (LSB-first)
 *                 [Custom sm_120 Verify Kernel, §"The Debugging Gauntlet":
 *                  mask row stride is prefix + q_len; mask_indptr has B entries]
 *   row(j)      = kv_indices[kv_indptr[b] + j]        if j <  P_b
 *               = out_cache_loc[q0_b + (j - P_b)]     if j >= P_b
 *                 [Capture Safety to MoE Ceiling, §"The Architecture of Capture
 *                  Safety": two-array row selection]
 *   s_j         = sm_scale * ( sum_{d<512} q_nope[d]*kv[row(j), d]
 *                            + sum_{d<64}  q_rope[d]*kv[row(j), 512+d] )
 *   m           = max_{visible j} s_j,   Z = sum_{visible j} exp(s_j - m)
 *   O[d]        = sum_{visible j} exp(s_j - m) * kv[row(j), d] / Z,  d < 512
 *   LSE         = m + ln Z        (O = 0, LSE = -inf when nothing is visible)
 *
 * The absorbed-query form (scores against the 576-wide latent+RoPE row,
 * values = the 512 latent entries of the same row) is the MLA verify step the
 * pages accelerate [Custom sm_120 Verify Kernel, §"The Bottleneck: Triton's
 * Scattered KV Access at 14 GB/s"].  bf16 inputs are widened exactly.
 *
 * oracle_mla_verify_split_merge() evaluates the same quantity the way the
 * pages' kernel is organised -- per-split partial softmax statistics, then a
 * second reduction that merges the partials by log-sum-exp [Custom sm_120
 * Verify Kernel, §"Building the Custom Kernel: From Occupancy Starvation to
 * Flash-Decode"] -- so that the split/merge identity itself is pinned.
 *
 * `mutation` != 0 plants one deliberate mistake (tests use it to show that
 * the pins catch such mistakes); 0 is the oracle proper.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define D_LATENT 512
#define D_ROPE 64
#define D_ROW 576

enum {
  MUT_NONE = 0,
  MUT_MASK_STRIDE_PREFIX = 1, /* mask row stride P_b instead of P_b + T   */
  MUT_PREFIX_ONLY = 2,        /* draft rows dropped: only P_b keys         */
  MUT_MASK_INDPTR_NEXT = 3,   /* request b reads request b+1's mask offset */
  MUT_NO_ROPE = 4,            /* RoPE term left out of the score           */
  MUT_MSB_FIRST = 5,          /* mask bits read MSB-first                  */
  MUT_LSE_NO_MAX = 6,         /* LSE = ln Z, max not added back            */
  MUT_NO_SCALE = 7,           /* sm_scale not applied                      */
  MUT_V_SHIFT = 8,            /* values taken from columns 64..575         */
  MUT_DRAFT_REVERSED = 9,     /* draft rows read in reverse order          */
  MUT_SOFTMAX_SIGN = 10,      /* exp(m - s) instead of exp(s - m)          */
  /* per-request draft counts (qo_indptr given) */
  MUT_QO_DRAFT_UNIFORM = 11,  /* draft rows at out_cache_loc[b*T + t]      */
  MUT_QO_QROW_UNIFORM = 12,   /* query row b*T + i instead of qo_indptr[b]+i */
  MUT_QO_MASK_STRIDE_T = 13   /* mask row stride P_b + T (the maximum)     */
};

static double bf16_to_f64(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static int mask_bit(const uint8_t* mask, int64_t bit, int mutation) {
  uint8_t byte = mask[bit >> 3];
  int k = (int)(bit & 7);
  if (mutation == MUT_MSB_FIRST) k = 7 - k;
  return (byte >> k) & 1;
}

typedef struct {
  int B, H, T;
  const int32_t* qo_indptr; /* NULL: request b has T tokens starting at token row b*T */
  const uint16_t* q_nope;
  const uint16_t* q_rope;
  const uint16_t* kv_pool;
  int64_t pool_rows;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* out_cache_loc;
  const uint8_t* custom_mask;
  const int32_t* mask_indptr;
  double sm_scale;
  int mutation;
} problem_t;

static int64_t q_start(const problem_t* p, int b) {
  return p->qo_indptr ? (int64_t)p->qo_indptr[b] : (int64_t)b * p->T;
}

static int64_t q_count(const problem_t* p, int b) {
  return p->qo_indptr ? (int64_t)p->qo_indptr[b + 1] - p->qo_indptr[b] : (int64_t)p->T;
}

/* Request and token of token row `tok` (a row some request owns). */
static void token_owner(const problem_t* p, int64_t tok, int* b, int* i) {
  if (!p->qo_indptr) {
    *b = (int)(tok / p->T);
    *i = (int)(tok % p->T);
    return;
  }
  int r = 0;
  while (r + 1 < p->B && q_start(p, r + 1) <= tok) ++r;  /* requests with no tokens are passed */
  *b = r;
  *i = (int)(tok - q_start(p, r));
}

static int64_t n_token_rows(const problem_t* p) {
  return p->qo_indptr ? (int64_t)p->qo_indptr[p->B] : (int64_t)p->B * p->T;
}

/* Row of the pool that key position j of request b refers to; -1 if invalid. */
static int64_t key_row(const problem_t* p, int b, int64_t P, int64_t j) {
  int64_t r;
  if (j < P) {
    r = p->kv_indices[p->kv_indptr[b] + j];
  } else {
    int64_t t = j - P;
    if (p->mutation == MUT_DRAFT_REVERSED) t = q_count(p, b) - 1 - t;
    const int64_t base = (p->mutation == MUT_QO_DRAFT_UNIFORM) ? (int64_t)b * p->T : q_start(p, b);
    r = p->out_cache_loc[base + t];
  }
  if (r < 0 || r >= p->pool_rows) return -1;
  return r;
}

static int key_visible(const problem_t* p, int b, int i, int64_t P, int64_t j) {
  int64_t L = P + q_count(p, b);
  int64_t stride = (p->mutation == MUT_MASK_STRIDE_PREFIX) ? P : (p->mutation == MUT_QO_MASK_STRIDE_T) ? P + p->T : L;
  int bb = b;
  if (p->mutation == MUT_MASK_INDPTR_NEXT) bb = (b + 1 < p->B) ? b + 1 : b;
  int64_t bit = (int64_t)p->mask_indptr[bb] + (int64_t)i * stride + j;
  return mask_bit(p->custom_mask, bit, p->mutation);
}

static double score(const problem_t* p, int64_t qrow, int h, int64_t row) {
  const uint16_t* qn = p->q_nope + (qrow * p->H + h) * D_LATENT;
  const uint16_t* qr = p->q_rope + (qrow * p->H + h) * D_ROPE;
  const uint16_t* kv = p->kv_pool + row * D_ROW;
  double acc = 0.0;
  for (int d = 0; d < D_LATENT; ++d) acc += bf16_to_f64(qn[d]) * bf16_to_f64(kv[d]);
  if (p->mutation != MUT_NO_ROPE)
    for (int d = 0; d < D_ROPE; ++d) acc += bf16_to_f64(qr[d]) * bf16_to_f64(kv[D_LATENT + d]);
  if (p->mutation != MUT_NO_SCALE) acc *= p->sm_scale;
  return acc;
}

static const uint16_t* value_row(const problem_t* p, int64_t row) {
  int off = (p->mutation == MUT_V_SHIFT) ? D_ROPE : 0;
  return p->kv_pool + row * D_ROW + off;
}

/*
 * Softmax attention of one output row over the key range [j0, j1) of its
 * request.  Writes the normalised O (512) and the natural-log LSE.  Returns 0,
 * or -1 when a referenced pool row is out of range.
 */
static int attend_range(const problem_t* p, int b, int i, int h, int64_t j0, int64_t j1,
                        double* s_buf, double* o, double* lse) {
  int64_t P = p->kv_indptr[b + 1] - p->kv_indptr[b];
  int64_t L = (p->mutation == MUT_PREFIX_ONLY) ? P : P + q_count(p, b);
  if (j1 > L) j1 = L;
  int64_t qrow = (p->mutation == MUT_QO_QROW_UNIFORM) ? (int64_t)b * p->T + i : q_start(p, b) + i;
  double m = -INFINITY;
  for (int64_t j = j0; j < j1; ++j) {
    s_buf[j - j0] = -INFINITY;
    if (!key_visible(p, b, i, P, j)) continue;
    int64_t r = key_row(p, b, P, j);
    if (r < 0) return -1;
    double s = score(p, qrow, h, r);
    s_buf[j - j0] = s;
    if (s > m) m = s;
  }
  for (int d = 0; d < D_LATENT; ++d) o[d] = 0.0;
  if (m == -INFINITY) {
    *lse = -INFINITY;
    return 0;
  }
  double Z = 0.0;
  for (int64_t j = j0; j < j1; ++j) {
    double s = s_buf[j - j0];
    if (s == -INFINITY) continue;
    double w = (p->mutation == MUT_SOFTMAX_SIGN) ? exp(m - s) : exp(s - m);
    Z += w;
    const uint16_t* v = value_row(p, key_row(p, b, P, j));
    for (int d = 0; d < D_LATENT; ++d) o[d] += w * bf16_to_f64(v[d]);
  }
  for (int d = 0; d < D_LATENT; ++d) o[d] /= Z;
  *lse = (p->mutation == MUT_LSE_NO_MAX) ? log(Z) : m + log(Z);
  return 0;
}

static int64_t max_len(const problem_t* p) {
  int64_t mx = 0;
  for (int b = 0; b < p->B; ++b) {
    int64_t L = (int64_t)(p->kv_indptr[b + 1] - p->kv_indptr[b]) + q_count(p, b);
    if (L > mx) mx = L;
  }
  return mx;
}

/*
 * Direct evaluation.  rows_sel lists global output rows r = (q0_b + i)*H + h
 * (NULL = all token rows x H in order).  o_out is [n_sel, 512], lse_out
 * [n_sel].  qo_indptr may be NULL (uniform T).  Returns 0, or -1 if some
 * referenced pool row is out of range.
 */
int oracle_mla_verify(int B, int H, int T, const int32_t* qo_indptr, const uint16_t* q_nope, const uint16_t* q_rope,
                      const uint16_t* kv_pool, int64_t pool_rows, const int32_t* kv_indptr,
                      const int32_t* kv_indices, const int32_t* out_cache_loc,
                      const uint8_t* custom_mask, const int32_t* mask_indptr, double sm_scale,
                      const int64_t* rows_sel, int64_t n_sel, double* o_out, double* lse_out,
                      int nthreads, int mutation) {
  problem_t p = {B, H, T, qo_indptr, q_nope, q_rope, kv_pool, pool_rows, kv_indptr, kv_indices,
                 out_cache_loc, custom_mask, mask_indptr, sm_scale, mutation};
  int64_t n = rows_sel ? n_sel : n_token_rows(&p) * H;
  int64_t Lmax = max_len(&p);
  int err = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double* s_buf = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t k = 0; k < n; ++k) {
      int64_t r = rows_sel ? rows_sel[k] : k;
      int h = (int)(r % H);
      int b, i;
      token_owner(&p, r / H, &b, &i);
      int64_t L = (int64_t)(kv_indptr[b + 1] - kv_indptr[b]) + q_count(&p, b);
      if (attend_range(&p, b, i, h, 0, L, s_buf, o_out + k * D_LATENT, lse_out + k) != 0) {
#pragma omp atomic write
        err = -1;
      }
    }
    free(s_buf);
  }
  return err;
}

/*
 * Split-then-merge evaluation.  Request b's key range is cut into nsplit
 * chunks of `chunk` keys (chunk = max(min_chunk, round_up(ceil(L_b/nsplit),
 * granule))); split s covers [s*chunk, min(L_b, (s+1)*chunk)).  Each split
 * yields a normalised partial (O_s, lse_s) over its keys, and the partials
 * are merged by log-sum-exp: M = max_s lse_s, w_s = exp(lse_s - M),
 * O = sum_s w_s O_s / sum_s w_s, LSE = M + ln sum_s w_s.  Empty or fully
 * masked splits carry lse_s = -inf and weight 0.
 */
int oracle_mla_verify_split_merge(int B, int H, int T, const int32_t* qo_indptr, const uint16_t* q_nope,
                                  const uint16_t* q_rope, const uint16_t* kv_pool,
                                  int64_t pool_rows, const int32_t* kv_indptr,
                                  const int32_t* kv_indices, const int32_t* out_cache_loc,
                                  const uint8_t* custom_mask, const int32_t* mask_indptr,
                                  double sm_scale, int nsplit, int64_t granule, int64_t min_chunk,
                                  const int64_t* rows_sel, int64_t n_sel, double* o_out,
                                  double* lse_out, int nthreads) {
  problem_t p = {B, H, T, qo_indptr, q_nope, q_rope, kv_pool, pool_rows, kv_indptr, kv_indices,
                 out_cache_loc, custom_mask, mask_indptr, sm_scale, MUT_NONE};
  int64_t n = rows_sel ? n_sel : n_token_rows(&p) * H;
  int64_t Lmax = max_len(&p);
  int err = 0;
  if (nsplit < 1 || granule < 1) return -2;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double* s_buf = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
    double* o_s = (double*)malloc(sizeof(double) * (size_t)nsplit * D_LATENT);
    double* lse_s = (double*)malloc(sizeof(double) * (size_t)nsplit);
#pragma omp for schedule(dynamic, 1)
    for (int64_t k = 0; k < n; ++k) {
      int64_t r = rows_sel ? rows_sel[k] : k;
      int h = (int)(r % H);
      int b, i;
      token_owner(&p, r / H, &b, &i);
      int64_t L = (int64_t)(kv_indptr[b + 1] - kv_indptr[b]) + q_count(&p, b);
      int64_t per = (L + nsplit - 1) / nsplit;
      int64_t chunk = ((per + granule - 1) / granule) * granule;
      if (chunk < min_chunk) chunk = min_chunk;
      double M = -INFINITY;
      for (int s = 0; s < nsplit; ++s) {
        int64_t j0 = (int64_t)s * chunk, j1 = j0 + chunk;
        if (j1 > L) j1 = L;
        if (j0 >= j1) {
          lse_s[s] = -INFINITY;
          continue;
        }
        if (attend_range(&p, b, i, h, j0, j1, s_buf, o_s + (size_t)s * D_LATENT, lse_s + s) != 0) {
#pragma omp atomic write
          err = -1;
        }
        if (lse_s[s] > M) M = lse_s[s];
      }
      double* o = o_out + k * D_LATENT;
      for (int d = 0; d < D_LATENT; ++d) o[d] = 0.0;
      if (M == -INFINITY) {
        lse_out[k] = -INFINITY;
        continue;
      }
      double W = 0.0;
      for (int s = 0; s < nsplit; ++s) {
        if (lse_s[s] == -INFINITY) continue;
        double w = exp(lse_s[s] - M);
        W += w;
        for (int d = 0; d < D_LATENT; ++d) o[d] += w * o_s[(size_t)s * D_LATENT + d];
      }
      for (int d = 0; d < D_LATENT; ++d) o[d] /= W;
      lse_out[k] = M + log(W);
    }
    free(s_buf);
    free(o_s);
    free(lse_s);
  }
  return err;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
