/*
 * CPU fp64 oracle for IKBO target attention.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the bench's CPU-baseline leg
 * may load this library.  It shares no code with the CUDA path: it reads the
 * same bf16 input bits and computes, in double precision, what the method is
 * defined to compute.
 *
 * Definition followed ("In-Kernel Broadcast Optimization: Co-Designing
 * Kernels for RecSys Inference", §3 and §3.1 with Fig. 10): conventional
 * target attention first broadcasts each user's K/V sequence to every one of
 * that user's candidates and then runs scaled-dot-product attention per
 * candidate; IKBO indexes the user's K/V through the candidate-to-user map
 * and is mathematically equivalent.  The model is encoder driven, so the
 * attention is full (no causal mask).  This oracle takes the broadcast form
 * literally: for every (candidate, head) it copies the user's K and V rows
 * into private scratch (the materialised broadcast) and then evaluates
 *
 *     s_j   = scale * sum_d q[c,h,t,d] * K_c[j,d]          j = 0 .. L_u - 1
 *     p_j   = exp(s_j - max_j s_j) / sum_j exp(s_j - max_j s_j)
 *     out[c,h,t,:] = sum_j p_j * V_c[j,:]
 *
 * with u = cand_to_user[c] and K_c = K[user_offsets[u] : user_offsets[u+1], h, :].
 * Subtracting the row maximum does not change the softmax; it only keeps
 * exp() finite.  A user with an empty sequence (L_u = 0) yields an all-zero
 * row: the pages are silent on that case, and zero is the limit of a sum
 * over no keys.
 *
 * Layouts (bf16 given as raw uint16 bits, widened exactly):
 *   q   [n_cand, H, Lq, D]      k, v [T, H, D] (users packed back to back)
 *   out [n_sel, H, Lq, D] fp64, row i belongs to candidate cands[i]
 *       (or to candidate i when cands is NULL and n_sel == n_cand).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_INDEX -2
#define ORACLE_ERR_OFFSETS -3
#define ORACLE_ERR_NOMEM -4

static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static int check_structure(const int32_t* offsets, const int32_t* c2u, int64_t n_cand,
                           int64_t n_user) {
  if (offsets[0] != 0) return ORACLE_ERR_OFFSETS;
  for (int64_t u = 0; u < n_user; ++u)
    if (offsets[u + 1] < offsets[u]) return ORACLE_ERR_OFFSETS;
  for (int64_t c = 0; c < n_cand; ++c)
    if (c2u[c] < 0 || (int64_t)c2u[c] >= n_user) return ORACLE_ERR_INDEX;
  return ORACLE_OK;
}

/* Attention of one query row over an already materialised K/V copy. */
static void attend_row(const double* qrow, const double* Kc, const double* Vc, int64_t L, int D,
                       double scale, double* s, double* orow) {
  for (int d = 0; d < D; ++d) orow[d] = 0.0;
  if (L == 0) return;
  double m = -INFINITY;
  for (int64_t j = 0; j < L; ++j) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qrow[d] * Kc[j * D + d];
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < L; ++j) {
    s[j] = exp(s[j] - m);
    l += s[j];
  }
  for (int64_t j = 0; j < L; ++j) {
    double w = s[j] / l;
    for (int d = 0; d < D; ++d) orow[d] += w * Vc[j * D + d];
  }
}

/*
 * out[i, h, t, :] for every selected candidate i (all candidates when
 * cands == NULL).  Returns 0, or a negative ORACLE_ERR_* code.
 */
int ikbo_oracle_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const int32_t* user_offsets, const int32_t* cand_to_user, int64_t n_cand,
                    int64_t n_user, int32_t H, int32_t Lq, int32_t D, double scale,
                    const int64_t* cands, int64_t n_sel, double* out) {
  if (!q || !k || !v || !user_offsets || !cand_to_user || !out) return ORACLE_ERR_ARG;
  if (n_cand < 0 || n_user < 0 || H < 1 || Lq < 1 || D < 1 || n_sel < 0) return ORACLE_ERR_ARG;
  if (!cands && n_sel != n_cand) return ORACLE_ERR_ARG;
  int rc = check_structure(user_offsets, cand_to_user, n_cand, n_user);
  if (rc) return rc;
  if (cands)
    for (int64_t i = 0; i < n_sel; ++i)
      if (cands[i] < 0 || cands[i] >= n_cand) return ORACLE_ERR_ARG;

  int64_t Lmax = 0;
  for (int64_t u = 0; u < n_user; ++u) {
    int64_t L = (int64_t)user_offsets[u + 1] - user_offsets[u];
    if (L > Lmax) Lmax = L;
  }
  int failed = 0;
  const int64_t n_pairs = n_sel * (int64_t)H;

#pragma omp parallel
  {
    /* Per-thread scratch: the materialised copy of one user's K/V for one head. */
    double* Kc = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1) * D);
    double* Vc = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1) * D);
    double* s = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
    double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
    if (!Kc || !Vc || !s || !qrow) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t pair = 0; pair < n_pairs; ++pair) {
        int64_t i = pair / H;
        int h = (int)(pair % H);
        int64_t c = cands ? cands[i] : i;
        int64_t u = cand_to_user[c];
        int64_t base = user_offsets[u];
        int64_t L = (int64_t)user_offsets[u + 1] - base;
        /* broadcast: this candidate's own copy of its user's K and V rows */
        for (int64_t j = 0; j < L; ++j)
          for (int d = 0; d < D; ++d) {
            int64_t src = ((base + j) * H + h) * (int64_t)D + d;
            Kc[j * D + d] = bf16_to_double(k[src]);
            Vc[j * D + d] = bf16_to_double(v[src]);
          }
        for (int t = 0; t < Lq; ++t) {
          int64_t qoff = ((c * H + h) * (int64_t)Lq + t) * D;
          for (int d = 0; d < D; ++d) qrow[d] = bf16_to_double(q[qoff + d]);
          double* orow = out + ((i * H + h) * (int64_t)Lq + t) * D;
          attend_row(qrow, Kc, Vc, L, D, scale, s, orow);
        }
      }
    }
    free(Kc);
    free(Vc);
    free(s);
    free(qrow);
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * The attention weights p_j of one query row (candidate c, head h, token t):
 * probs[0 .. L_u-1].  Same definition as above, exposed so that tests can
 * check the weights themselves (non-negative, summing to one).
 */
int ikbo_oracle_weights(const uint16_t* q, const uint16_t* k, const int32_t* user_offsets,
                        const int32_t* cand_to_user, int64_t n_cand, int64_t n_user, int32_t H,
                        int32_t Lq, int32_t D, double scale, int64_t c, int32_t h, int32_t t,
                        double* probs) {
  if (!q || !k || !user_offsets || !cand_to_user || !probs) return ORACLE_ERR_ARG;
  if (c < 0 || c >= n_cand || h < 0 || h >= H || t < 0 || t >= Lq) return ORACLE_ERR_ARG;
  int rc = check_structure(user_offsets, cand_to_user, n_cand, n_user);
  if (rc) return rc;
  int64_t u = cand_to_user[c];
  int64_t base = user_offsets[u];
  int64_t L = (int64_t)user_offsets[u + 1] - base;
  if (L == 0) return ORACLE_OK;
  double m = -INFINITY;
  int64_t qoff = ((c * H + h) * (int64_t)Lq + t) * D;
  for (int64_t j = 0; j < L; ++j) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d)
      acc += bf16_to_double(q[qoff + d]) * bf16_to_double(k[((base + j) * H + h) * (int64_t)D + d]);
    probs[j] = scale * acc;
    if (probs[j] > m) m = probs[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < L; ++j) {
    probs[j] = exp(probs[j] - m);
    l += probs[j];
  }
  for (int64_t j = 0; j < L; ++j) probs[j] /= l;
  return ORACLE_OK;
}

/*
 * Self-attention over the user sequence ("In-Kernel Broadcast Optimization",
 * §3.3 and §1: the user's history attends to itself, with the same keys and
 * values as the target attention and queries taken from the user side; full
 * attention, no causal mask, as the model is encoder driven).  For every
 * selected sequence row r of user u (off[u] <= r < off[u+1]) and head h:
 *
 *     out[r,h,:] = sum_j softmax_j(scale * q_user[r,h,:] . K[off[u]+j,h,:]) V[off[u]+j,h,:]
 *
 * over j = 0 .. L_u - 1.  Layouts: q_user, k, v [T, H, D] bf16 bits with
 * T = user_offsets[n_user]; out [n_sel, H, D] fp64, row i for sequence row
 * rows[i] (all rows when rows is NULL and n_sel == T).
 */
int ikbo_oracle_self_fwd(const uint16_t* q_user, const uint16_t* k, const uint16_t* v,
                         const int32_t* user_offsets, int64_t n_user, int32_t H, int32_t D,
                         double scale, const int64_t* rows, int64_t n_sel, double* out) {
  if (!q_user || !k || !v || !user_offsets || !out) return ORACLE_ERR_ARG;
  if (n_user < 0 || H < 1 || D < 1 || n_sel < 0) return ORACLE_ERR_ARG;
  int rc = check_structure(user_offsets, NULL, 0, n_user);
  if (rc) return rc;
  const int64_t T = user_offsets[n_user];
  if (!rows && n_sel != T) return ORACLE_ERR_ARG;
  if (rows)
    for (int64_t i = 0; i < n_sel; ++i)
      if (rows[i] < 0 || rows[i] >= T) return ORACLE_ERR_ARG;
  int64_t Lmax = 0;
  for (int64_t u = 0; u < n_user; ++u) {
    int64_t L = (int64_t)user_offsets[u + 1] - user_offsets[u];
    if (L > Lmax) Lmax = L;
  }
  int failed = 0;
  const int64_t n_pairs = n_sel * (int64_t)H;

#pragma omp parallel
  {
    double* Ku = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1) * D);
    double* Vu = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1) * D);
    double* s = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
    double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
    if (!Ku || !Vu || !s || !qrow) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t pair = 0; pair < n_pairs; ++pair) {
        int64_t i = pair / H;
        int h = (int)(pair % H);
        int64_t r = rows ? rows[i] : i;
        /* the user whose sequence holds row r (the last u with off[u] <= r) */
        int64_t u = 0;
        while (u + 1 < n_user && user_offsets[u + 1] <= r) ++u;
        int64_t base = user_offsets[u];
        int64_t L = (int64_t)user_offsets[u + 1] - base;
        for (int64_t j = 0; j < L; ++j)
          for (int d = 0; d < D; ++d) {
            int64_t src = ((base + j) * H + h) * (int64_t)D + d;
            Ku[j * D + d] = bf16_to_double(k[src]);
            Vu[j * D + d] = bf16_to_double(v[src]);
          }
        for (int d = 0; d < D; ++d) qrow[d] = bf16_to_double(q_user[(r * H + h) * (int64_t)D + d]);
        attend_row(qrow, Ku, Vu, L, D, scale, s, out + (i * H + h) * (int64_t)D);
      }
    }
    free(Ku);
    free(Vu);
    free(s);
    free(qrow);
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

int ikbo_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
