/*
 * Exact softmax attention, forward and backward, in plain fp64 C.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the oracle that the CUDA path is checked
 * against.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it; the library under exact_attention_98_gb300/ never does, and
 * the two share no code, header, table or constant.
 *
 * What is computed, and where it comes from:
 *   - Attention is two matrix products around a softmax, S = Q·K^T and
 *     O = P·V ("FlashAttention-4 : comment Together AI a accéléré l'attention
 *     sur GPU Blackwell", section "Pourquoi l'approche standard ne fonctionne
 *     plus"; the same two products in "FlashAttention-3 и FlashAttention-4",
 *     section "Режим 2-CTA MMA").
 *   - The tiled FlashAttention schedules leave the attention mechanism itself
 *     unchanged ("FlashAttention-3 и FlashAttention-4", section "Ключевая идея
 *     FlashAttention-3"); pipelining, the emulated exponential and conditional
 *     rescaling only change the cost (FlashAttention-4 abstract, items 1-2).
 *     So the oracle is the plain definition, not an emulation of any tiling:
 *       s_ij  = scale * sum_t q_it k_jt        for allowed j
 *       M_i   = max_j s_ij
 *       l_i   = sum_j exp(s_ij - M_i)
 *       P_ij  = exp(s_ij - M_i) / l_i
 *       O_i   = sum_j P_ij v_j
 *       LSE_i = M_i + ln l_i                   (natural log, scaled scores)
 *     "allowed" is every key, or key j <= query i when causal.
 *   - Backward: the pages give no formula for it.  With the loss
 *     L = sum(O * dO), the chain rule through P = softmax(S) and
 *     S = scale * Q K^T gives
 *       D_i   = sum_t dO_it O_it
 *       dP_ij = dO_i . v_j
 *       dS_ij = P_ij (dP_ij - D_i)
 *       dQ_i  = scale * sum_j dS_ij k_j
 *       dK_j  = scale * sum_i dS_ij q_i
 *       dV_j  = sum_i P_ij dO_i
 *
 * Every function works on ONE (batch, head) slice, row-major [N, d].  Rows are
 * independent, so the only parallelism is an OpenMP loop over rows; there is
 * no blocking, fusion or reordering of the arithmetic.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

static int key_allowed(int i, int j, int causal) { return !causal || j <= i; }

/* x rounded to the nearest bfloat16 value (8 significant bits, ties to even),
 * directly from fp64.  Used only to model the point where the library hands
 * O to the backward pass in bf16. */
double oracle_round_bf16(double x) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  const double m = frexp(x, &e); /* x = m * 2^e, 0.5 <= |m| < 1 */
  return ldexp(nearbyint(ldexp(m, 8)), e - 8);
}

/* Scores of one query row against all keys: s[j] = scale * q . k_j, and the
 * row max and LSE over the allowed keys.  Returns the number of allowed keys. */
static int row_scores(const double* q_row, int i, const double* k, int N, int d,
                      double scale, int causal, double* s, double* M_out,
                      double* lse_out) {
  int n_allowed = 0;
  double M = -INFINITY;
  for (int j = 0; j < N; ++j) {
    if (!key_allowed(i, j, causal)) continue;
    double acc = 0.0;
    for (int t = 0; t < d; ++t) acc += q_row[t] * k[(size_t)j * d + t];
    s[j] = scale * acc;
    if (s[j] > M) M = s[j];
    ++n_allowed;
  }
  double l = 0.0;
  for (int j = 0; j < N; ++j)
    if (key_allowed(i, j, causal)) l += exp(s[j] - M);
  *M_out = M;
  *lse_out = M + log(l);
  return n_allowed;
}

/* Softmax probabilities of one row, P_ij = exp(s_ij - LSE_i); masked keys get
 * exactly 0.  exp(s - M)/l and exp(s - (M + ln l)) are the same number. */
static void row_probs(const double* s, int i, int N, int causal, double lse,
                      double* p) {
  for (int j = 0; j < N; ++j)
    p[j] = key_allowed(i, j, causal) ? exp(s[j] - lse) : 0.0;
}

/*
 * Forward for selected query rows of one head.
 *   q    : [nq, d]   the selected query rows
 *   qidx : [nq]      their positions in the sequence (for the causal mask);
 *                    NULL means row r is position r
 *   k, v : [N, d]
 *   o    : [nq, d]   out
 *   lse  : [nq]      out, natural log of sum_j exp(s_ij)
 */
int oracle_fwd_rows(const double* q, int nq, const int* qidx, const double* k,
                    const double* v, int N, int d, double scale, int causal,
                    double* o, double* lse) {
  if (nq < 0 || N < 1 || d < 1 || !q || !k || !v || !o || !lse)
    return ORACLE_BAD_ARG;
  int bad = 0, nomem = 0;
#pragma omp parallel for schedule(dynamic, 4)
  for (int r = 0; r < nq; ++r) {
    int i = qidx ? qidx[r] : r;
    if (i < 0 || i >= N) { bad = 1; continue; }
    double* s = (double*)malloc(sizeof(double) * (size_t)N * 2);
    if (!s) { nomem = 1; continue; }
    double* p = s + N;
    double M, L;
    row_scores(q + (size_t)r * d, i, k, N, d, scale, causal, s, &M, &L);
    row_probs(s, i, N, causal, L, p);
    for (int t = 0; t < d; ++t) {
      double acc = 0.0;
      for (int j = 0; j < N; ++j) acc += p[j] * v[(size_t)j * d + t];
      o[(size_t)r * d + t] = acc;
    }
    lse[r] = L;
    free(s);
  }
  if (bad) return ORACLE_BAD_ARG;
  return nomem ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Backward for one head, for selected rows of dQ and selected rows of dK/dV.
 *   q, k, v, dout : [N, d]
 *   qrows [nqr]   : rows i of dQ to produce  -> dq [nqr, d]
 *   krows [nkr]   : rows j of dK, dV         -> dk, dv [nkr, d]
 * dK_j and dV_j sum over every query row, so when nkr > 0 the softmax
 * statistics (LSE_i and D_i) of every row are computed first.  All of it uses
 * the oracle's own fp64 forward: O_i and LSE_i are not taken from outside.
 * Passing every row in qrows and krows gives the full backward of the head.
 *
 * o_bf16: 0 = D_i = dO_i . O_i with the exact fp64 O (the plain definition);
 *         1 = D_i = dO_i . bf16(O_i): the backward's O input as the library's
 *             API carries it between the passes (bf16), each element of the
 *             oracle's own fp64 O rounded to nearest-even bf16.  Everything
 *             else is identical.
 */
int oracle_bwd_rows(const double* q, const double* k, const double* v,
                    const double* dout, int N, int d, double scale, int causal,
                    const int* qrows, int nqr, double* dq, const int* krows,
                    int nkr, double* dk, double* dv, int o_bf16) {
  if (N < 1 || d < 1 || nqr < 0 || nkr < 0 || !q || !k || !v || !dout)
    return ORACLE_BAD_ARG;
  if ((nqr > 0 && (!qrows || !dq)) || (nkr > 0 && (!krows || !dk || !dv)))
    return ORACLE_BAD_ARG;
  for (int r = 0; r < nqr; ++r)
    if (qrows[r] < 0 || qrows[r] >= N) return ORACLE_BAD_ARG;
  for (int r = 0; r < nkr; ++r)
    if (krows[r] < 0 || krows[r] >= N) return ORACLE_BAD_ARG;

  /* Per-row statistics LSE_i and D_i, for the rows that are needed. */
  double* lse = (double*)malloc(sizeof(double) * (size_t)N);
  double* D = (double*)malloc(sizeof(double) * (size_t)N);
  char* need = (char*)calloc((size_t)N, 1);
  if (!lse || !D || !need) { free(lse); free(D); free(need); return ORACLE_NO_MEMORY; }
  if (nkr > 0) memset(need, 1, (size_t)N);
  for (int r = 0; r < nqr; ++r) need[qrows[r]] = 1;

  int nomem = 0;
#pragma omp parallel for schedule(dynamic, 4)
  for (int i = 0; i < N; ++i) {
    if (!need[i]) continue;
    double* s = (double*)malloc(sizeof(double) * (size_t)N * 2);
    if (!s) { nomem = 1; continue; }
    double* p = s + N;
    double M, L;
    row_scores(q + (size_t)i * d, i, k, N, d, scale, causal, s, &M, &L);
    row_probs(s, i, N, causal, L, p);
    double Di = 0.0;
    for (int t = 0; t < d; ++t) {
      double o_it = 0.0;
      for (int j = 0; j < N; ++j) o_it += p[j] * v[(size_t)j * d + t];
      if (o_bf16) o_it = oracle_round_bf16(o_it);
      Di += dout[(size_t)i * d + t] * o_it;
    }
    lse[i] = L;
    D[i] = Di;
    free(s);
  }
  if (nomem) { free(lse); free(D); free(need); return ORACLE_NO_MEMORY; }

  /* dQ_i = scale * sum_j P_ij (dP_ij - D_i) k_j */
#pragma omp parallel for schedule(dynamic, 4)
  for (int r = 0; r < nqr; ++r) {
    int i = qrows[r];
    double* s = (double*)malloc(sizeof(double) * (size_t)N * 2);
    if (!s) { nomem = 1; continue; }
    double* p = s + N;
    double M, L;
    row_scores(q + (size_t)i * d, i, k, N, d, scale, causal, s, &M, &L);
    row_probs(s, i, N, causal, lse[i], p);
    double* dq_row = dq + (size_t)r * d;
    for (int t = 0; t < d; ++t) dq_row[t] = 0.0;
    for (int j = 0; j < N; ++j) {
      if (!key_allowed(i, j, causal)) continue;
      double dP = 0.0;
      for (int t = 0; t < d; ++t) dP += dout[(size_t)i * d + t] * v[(size_t)j * d + t];
      double dS = p[j] * (dP - D[i]);
      for (int t = 0; t < d; ++t) dq_row[t] += dS * k[(size_t)j * d + t];
    }
    for (int t = 0; t < d; ++t) dq_row[t] *= scale;
    free(s);
  }

  /* dK_j = scale * sum_i dS_ij q_i ;  dV_j = sum_i P_ij dO_i */
#pragma omp parallel for schedule(dynamic, 4)
  for (int r = 0; r < nkr; ++r) {
    int j = krows[r];
    double* dk_row = dk + (size_t)r * d;
    double* dv_row = dv + (size_t)r * d;
    for (int t = 0; t < d; ++t) { dk_row[t] = 0.0; dv_row[t] = 0.0; }
    for (int i = 0; i < N; ++i) {
      if (!key_allowed(i, j, causal)) continue;
      double sij = 0.0, dP = 0.0;
      for (int t = 0; t < d; ++t) {
        sij += q[(size_t)i * d + t] * k[(size_t)j * d + t];
        dP += dout[(size_t)i * d + t] * v[(size_t)j * d + t];
      }
      double P = exp(scale * sij - lse[i]);
      double dS = P * (dP - D[i]);
      for (int t = 0; t < d; ++t) {
        dk_row[t] += dS * q[(size_t)i * d + t];
        dv_row[t] += P * dout[(size_t)i * d + t];
      }
    }
    for (int t = 0; t < d; ++t) dk_row[t] *= scale;
  }

  free(lse);
  free(D);
  free(need);
  return nomem ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Number of OpenMP threads the oracle runs with (for the baseline record). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
