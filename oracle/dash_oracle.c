/*
 * dash_oracle.c -- plain, slow, fp64 CPU oracle for softmax attention forward and
 * backward.  TEST INFRASTRUCTURE ONLY: it is called by the tests, by the smoke check
 * and by the bench's CPU-baseline leg, never by the product path.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes.  The DASH pages ("DASH: Deterministic Attention Scheduling for
 * High-throughput Reproducible LLM Training", gist.science technical summary, section 1
 * "Problem statement") describe the backward pass of FlashAttention-style attention
 * whose gradients -- dQ in particular -- must be accumulated in a fixed order.  The
 * pages never write the attention arithmetic itself, so this file is the textbook
 * definition of softmax attention and of its gradient, evaluated in double precision
 * from the exact values of the (bf16) inputs.  The tile schedules of the pages only
 * reorder fp32 additions inside the GPU path; they do not change the mathematical
 * result, so the oracle has no notion of tiles or schedules.
 *
 * Definitions (per batch b, query head h, kv head g = floor(h / G), G = H / Hkv):
 *   allowed(i,j) = full mask ? 1 : (j <= i)                          (causal = top-left)
 *   s_ij   = scale * sum_d Q[b,i,h,d] K[b,j,g,d]
 *   LSE_i  = m_i + ln sum_{allowed j} exp(s_ij - m_i),  m_i = max_{allowed j} s_ij
 *   P_ij   = allowed ? exp(s_ij - LSE_i) : 0
 *   O_i    = sum_j P_ij V[b,j,g,:]
 *   Dvec_i = sum_d dO_id O_id
 *   dP_ij  = sum_d dO_id V_jd
 *   dS_ij  = P_ij (dP_ij - Dvec_i)
 *   dQ_i   = scale sum_j dS_ij K_j
 *   dV_j   = sum_{h in group g} sum_i P_ij dO_i
 *   dK_j   = scale sum_{h in group g} sum_i dS_ij Q_i
 *
 * Layout: Q, O, dO, dQ are [B, S, H, D]; K, V, dK, dV are [B, S, Hkv, D]; LSE and the
 * row statistics are [B, H, S]; all contiguous double.  Rows are independent, so the
 * loops over rows run in parallel with OpenMP; every sum is taken in index order by
 * one thread, which makes the oracle deterministic as well.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX_Q(b, i, h, d) ((((size_t)(b) * S + (i)) * H + (h)) * D + (d))
#define IDX_K(b, j, g, d) ((((size_t)(b) * S + (j)) * Hkv + (g)) * D + (d))
#define IDX_R(b, h, i) (((size_t)(b) * H + (h)) * S + (i))

static int allowed(int causal, int i, int j) { return causal ? (j <= i) : 1; }

/* s_ij for one query row: fills s[0..S) (entries outside the mask are left unused) and
 * returns LSE_i.  Definition of s_ij, m_i and LSE_i above. */
static double score_row(const double *q, const double *k, int S, int H, int Hkv, int D,
                        double scale, int causal, int b, int h, int i, double *s) {
  const int g = h / (H / Hkv);
  double m = -INFINITY;
  for (int j = 0; j < S; ++j) {
    if (!allowed(causal, i, j)) continue;
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += q[IDX_Q(b, i, h, d)] * k[IDX_K(b, j, g, d)];
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int j = 0; j < S; ++j)
    if (allowed(causal, i, j)) l += exp(s[j] - m);
  return m + log(l);
}

/* Forward: O [B,S,H,D] and LSE [B,H,S]. */
void dash_oracle_fwd(const double *q, const double *k, const double *v, int B, int S, int H,
                     int Hkv, int D, double scale, int causal, double *o, double *lse) {
  if (B <= 0 || S <= 0 || H <= 0 || Hkv <= 0 || D <= 0 || H % Hkv) return;
  const long long rows = (long long)B * H * S;
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)S);
#pragma omp for schedule(dynamic, 4)
    for (long long r = 0; r < rows; ++r) {
      const int i = (int)(r % S), h = (int)((r / S) % H), b = (int)(r / ((long long)S * H));
      const int g = h / (H / Hkv);
      const double L = score_row(q, k, S, H, Hkv, D, scale, causal, b, h, i, s);
      lse[IDX_R(b, h, i)] = L;
      for (int d = 0; d < D; ++d) o[IDX_Q(b, i, h, d)] = 0.0;
      for (int j = 0; j < S; ++j) {
        if (!allowed(causal, i, j)) continue;
        const double p = exp(s[j] - L);
        for (int d = 0; d < D; ++d) o[IDX_Q(b, i, h, d)] += p * v[IDX_K(b, j, g, d)];
      }
    }
    free(s);
  }
}

/* Backward: dQ [B,S,H,D], dK and dV [B,S,Hkv,D].  O and LSE (forward outputs, recomputed
 * here from the definition) are written to o / lse when those are non-NULL.  Returns the
 * number of OpenMP threads used. */
int dash_oracle_bwd(const double *q, const double *k, const double *v, const double *dout,
                    int B, int S, int H, int Hkv, int D, double scale, int causal, double *dq,
                    double *dk, double *dv, double *o, double *lse) {
  if (B <= 0 || S <= 0 || H <= 0 || Hkv <= 0 || D <= 0 || H % Hkv) return 0;
  const int G = H / Hkv;
  double *LSE = (double *)malloc(sizeof(double) * (size_t)B * H * S);
  double *Dvec = (double *)malloc(sizeof(double) * (size_t)B * H * S);
  int threads = 1;

  /* Row pass: LSE_i, O_i, Dvec_i and dQ_i for every query row i of every head. */
  const long long rows = (long long)B * H * S;
#pragma omp parallel
  {
#ifdef _OPENMP
#pragma omp single
    threads = omp_get_num_threads();
#endif
    double *s = (double *)malloc(sizeof(double) * (size_t)S);
    double *orow = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 4)
    for (long long r = 0; r < rows; ++r) {
      const int i = (int)(r % S), h = (int)((r / S) % H), b = (int)(r / ((long long)S * H));
      const int g = h / G;
      const double L = score_row(q, k, S, H, Hkv, D, scale, causal, b, h, i, s);
      LSE[IDX_R(b, h, i)] = L;
      for (int d = 0; d < D; ++d) orow[d] = 0.0;
      for (int j = 0; j < S; ++j) {
        if (!allowed(causal, i, j)) continue;
        const double p = exp(s[j] - L);
        for (int d = 0; d < D; ++d) orow[d] += p * v[IDX_K(b, j, g, d)];
      }
      double dvec = 0.0;
      for (int d = 0; d < D; ++d) dvec += dout[IDX_Q(b, i, h, d)] * orow[d];
      Dvec[IDX_R(b, h, i)] = dvec;
      if (o)
        for (int d = 0; d < D; ++d) o[IDX_Q(b, i, h, d)] = orow[d];
      for (int d = 0; d < D; ++d) dq[IDX_Q(b, i, h, d)] = 0.0;
      for (int j = 0; j < S; ++j) {
        if (!allowed(causal, i, j)) continue;
        const double p = exp(s[j] - L);
        double dp = 0.0;
        for (int d = 0; d < D; ++d) dp += dout[IDX_Q(b, i, h, d)] * v[IDX_K(b, j, g, d)];
        const double ds = p * (dp - dvec);
        for (int d = 0; d < D; ++d) dq[IDX_Q(b, i, h, d)] += ds * k[IDX_K(b, j, g, d)];
      }
      for (int d = 0; d < D; ++d) dq[IDX_Q(b, i, h, d)] *= scale;
    }
    free(orow);
    free(s);
  }

  /* Key pass: dV_j and dK_j for every key row j of every kv head, summing over the G
   * query heads of the group in ascending order and over query rows i in ascending
   * order.  P_ij and dS_ij are re-evaluated from their definitions with the LSE_i and
   * Dvec_i of the row pass. */
  const long long krows = (long long)B * Hkv * S;
#pragma omp parallel for schedule(dynamic, 4)
  for (long long r = 0; r < krows; ++r) {
    const int j = (int)(r % S), g = (int)((r / S) % Hkv), b = (int)(r / ((long long)S * Hkv));
    for (int d = 0; d < D; ++d) {
      dk[IDX_K(b, j, g, d)] = 0.0;
      dv[IDX_K(b, j, g, d)] = 0.0;
    }
    for (int hh = 0; hh < G; ++hh) {
      const int h = g * G + hh;
      for (int i = 0; i < S; ++i) {
        if (!allowed(causal, i, j)) continue;
        double qk = 0.0, dp = 0.0;
        for (int d = 0; d < D; ++d) {
          qk += q[IDX_Q(b, i, h, d)] * k[IDX_K(b, j, g, d)];
          dp += dout[IDX_Q(b, i, h, d)] * v[IDX_K(b, j, g, d)];
        }
        const double p = exp(scale * qk - LSE[IDX_R(b, h, i)]);
        const double ds = p * (dp - Dvec[IDX_R(b, h, i)]);
        for (int d = 0; d < D; ++d) {
          dv[IDX_K(b, j, g, d)] += p * dout[IDX_Q(b, i, h, d)];
          dk[IDX_K(b, j, g, d)] += ds * q[IDX_Q(b, i, h, d)];
        }
      }
    }
    for (int d = 0; d < D; ++d) dk[IDX_K(b, j, g, d)] *= scale;
  }

  if (lse) memcpy(lse, LSE, sizeof(double) * (size_t)B * H * S);
  free(LSE);
  free(Dvec);
  return threads;
}

/* Sampled gradients of one (batch, kv head) group at full length, for parity checks at
 * sizes where the whole backward is too slow on the CPU.  Same definitions as above,
 * evaluated for chosen rows only: LSE_i and Dvec_i for every query row of every head of
 * the group (a full pass), then dQ_i (each query head) for the query rows qrows[0..nq)
 * and dK_j, dV_j (summed over the group's heads) for the key rows krows[0..nk).
 * Slice layout: q, dout [S, G, D]; k, v [S, D]; dq out [nq, G, D]; dk, dv out [nk, D].
 * Returns the number of OpenMP threads used. */
#define SQ(i, hh, d) (((size_t)(i) * G + (hh)) * D + (d))
#define SK(j, d) ((size_t)(j) * D + (d))
int dash_oracle_bwd_rows(const double *q, const double *k, const double *v,
                         const double *dout, int S, int G, int D, double scale, int causal,
                         int nq, const int *qrows, int nk, const int *krows, double *dq,
                         double *dk, double *dv) {
  if (S <= 0 || G <= 0 || D <= 0 || nq < 0 || nk < 0) return 0;
  double *LSE = (double *)malloc(sizeof(double) * (size_t)G * S);
  double *Dvec = (double *)malloc(sizeof(double) * (size_t)G * S);
  int threads = 1;
#pragma omp parallel
  {
#ifdef _OPENMP
#pragma omp single
    threads = omp_get_num_threads();
#endif
    double *s = (double *)malloc(sizeof(double) * (size_t)S);
    double *orow = (double *)malloc(sizeof(double) * (size_t)D);
    /* LSE_i, O_i and Dvec_i of every row of every head of the group */
#pragma omp for schedule(dynamic, 4)
    for (long long r = 0; r < (long long)G * S; ++r) {
      const int hh = (int)(r / S), i = (int)(r % S);
      double m = -INFINITY;
      for (int j = 0; j < S; ++j) {
        if (!allowed(causal, i, j)) continue;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[SQ(i, hh, d)] * k[SK(j, d)];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
      }
      double l = 0.0;
      for (int j = 0; j < S; ++j)
        if (allowed(causal, i, j)) l += exp(s[j] - m);
      const double L = m + log(l);
      for (int d = 0; d < D; ++d) orow[d] = 0.0;
      for (int j = 0; j < S; ++j) {
        if (!allowed(causal, i, j)) continue;
        const double p = exp(s[j] - L);
        for (int d = 0; d < D; ++d) orow[d] += p * v[SK(j, d)];
      }
      double dvec = 0.0;
      for (int d = 0; d < D; ++d) dvec += dout[SQ(i, hh, d)] * orow[d];
      LSE[(size_t)hh * S + i] = L;
      Dvec[(size_t)hh * S + i] = dvec;
    }
    /* dQ_i = scale sum_j P_ij (dP_ij - Dvec_i) K_j for the sampled query rows */
#pragma omp for schedule(dynamic, 1)
    for (long long r = 0; r < (long long)nq * G; ++r) {
      const int n = (int)(r / G), hh = (int)(r % G), i = qrows[n];
      for (int d = 0; d < D; ++d) dq[((size_t)n * G + hh) * D + d] = 0.0;
      for (int j = 0; j < S; ++j) {
        if (!allowed(causal, i, j)) continue;
        double sc = 0.0, dp = 0.0;
        for (int d = 0; d < D; ++d) {
          sc += q[SQ(i, hh, d)] * k[SK(j, d)];
          dp += dout[SQ(i, hh, d)] * v[SK(j, d)];
        }
        const double p = exp(scale * sc - LSE[(size_t)hh * S + i]);
        const double ds = p * (dp - Dvec[(size_t)hh * S + i]);
        for (int d = 0; d < D; ++d) dq[((size_t)n * G + hh) * D + d] += scale * ds * k[SK(j, d)];
      }
    }
    /* dV_j = sum_hh sum_i P_ij dO_i and dK_j = scale sum_hh sum_i dS_ij Q_i, sampled key rows */
#pragma omp for schedule(dynamic, 1)
    for (int n = 0; n < nk; ++n) {
      const int j = krows[n];
      for (int d = 0; d < D; ++d) {
        dk[(size_t)n * D + d] = 0.0;
        dv[(size_t)n * D + d] = 0.0;
      }
      for (int hh = 0; hh < G; ++hh) {
        for (int i = 0; i < S; ++i) {
          if (!allowed(causal, i, j)) continue;
          double sc = 0.0, dp = 0.0;
          for (int d = 0; d < D; ++d) {
            sc += q[SQ(i, hh, d)] * k[SK(j, d)];
            dp += dout[SQ(i, hh, d)] * v[SK(j, d)];
          }
          const double p = exp(scale * sc - LSE[(size_t)hh * S + i]);
          const double ds = p * (dp - Dvec[(size_t)hh * S + i]);
          for (int d = 0; d < D; ++d) {
            dv[(size_t)n * D + d] += p * dout[SQ(i, hh, d)];
            dk[(size_t)n * D + d] += scale * ds * q[SQ(i, hh, d)];
          }
        }
      }
    }
    free(s);
    free(orow);
  }
  free(LSE);
  free(Dvec);
  return threads;
}
#undef SQ
#undef SK
