/*
 * oracle.c — the reference for causal grouped-query attention, forward and
 * backward, computed slowly and plainly in double precision on the CPU.
 *
 * TEST INFRASTRUCTURE. This is the checker of the CUDA library, not a part of
 * it: only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * it. It shares no code, header or table with the CUDA path.
 *
 * Source: "A transformer in PTX" (mnemonic-site, 5-transformer).
 *  - §The model: a causal decoder; attention is grouped-query, several query
 *    heads share one key/value head (6 query heads of 64 over 2 kv heads in the
 *    dev preset).
 *  - §Flash attention: the naive kernels write the whole T x T score matrix;
 *    the flash kernel reaches the same softmax(QK^T * scale) V by tiles, with
 *    the scores scaled by 1/sqrt(d) (the page's log2(e)/sqrt(64) is that
 *    scale in log2 units) and the per-row log-sum-exp saved for the backward.
 *  - §The same bits every time: the backward recomputes the probabilities;
 *    dQ is owned per query row, dK/dV per key row summed over every query head
 *    that shares the kv head, each sum in one fixed order.
 *
 * Because the flash kernels reach, up to rounding order, the plain definition
 * of attention, this file is that definition written out:
 *   s_ij   = scale * sum_c q_ic k_jc           (every entry is computed)
 *   s_ij   = -inf for j > i when causal        (key j visible to query i iff j <= i)
 *   LSE_i  = log sum_j exp(s_ij)                (natural log, max subtracted first)
 *   P_ij   = exp(s_ij - LSE_i)
 *   O_i    = sum_j P_ij v_j
 * and, for the loss L = sum(O * dO):
 *   dV_j   = sum_{h in group} sum_i P_ij dO_i
 *   dP_ij  = dO_i . v_j
 *   D_i    = dO_i . O_i
 *   dS_ij  = P_ij (dP_ij - D_i)
 *   dQ_i   = scale sum_j dS_ij k_j
 *   dK_j   = scale sum_{h in group} sum_i dS_ij q_i
 * Query head h reads kv head h / (Hq/Hkv) (contiguous groups).
 *
 * Layouts: q, o, dO, dq are [B,T,Hq,d]; k, v, dk, dv are [B,T,Hkv,d];
 * lse and D are [B,Hq,T]. All arrays are double, C-contiguous.
 * Every function returns 0 on success and -1 on a bad shape.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX(b, t, h, c, T, H, D) (((((size_t)(b) * (size_t)(T) + (size_t)(t)) * (size_t)(H) + (size_t)(h)) * (size_t)(D)) + (size_t)(c))
#define LIDX(b, h, t, H, T) ((((size_t)(b) * (size_t)(H)) + (size_t)(h)) * (size_t)(T) + (size_t)(t))

static int bad_shape(int B, int T, int Hq, int Hkv, int d) {
  return B <= 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (Hq % Hkv) != 0;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Last key index query i may see. */
static int last_key(int i, int T, int causal) { return causal ? i : T - 1; }

/*
 * Row i of the probability matrix of query head h in batch b, written to prow
 * (T entries; invisible keys get exactly 0). Returns LSE_i.
 */
static double probs_row(const double* q, const double* k, int T, int Hq, int Hkv, int d, int causal,
                        double scale, int b, int h, int i, double* prow) {
  const int kv = h / (Hq / Hkv);
  const int jmax = last_key(i, T, causal);
  double m = -INFINITY;
  for (int j = 0; j <= jmax; ++j) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += q[IDX(b, i, h, c, T, Hq, d)] * k[IDX(b, j, kv, c, T, Hkv, d)];
    prow[j] = scale * acc;
    if (prow[j] > m) m = prow[j];
  }
  double sum = 0.0;
  for (int j = 0; j <= jmax; ++j) sum += exp(prow[j] - m);
  const double lse = m + log(sum);
  for (int j = 0; j <= jmax; ++j) prow[j] = exp(prow[j] - lse);
  for (int j = jmax + 1; j < T; ++j) prow[j] = 0.0;
  return lse;
}

/*
 * The full T x T probability matrix of one (b, h) (row-major, P[i*T + j]) and
 * its LSE row. Exposed so that tests can check the softmax itself.
 */
int oracle_probs(const double* q, const double* k, int B, int T, int Hq, int Hkv, int d, int causal,
                 double scale, int b, int h, double* P, double* lse, int nthreads) {
  if (bad_shape(B, T, Hq, Hkv, d) || b < 0 || b >= B || h < 0 || h >= Hq) return -1;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
  for (int i = 0; i < T; ++i)
    lse[i] = probs_row(q, k, T, Hq, Hkv, d, causal, scale, b, h, i, P + (size_t)i * T);
  return 0;
}

/* Forward: O and LSE. */
int oracle_fwd(const double* q, const double* k, const double* v, double* o, double* lse, int B, int T, int Hq,
               int Hkv, int d, int causal, double scale, int nthreads) {
  if (bad_shape(B, T, Hq, Hkv, d)) return -1;
  set_threads(nthreads);
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < Hq; ++h) {
      const int kv = h / (Hq / Hkv);
#pragma omp parallel
      {
        double* prow = (double*)malloc(sizeof(double) * (size_t)T);
#pragma omp for schedule(dynamic, 16)
        for (int i = 0; i < T; ++i) {
          lse[LIDX(b, h, i, Hq, T)] = probs_row(q, k, T, Hq, Hkv, d, causal, scale, b, h, i, prow);
          double* oi = o + IDX(b, i, h, 0, T, Hq, d);
          for (int c = 0; c < d; ++c) oi[c] = 0.0;
          const int jmax = last_key(i, T, causal);
          for (int j = 0; j <= jmax; ++j) {
            const double p = prow[j];
            const double* vj = v + IDX(b, j, kv, 0, T, Hkv, d);
            for (int c = 0; c < d; ++c) oi[c] += p * vj[c];
          }
        }
        free(prow);
      }
    }
  }
  return 0;
}

/*
 * Backward of L = sum(O * dO). Also returns O, LSE and D (each may be NULL if
 * not wanted). dk and dv are overwritten. Per (b, h) the full P and dS
 * matrices are materialised; query heads are visited in ascending order so the
 * group sums of dK and dV each have one owner and one order.
 */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dout, double* o, double* lse,
               double* Dvec, double* dq, double* dk, double* dv, int B, int T, int Hq, int Hkv, int d, int causal,
               double scale, int nthreads) {
  if (bad_shape(B, T, Hq, Hkv, d)) return -1;
  set_threads(nthreads);
  const size_t TT = (size_t)T * (size_t)T;
  double* P = (double*)malloc(sizeof(double) * TT);
  double* dS = (double*)malloc(sizeof(double) * TT);
  double* Orow = (double*)malloc(sizeof(double) * (size_t)T * (size_t)d);
  if (!P || !dS || !Orow) {
    free(P);
    free(dS);
    free(Orow);
    return -2;
  }
  memset(dk, 0, sizeof(double) * (size_t)B * T * Hkv * d);
  memset(dv, 0, sizeof(double) * (size_t)B * T * Hkv * d);
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < Hq; ++h) {
      const int kv = h / (Hq / Hkv);
      /* rows: P, O, D, dP, dS, dQ */
#pragma omp parallel for schedule(dynamic, 8)
      for (int i = 0; i < T; ++i) {
        double* prow = P + (size_t)i * T;
        double* srow = dS + (size_t)i * T;
        const double l = probs_row(q, k, T, Hq, Hkv, d, causal, scale, b, h, i, prow);
        const int jmax = last_key(i, T, causal);
        double* oi = Orow + (size_t)i * d;
        for (int c = 0; c < d; ++c) oi[c] = 0.0;
        for (int j = 0; j <= jmax; ++j) {
          const double* vj = v + IDX(b, j, kv, 0, T, Hkv, d);
          for (int c = 0; c < d; ++c) oi[c] += prow[j] * vj[c];
        }
        const double* doi = dout + IDX(b, i, h, 0, T, Hq, d);
        double Di = 0.0;
        for (int c = 0; c < d; ++c) Di += doi[c] * oi[c];
        for (int j = 0; j <= jmax; ++j) {
          const double* vj = v + IDX(b, j, kv, 0, T, Hkv, d);
          double dp = 0.0;
          for (int c = 0; c < d; ++c) dp += doi[c] * vj[c];
          srow[j] = prow[j] * (dp - Di);
        }
        for (int j = jmax + 1; j < T; ++j) srow[j] = 0.0;
        double* dqi = dq + IDX(b, i, h, 0, T, Hq, d);
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        for (int j = 0; j <= jmax; ++j) {
          const double* kj = k + IDX(b, j, kv, 0, T, Hkv, d);
          for (int c = 0; c < d; ++c) dqi[c] += srow[j] * kj[c];
        }
        for (int c = 0; c < d; ++c) dqi[c] *= scale;
        if (o) {
          double* og = o + IDX(b, i, h, 0, T, Hq, d);
          for (int c = 0; c < d; ++c) og[c] = oi[c];
        }
        if (lse) lse[LIDX(b, h, i, Hq, T)] = l;
        if (Dvec) Dvec[LIDX(b, h, i, Hq, T)] = Di;
      }
      /* columns: dV_j += sum_i P_ij dO_i and dK_j += sum_i dS_ij q_i, i ascending.
         A thread owns 8 consecutive key rows j at a time (one cache line of a P row). */
      const int nblk = (T + 7) / 8;
#pragma omp parallel for schedule(dynamic, 4)
      for (int blk = 0; blk < nblk; ++blk) {
        const int j0 = blk * 8;
        const int j1 = (j0 + 8 < T) ? j0 + 8 : T;
        const int i0 = causal ? j0 : 0;
        for (int i = i0; i < T; ++i) {
          const double* doi = dout + IDX(b, i, h, 0, T, Hq, d);
          const double* qi = q + IDX(b, i, h, 0, T, Hq, d);
          for (int j = j0; j < j1; ++j) {
            const double p = P[(size_t)i * T + j];
            const double s = dS[(size_t)i * T + j];
            double* dvj = dv + IDX(b, j, kv, 0, T, Hkv, d);
            double* dkj = dk + IDX(b, j, kv, 0, T, Hkv, d);
            for (int c = 0; c < d; ++c) {
              dvj[c] += p * doi[c];
              dkj[c] += s * qi[c];
            }
          }
        }
      }
    }
    /* dK carries the score scale once, after the group sum */
    for (size_t x = IDX(b, 0, 0, 0, T, Hkv, d); x < IDX(b + 1, 0, 0, 0, T, Hkv, d); ++x) dk[x] *= scale;
  }
  free(P);
  free(dS);
  free(Orow);
  return 0;
}
