/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the O = f(A.B).C unit.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  The
 * product path (chain_gb300) never calls it and shares no code, header,
 * table or helper with it.
 *
 * Every function computes the plain definition, materialising what the GPU
 * path never materialises (full score rows, the full hidden activation row),
 * with no blocking, fusion or reordering beyond what the definition states.
 * Inputs are read as stored (bf16 or e4m3 bit patterns, fp32 or fp64) and
 * widened exactly to double; all arithmetic is double.
 *
 * Sources (page titles of the method's write-ups):
 *  - "Memory-efficient tensor parallelism" (FITEE 10.1631/FITEE.2400602),
 *    abstract: the unit is two consecutive matrix products with a function
 *    between them, O = f(AB)C.
 *  - "Ulysses Sequence Parallelism: Entrainement avec des Contextes de
 *    Millions de Jetons", "Contexte Technique": attention tiled so that the
 *    n x n score matrix is never stored; sequence shards redistributed so
 *    each device holds every position for a subset of heads.
 *  - "AutoSP: Unlocking Long-Context LLM Training Via Compiler-Based Sequence
 *    Parallelism", section 2.A item 4 (causal masks recomputed on global
 *    positions) and section 2.B (recompute rather than store activations for
 *    the backward pass).
 * The readings the pages leave open (scale placement, natural-log LSE,
 * causal convention j <= i, GeLU tanh form) are the ones stated at each
 * function.
 *
 * Parity pins (in tests/): closed forms for uniform scores and causal row 0,
 * hand-derived goldens, independent library routines (scaled-dot-product
 * attention, autograd, tanh-GeLU in fp64), central finite differences,
 * the blocked online merge against the unblocked definition, associativity
 * of the identity chain, and permutation round trips.  No function here is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BF16 0
#define ORACLE_F32 1
#define ORACLE_F64 2
#define ORACLE_E4M3 3

#define ORACLE_F_IDENTITY 0
#define ORACLE_F_SOFTMAX 1
#define ORACLE_F_GELU_TANH 2

/* The 8-bit float e4m3 from its definition: sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 is subnormal (2^-6 * m/8); no
 * infinities; exponent 15 with mantissa 7 is NaN. */
static double e4m3_value(uint8_t b) {
  const int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

void oracle_e4m3_decode(const uint8_t *in, int64_t count, double *out) {
  for (int64_t i = 0; i < count; ++i) out[i] = e4m3_value(in[i]);
}

/* Exact widening of one stored element to double.  A bf16 value is the top
 * 16 bits of an IEEE binary32, so shifting the pattern up reproduces it. */
static double elem(const void *base, int dtype, int64_t i) {
  if (dtype == ORACLE_E4M3) return e4m3_value(((const uint8_t *)base)[i]);
  if (dtype == ORACLE_BF16) {
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  if (dtype == ORACLE_F32) return (double)((const float *)base)[i];
  return ((const double *)base)[i];
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------
 * Softmax attention forward, plain definition (FITEE abstract, O = f(AB)C
 * with A = Q, B = K^T, f = row softmax of the scaled scores, C = V).
 *
 * Layout: Q, K [BH][n][d], V [BH][n][dv], row-major, contiguous.
 * For each requested (bh, i):
 *   S_j   = scale * sum_e Q[i][e] K[j][e]   for every key j, j <= i if causal
 *           (causal masked keys are excluded outright, AutoSP 2.A item 4)
 *   m     = max_j S_j,  l = sum_j exp(S_j - m)
 *   P_j   = exp(S_j - m) / l
 *   O[i]  = sum_j P_j V[j]
 *   LSE_i = m + ln l                        (natural log, scale included)
 * Outputs O [R][dv] and LSE [R] in request order.
 * ---------------------------------------------------------------------- */
int oracle_softmax_fwd(int dtype, const void *Q, const void *K, const void *V,
                       int64_t BH, int64_t n, int64_t d, int64_t dv,
                       double scale, int causal, int64_t R,
                       const int64_t *req_bh, const int64_t *req_row,
                       double *O, double *LSE) {
  if (n <= 0 || d <= 0 || dv <= 0) return -1;
  for (int64_t r = 0; r < R; ++r)
    if (req_bh[r] < 0 || req_bh[r] >= BH || req_row[r] < 0 || req_row[r] >= n)
      return -2;
  int bad = 0;
#pragma omp parallel
  {
    double *S = (double *)malloc(sizeof(double) * (size_t)n);
    if (!S) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < R; ++r) {
      if (!S) continue;
      const int64_t bh = req_bh[r], i = req_row[r];
      const int64_t nk = causal ? i + 1 : n;
      const int64_t qo = (bh * n + i) * d;
      double m = -INFINITY;
      for (int64_t j = 0; j < nk; ++j) {
        const int64_t ko = (bh * n + j) * d;
        double acc = 0.0;
        for (int64_t e = 0; e < d; ++e)
          acc += elem(Q, dtype, qo + e) * elem(K, dtype, ko + e);
        S[j] = scale * acc;
        if (S[j] > m) m = S[j];
      }
      double l = 0.0;
      for (int64_t j = 0; j < nk; ++j) l += exp(S[j] - m);
      double *o = O + r * dv;
      for (int64_t e = 0; e < dv; ++e) o[e] = 0.0;
      for (int64_t j = 0; j < nk; ++j) {
        const double p = exp(S[j] - m) / l;
        const int64_t vo = (bh * n + j) * dv;
        for (int64_t e = 0; e < dv; ++e) o[e] += p * elem(V, dtype, vo + e);
      }
      LSE[r] = m + log(l);
    }
    free(S);
  }
  return bad ? -3 : 0;
}

/* ------------------------------------------------------------------------
 * The same forward as a pq x pk block decomposition: query rows split into
 * pq contiguous blocks, keys into pk contiguous blocks.  Each (row block,
 * key block) pair yields, per row, its partial (m_b, l_b, U_b) with
 * U_b = sum_{j in b} exp(S_j - m_b) V[j]; partials are merged with
 * m = max_b m_b, l = sum_b exp(m_b - m) l_b, O = sum_b exp(m_b - m) U_b / l.
 * This is the blockwise merge that lets METP split O into sub-tasks (FITEE
 * abstract); in exact arithmetic it equals oracle_softmax_fwd.  Blocks with
 * no unmasked key contribute nothing.  All rows of all heads; small sizes.
 * ---------------------------------------------------------------------- */
int oracle_softmax_fwd_blocked(int dtype, const void *Q, const void *K,
                               const void *V, int64_t BH, int64_t n, int64_t d,
                               int64_t dv, double scale, int causal, int64_t pq,
                               int64_t pk, double *O, double *LSE) {
  if (n <= 0 || pq <= 0 || pk <= 0 || pq > n || pk > n) return -1;
  double *mb = (double *)malloc(sizeof(double) * (size_t)pk);
  double *lb = (double *)malloc(sizeof(double) * (size_t)pk);
  double *Ub = (double *)malloc(sizeof(double) * (size_t)(pk * dv));
  if (!mb || !lb || !Ub) {
    free(mb); free(lb); free(Ub);
    return -3;
  }
  for (int64_t bh = 0; bh < BH; ++bh) {
    for (int64_t qb = 0; qb < pq; ++qb) {
      const int64_t r0 = qb * n / pq, r1 = (qb + 1) * n / pq;
      for (int64_t i = r0; i < r1; ++i) {
        const int64_t qo = (bh * n + i) * d;
        /* partial state of each key block for row i */
        for (int64_t kb = 0; kb < pk; ++kb) {
          const int64_t c0 = kb * n / pk, c1 = (kb + 1) * n / pk;
          double m = -INFINITY;
          for (int64_t j = c0; j < c1; ++j) {
            if (causal && j > i) break;
            double acc = 0.0;
            for (int64_t e = 0; e < d; ++e)
              acc += elem(Q, dtype, qo + e) * elem(K, dtype, (bh * n + j) * d + e);
            if (scale * acc > m) m = scale * acc;
          }
          mb[kb] = m;
          lb[kb] = 0.0;
          for (int64_t e = 0; e < dv; ++e) Ub[kb * dv + e] = 0.0;
          if (m == -INFINITY) continue; /* fully masked block */
          for (int64_t j = c0; j < c1; ++j) {
            if (causal && j > i) break;
            double acc = 0.0;
            for (int64_t e = 0; e < d; ++e)
              acc += elem(Q, dtype, qo + e) * elem(K, dtype, (bh * n + j) * d + e);
            const double w = exp(scale * acc - m);
            lb[kb] += w;
            for (int64_t e = 0; e < dv; ++e)
              Ub[kb * dv + e] += w * elem(V, dtype, (bh * n + j) * dv + e);
          }
        }
        /* merge */
        double m = -INFINITY;
        for (int64_t kb = 0; kb < pk; ++kb)
          if (mb[kb] > m) m = mb[kb];
        double l = 0.0;
        double *o = O + (bh * n + i) * dv;
        for (int64_t e = 0; e < dv; ++e) o[e] = 0.0;
        for (int64_t kb = 0; kb < pk; ++kb) {
          if (mb[kb] == -INFINITY) continue;
          const double a = exp(mb[kb] - m);
          l += a * lb[kb];
          for (int64_t e = 0; e < dv; ++e) o[e] += a * Ub[kb * dv + e];
        }
        for (int64_t e = 0; e < dv; ++e) o[e] /= l;
        LSE[bh * n + i] = m + log(l);
      }
    }
  }
  free(mb); free(lb); free(Ub);
  return 0;
}

/* The stored elements [off, off + count) widened exactly to double. */
static double *widen(const void *base, int dtype, int64_t off, int64_t count) {
  double *w = (double *)malloc(sizeof(double) * (size_t)(count > 0 ? count : 1));
  if (!w) return NULL;
  for (int64_t t = 0; t < count; ++t) w[t] = elem(base, dtype, off + t);
  return w;
}

/* ------------------------------------------------------------------------
 * Softmax attention backward by the textbook chain rule, without any
 * recompute trick (the GPU path recomputes S and P from the LSE, AutoSP 2.B;
 * the oracle simply redoes the forward row by row).
 *
 * For each row i in [i0, i1) of each head in [bh0, bh1):
 *   P_ij  as in oracle_softmax_fwd
 *   dP_ij = sum_e dO[i][e] V[j][e]
 *   D_i   = sum_j P_ij dP_ij
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ[i] = scale * sum_j dS_ij K[j]
 *   dK[j] += scale * dS_ij Q[i],  dV[j] += P_ij dO[i]
 * dQ [bh1-bh0][i1-i0][d] and D [bh1-bh0][i1-i0] cover the requested rows;
 * dK [bh1-bh0][j1-j0][d], dV [..][j1-j0][dv] hold the contributions of those
 * rows to key columns [j0, j1).  With i0 = j0 = 0, i1 = j1 = n the result is
 * the full gradient; with causal masking, columns j >= i0 are complete
 * whenever i1 = n (no row before i0 reaches them).
 * ---------------------------------------------------------------------- */
int oracle_softmax_bwd(int dtype, const void *Q, const void *K, const void *V,
                       const void *dO, int64_t BH, int64_t n, int64_t d,
                       int64_t dv, double scale, int causal, int64_t bh0,
                       int64_t bh1, int64_t i0, int64_t i1, int64_t j0,
                       int64_t j1, double *dQ, double *dK, double *dV,
                       double *D) {
  if (n <= 0 || bh0 < 0 || bh1 > BH || bh0 >= bh1 || i0 < 0 || i1 > n ||
      i0 >= i1 || j0 < 0 || j1 > n || j0 >= j1)
    return -1;
  const int64_t nh = bh1 - bh0, nr = i1 - i0, nc = j1 - j0;
  /* the requested heads, widened to double once (exact) */
  double *q = widen(Q, dtype, bh0 * n * d, nh * n * d);
  double *k = widen(K, dtype, bh0 * n * d, nh * n * d);
  double *v = widen(V, dtype, bh0 * n * dv, nh * n * dv);
  double *g = widen(dO, dtype, bh0 * n * dv, nh * n * dv);
  const int nt = oracle_num_threads();
  double **pKt = (double **)calloc((size_t)nt, sizeof(double *));
  double **pVt = (double **)calloc((size_t)nt, sizeof(double *));
  int bad = !q || !k || !v || !g || !pKt || !pVt;
  if (!bad) {
#pragma omp parallel num_threads(nt)
    {
      int t = 0;
#ifdef _OPENMP
      t = omp_get_thread_num();
#endif
      double *S = (double *)malloc(sizeof(double) * (size_t)n);
      double *dP = (double *)malloc(sizeof(double) * (size_t)n);
      /* this thread's share of the dK, dV sums over rows */
      double *pK = (double *)calloc((size_t)(nh * nc * d), sizeof(double));
      double *pV = (double *)calloc((size_t)(nh * nc * dv), sizeof(double));
      pKt[t] = pK;
      pVt[t] = pV;
      if (!S || !dP || !pK || !pV) {
#pragma omp atomic write
        bad = 1;
      }
      /* rows dealt round-robin: each thread's share of the row sums is the
       * same on every run */
#pragma omp for schedule(static, 1) collapse(2)
      for (int64_t h = 0; h < nh; ++h) {
        for (int64_t r = 0; r < nr; ++r) {
          if (!S || !dP || !pK || !pV) continue;
          const int64_t i = i0 + r;
          const int64_t nk = causal ? i + 1 : n;
          const double *qi = q + (h * n + i) * d, *gi = g + (h * n + i) * dv;
          double m = -INFINITY;
          for (int64_t j = 0; j < nk; ++j) {
            const double *kj = k + (h * n + j) * d, *vj = v + (h * n + j) * dv;
            double acc = 0.0;
            for (int64_t e = 0; e < d; ++e) acc += qi[e] * kj[e];
            S[j] = scale * acc;
            if (S[j] > m) m = S[j];
            double gv = 0.0;
            for (int64_t e = 0; e < dv; ++e) gv += gi[e] * vj[e];
            dP[j] = gv;
          }
          double l = 0.0;
          for (int64_t j = 0; j < nk; ++j) l += exp(S[j] - m);
          double Di = 0.0;
          for (int64_t j = 0; j < nk; ++j) {
            S[j] = exp(S[j] - m) / l; /* S now holds P */
            Di += S[j] * dP[j];
          }
          D[h * nr + r] = Di;
          double *dq = dQ + (h * nr + r) * d;
          for (int64_t e = 0; e < d; ++e) dq[e] = 0.0;
          for (int64_t j = 0; j < nk; ++j) {
            const double ds = S[j] * (dP[j] - Di);
            const double *kj = k + (h * n + j) * d;
            for (int64_t e = 0; e < d; ++e) dq[e] += scale * ds * kj[e];
            if (j >= j0 && j < j1) {
              double *kk = pK + (h * nc + (j - j0)) * d;
              double *vv = pV + (h * nc + (j - j0)) * dv;
              for (int64_t e = 0; e < d; ++e) kk[e] += scale * ds * qi[e];
              for (int64_t e = 0; e < dv; ++e) vv[e] += S[j] * gi[e];
            }
          }
        }
      }
      free(S);
      free(dP);
    }
  }
  /* dK, dV: the threads' shares added in thread order (deterministic) */
  memset(dK, 0, sizeof(double) * (size_t)(nh * nc * d));
  memset(dV, 0, sizeof(double) * (size_t)(nh * nc * dv));
  for (int t = 0; t < nt && !bad; ++t) {
    if (!pKt[t] || !pVt[t]) continue; /* a thread that ran no iteration */
    for (int64_t u = 0; u < nh * nc * d; ++u) dK[u] += pKt[t][u];
    for (int64_t u = 0; u < nh * nc * dv; ++u) dV[u] += pVt[t][u];
  }
  for (int t = 0; t < nt && pKt && pVt; ++t) {
    free(pKt[t]);
    free(pVt[t]);
  }
  free(pKt); free(pVt);
  free(q); free(k); free(v); free(g);
  return bad ? -3 : 0;
}

/* tanh form of GeLU (Hendrycks & Gimpel): 0.5 t (1 + tanh(sqrt(2/pi)(t + 0.044715 t^3))) */
static double gelu_tanh(double t) {
  const double k = sqrt(2.0 / M_PI);
  return 0.5 * t * (1.0 + tanh(k * (t + 0.044715 * t * t * t)));
}

/* ------------------------------------------------------------------------
 * General chain O = f(A B) C (FITEE abstract) for requested rows of A.
 * A [M][K], B [K][N], C [N][P], row-major.  For each requested row r:
 *   T_c = sum_k A[r][k] B[k][c]        (the full row of the intermediate)
 *   H   = f(T):  identity; gelu_tanh elementwise; or row softmax of scale*T
 *   O[r] = sum_c H_c C[c]
 * The intermediate is kept in double and never rounded.  (For f = softmax
 * the scale multiplies T; elsewhere it is ignored.)
 * ---------------------------------------------------------------------- */
int oracle_chain_fwd(int dtype, const void *A, const void *B, const void *C,
                     int64_t M, int64_t K, int64_t N, int64_t P, int f,
                     double scale, int64_t R, const int64_t *rows, double *O) {
  if (M <= 0 || K <= 0 || N <= 0 || P <= 0) return -1;
  if (f != ORACLE_F_IDENTITY && f != ORACLE_F_SOFTMAX && f != ORACLE_F_GELU_TANH) return -1;
  for (int64_t r = 0; r < R; ++r)
    if (rows[r] < 0 || rows[r] >= M) return -2;
  int bad = 0;
#pragma omp parallel
  {
    double *T = (double *)malloc(sizeof(double) * (size_t)N);
    if (!T) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < R; ++r) {
      if (!T) continue;
      const int64_t a = rows[r];
      for (int64_t c = 0; c < N; ++c) T[c] = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double av = elem(A, dtype, a * K + k);
        for (int64_t c = 0; c < N; ++c) T[c] += av * elem(B, dtype, k * N + c);
      }
      if (f == ORACLE_F_GELU_TANH) {
        for (int64_t c = 0; c < N; ++c) T[c] = gelu_tanh(T[c]);
      } else if (f == ORACLE_F_SOFTMAX) {
        double m = -INFINITY, l = 0.0;
        for (int64_t c = 0; c < N; ++c) {
          T[c] *= scale;
          if (T[c] > m) m = T[c];
        }
        for (int64_t c = 0; c < N; ++c) l += exp(T[c] - m);
        for (int64_t c = 0; c < N; ++c) T[c] = exp(T[c] - m) / l;
      }
      double *o = O + r * P;
      for (int64_t e = 0; e < P; ++e) o[e] = 0.0;
      for (int64_t c = 0; c < N; ++c) {
        const double h = T[c];
        for (int64_t e = 0; e < P; ++e) o[e] += h * elem(C, dtype, c * P + e);
      }
    }
    free(T);
  }
  return bad ? -3 : 0;
}

/* derivative of the tanh form of GeLU: with u = k (t + 0.044715 t^3),
 * k = sqrt(2/pi):  0.5 (1 + tanh u) + 0.5 t (1 - tanh^2 u) k (1 + 3*0.044715 t^2) */
static double gelu_tanh_grad(double t) {
  const double k = sqrt(2.0 / M_PI);
  const double th = tanh(k * (t + 0.044715 * t * t * t));
  return 0.5 * (1.0 + th) + 0.5 * t * (1.0 - th * th) * k * (1.0 + 3.0 * 0.044715 * t * t);
}

/* ------------------------------------------------------------------------
 * Backward of the chain O = f(A B) C for f = identity or gelu_tanh, the
 * intermediate recomputed from A and B instead of stored (AutoSP, section
 * 2.B).  Given dO [M][P], by the chain rule:
 *   T = A B,  H = f(T),  dH = dO C^T,  dT = dH * f'(T)   (elementwise)
 *   dC = H^T dO,   dA = dT B^T,   dB = A^T dT.
 * Outputs for requested rows ra of dA:            dA_out [RA][K]
 * and requested hidden units rh: row h of dC,      dC_out [RH][P]
 *                                column h of dB,   dB_out [RH][K]
 * Everything in double; T, H, dH, dT are never rounded.
 * ---------------------------------------------------------------------- */
int oracle_chain_bwd(int dtype, const void *A, const void *B, const void *C, const void *dO,
                     int64_t M, int64_t K, int64_t N, int64_t P, int f, int64_t RA,
                     const int64_t *ra, int64_t RH, const int64_t *rh, double *dA_out,
                     double *dB_out, double *dC_out) {
  if (M <= 0 || K <= 0 || N <= 0 || P <= 0) return -1;
  if (f != ORACLE_F_IDENTITY && f != ORACLE_F_GELU_TANH) return -1;
  for (int64_t r = 0; r < RA; ++r)
    if (ra[r] < 0 || ra[r] >= M) return -2;
  for (int64_t r = 0; r < RH; ++r)
    if (rh[r] < 0 || rh[r] >= N) return -2;
  int bad = 0;
  /* rows of dA: one full row of T, dH and dT per requested row */
#pragma omp parallel
  {
    double *dT = (double *)malloc(sizeof(double) * (size_t)N);
    if (!dT) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < RA; ++r) {
      if (!dT) continue;
      const int64_t a = ra[r];
      for (int64_t c = 0; c < N; ++c) {
        double t = 0.0, dh = 0.0;
        for (int64_t k = 0; k < K; ++k) t += elem(A, dtype, a * K + k) * elem(B, dtype, k * N + c);
        for (int64_t e = 0; e < P; ++e) dh += elem(dO, dtype, a * P + e) * elem(C, dtype, c * P + e);
        dT[c] = dh * (f == ORACLE_F_GELU_TANH ? gelu_tanh_grad(t) : 1.0);
      }
      for (int64_t k = 0; k < K; ++k) {
        double acc = 0.0;
        for (int64_t c = 0; c < N; ++c) acc += dT[c] * elem(B, dtype, k * N + c);
        dA_out[r * K + k] = acc;
      }
    }
    free(dT);
  }
  /* hidden units: the full column h of T, H, dH and dT over all M rows */
#pragma omp parallel
  {
    double *Hc = (double *)malloc(sizeof(double) * (size_t)M);
    double *dTc = (double *)malloc(sizeof(double) * (size_t)M);
    if (!Hc || !dTc) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < RH; ++r) {
      if (!Hc || !dTc) continue;
      const int64_t h = rh[r];
      for (int64_t m = 0; m < M; ++m) {
        double t = 0.0, dh = 0.0;
        for (int64_t k = 0; k < K; ++k) t += elem(A, dtype, m * K + k) * elem(B, dtype, k * N + h);
        for (int64_t e = 0; e < P; ++e) dh += elem(dO, dtype, m * P + e) * elem(C, dtype, h * P + e);
        Hc[m] = f == ORACLE_F_GELU_TANH ? gelu_tanh(t) : t;
        dTc[m] = dh * (f == ORACLE_F_GELU_TANH ? gelu_tanh_grad(t) : 1.0);
      }
      for (int64_t e = 0; e < P; ++e) {
        double acc = 0.0;
        for (int64_t m = 0; m < M; ++m) acc += Hc[m] * elem(dO, dtype, m * P + e);
        dC_out[r * P + e] = acc;
      }
      for (int64_t k = 0; k < K; ++k) {
        double acc = 0.0;
        for (int64_t m = 0; m < M; ++m) acc += elem(A, dtype, m * K + k) * dTc[m];
        dB_out[r * K + k] = acc;
      }
    }
    free(Hc);
    free(dTc);
  }
  return bad ? -3 : 0;
}

/* ------------------------------------------------------------------------
 * Ulysses sequence-shard -> head-major redistribution ("Contexte
 * Technique": after the exchange each device holds every sequence position
 * for a subset of heads).  Shard s holds the contiguous positions
 * [s*n_loc, (s+1)*n_loc); heads go to groups contiguously, Hl = H/p per
 * group.  in [p][n_loc][H][d] -> out [Hl][p*n_loc][d] for group g:
 *   out[h][s*n_loc + t][e] = in[s][t][g*Hl + h][e]
 * Elements are moved as opaque byte strings of elem_bytes.
 * ---------------------------------------------------------------------- */
int oracle_relayout(const void *in, int64_t elem_bytes, int64_t p,
                    int64_t n_loc, int64_t H, int64_t d, int64_t g, void *out) {
  if (p <= 0 || H % p != 0 || g < 0 || g >= p || elem_bytes <= 0) return -1;
  const int64_t Hl = H / p;
  const unsigned char *src = (const unsigned char *)in;
  unsigned char *dst = (unsigned char *)out;
  for (int64_t h = 0; h < Hl; ++h)
    for (int64_t s = 0; s < p; ++s)
      for (int64_t t = 0; t < n_loc; ++t)
        for (int64_t e = 0; e < d; ++e) {
          const int64_t o = (h * (p * n_loc) + s * n_loc + t) * d + e;
          const int64_t i = ((s * n_loc + t) * H + g * Hl + h) * d + e;
          memcpy(dst + o * elem_bytes, src + i * elem_bytes, (size_t)elem_bytes);
        }
  return 0;
}

/* Inverse of oracle_relayout (the second Ulysses exchange, head-major back
 * to sequence shards): writes only the heads of group g in out
 * [p][n_loc][H][d]; other heads are left untouched. */
int oracle_relayout_inverse(const void *in, int64_t elem_bytes, int64_t p,
                            int64_t n_loc, int64_t H, int64_t d, int64_t g,
                            void *out) {
  if (p <= 0 || H % p != 0 || g < 0 || g >= p || elem_bytes <= 0) return -1;
  const int64_t Hl = H / p;
  const unsigned char *src = (const unsigned char *)in;
  unsigned char *dst = (unsigned char *)out;
  for (int64_t s = 0; s < p; ++s)
    for (int64_t t = 0; t < n_loc; ++t)
      for (int64_t h = 0; h < Hl; ++h)
        for (int64_t e = 0; e < d; ++e) {
          const int64_t o = ((s * n_loc + t) * H + g * Hl + h) * d + e;
          const int64_t i = (h * (p * n_loc) + s * n_loc + t) * d + e;
          memcpy(dst + o * elem_bytes, src + i * elem_bytes, (size_t)elem_bytes);
        }
  return 0;
}
