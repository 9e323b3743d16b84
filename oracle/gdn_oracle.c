/*
 * gdn_oracle.c -- fp64 CPU oracle for the gated delta rule forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only through the seeded input generator.
 *
 * Two deliberately independent walks of the same operation:
 *
 *  1. gdn_oracle_token_serial -- the plain definition.  One token at a time,
 *     no chunking, no exp2, no factoring.  This is the "token-serial oracle"
 *     of ROCm/rocm-libraries PR #11223 ("Correctness": it walks the gated
 *     delta rule one token at a time, so agreement tests the chunkwise
 *     factorisation itself).  Per sequence and value head hv, with the state
 *     S (dk x dv, K-first: row = key channel, logismos issue #46, "Verified
 *     implementation boundary"), natural-log decay g (issue #46, comment of
 *     Sep 8: "natural-log decay") and for t = 1..L:
 *
 *         a      = exp(g_t)            (GDN: one scalar per token and head;
 *                                       KDA: one value per key channel)
 *         S      = diag(a) S           (decay first)
 *         u      = v_t - S^T k_t       (delta against the decayed state)
 *         S      = S + beta_t k_t u^T  (rank-1 write)
 *         o_t    = scale S^T q_t       (read with the updated state)
 *
 *     hT = S after the last token.  The value head hv reads q/k head
 *     hv / (HV/H) (grouped heads, issue #46 "generic grouped-head mapping").
 *
 *  2. gdn_oracle_chunked -- the chunk-parallel WY form of stratat pull #1296
 *     ("What this is": per sub-chunk one C x C unit-lower-triangular solve plus
 *     GEMM-shaped folds) with the six state-independent tiles of PR #11223
 *     ("Summary": A, GK, GQ, Aqk, Kt, dec).  Pairwise decays are formed
 *     directly as exp(b_r - b_s) per pair (and per channel for KDA), with no
 *     midpoint factoring (PR #11223 "Correctness", tile oracle), and T = (I+A)^-1
 *     is built by plain forward substitution.  Any chunk size C >= 1 is
 *     accepted; C = 1 and C = L are the two degenerate cuts.
 *
 * Layouts (all row-major, tokens packed sequence after sequence):
 *   q, k  [Ttot][H][dk]          v, o  [Ttot][HV][dv]
 *   g     [Ttot][HV]  (gate_mode 0, GDN)  or  [Ttot][HV][dk]  (gate_mode 1, KDA)
 *   beta  [Ttot][HV]             h0, hT [n_seqs][HV][dk][dv]   (h0 may be NULL)
 *   cu_seqlens [n_seqs + 1], nondecreasing, cu_seqlens[0] = 0, last = Ttot.
 * Return value: 0 on success, 1 on a malformed argument (nothing written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int check_common(const int64_t *cu, int n_seqs, int H, int HV, int dk,
                        int dv, int gate_mode) {
  if (!cu || n_seqs < 0 || H <= 0 || HV <= 0 || dk <= 0 || dv <= 0) return 1;
  if (HV % H != 0) return 1;
  if (gate_mode != 0 && gate_mode != 1) return 1;
  if (cu[0] != 0) return 1;
  for (int n = 0; n < n_seqs; n++)
    if (cu[n + 1] < cu[n]) return 1;
  return 0;
}

int gdn_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void gdn_oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * The token walk: the recurrence as stated above, one token at a time.
 */
int gdn_oracle_token_serial(const double *q, const double *k, const double *v,
                            const double *g, const double *beta,
                            const double *h0, double *o, double *hT,
                            const int64_t *cu, int n_seqs, int H, int HV,
                            int dk, int dv, double scale, int gate_mode) {
  if (check_common(cu, n_seqs, H, HV, dk, dv, gate_mode)) return 1;
  if (!q || !k || !v || !g || !beta || !o) return 1;
  const int group = HV / H;
  int failed = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int n = 0; n < n_seqs; n++) {
    for (int hv = 0; hv < HV; hv++) {
      const int hq = hv / group;
      double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
      double *u = (double *)malloc(sizeof(double) * (size_t)dv);
      double *acc = (double *)malloc(sizeof(double) * (size_t)dv);
      double *a = (double *)malloc(sizeof(double) * (size_t)dk);
      if (!S || !u || !acc || !a) {
#pragma omp atomic write
        failed = 1;
        free(S); free(u); free(acc); free(a);
        continue;
      }
      if (h0) {
        memcpy(S, h0 + ((size_t)n * HV + hv) * dk * dv,
               sizeof(double) * (size_t)dk * dv);
      } else {
        memset(S, 0, sizeof(double) * (size_t)dk * dv);
      }
      for (int64_t t = cu[n]; t < cu[n + 1]; t++) {
        const double *kt = k + ((size_t)t * H + hq) * dk;
        const double *qt = q + ((size_t)t * H + hq) * dk;
        const double *vt = v + ((size_t)t * HV + hv) * dv;
        const double bt = beta[(size_t)t * HV + hv];
        /* decay factors a_c = exp(g) */
        if (gate_mode == 0) {
          const double ai = exp(g[(size_t)t * HV + hv]);
          for (int c = 0; c < dk; c++) a[c] = ai;
        } else {
          const double *gt = g + ((size_t)t * HV + hv) * dk;
          for (int c = 0; c < dk; c++) a[c] = exp(gt[c]);
        }
        /* S = diag(a) S */
        for (int c = 0; c < dk; c++)
          for (int j = 0; j < dv; j++) S[(size_t)c * dv + j] *= a[c];
        /* u = v - S^T k */
        for (int j = 0; j < dv; j++) acc[j] = 0.0;
        for (int c = 0; c < dk; c++) {
          const double kc = kt[c];
          const double *Sr = S + (size_t)c * dv;
          for (int j = 0; j < dv; j++) acc[j] += Sr[j] * kc;
        }
        for (int j = 0; j < dv; j++) u[j] = vt[j] - acc[j];
        /* S += beta k u^T */
        for (int c = 0; c < dk; c++) {
          const double f = bt * kt[c];
          double *Sr = S + (size_t)c * dv;
          for (int j = 0; j < dv; j++) Sr[j] += f * u[j];
        }
        /* o = scale S^T q */
        for (int j = 0; j < dv; j++) acc[j] = 0.0;
        for (int c = 0; c < dk; c++) {
          const double qc = qt[c];
          const double *Sr = S + (size_t)c * dv;
          for (int j = 0; j < dv; j++) acc[j] += Sr[j] * qc;
        }
        for (int j = 0; j < dv; j++)
          o[((size_t)t * HV + hv) * dv + j] = scale * acc[j];
      }
      if (hT) {
        memcpy(hT + ((size_t)n * HV + hv) * dk * dv, S,
               sizeof(double) * (size_t)dk * dv);
      }
      free(S); free(u); free(acc); free(a);
    }
  }
  return failed;
}

/*
 * The chunked walk (the WY form).  For one chunk of L rows r, s = 0..L-1 and
 * the state S at its start:
 *
 *   b_r       = sum_{i<=r} g_i                  cumulative log-gate (per channel
 *                                               for KDA)
 *   D_rs(c)   = exp(b_r(c) - b_s(c)), s <= r    pairwise decay, formed directly
 *   A_rs      = beta_r sum_c k_r(c) k_s(c) D_rs(c)          for s <  r, else 0
 *   Aqk_rs    = scale  sum_c q_r(c) k_s(c) D_rs(c)          for s <= r, else 0
 *   T         = (I + A)^-1                      forward substitution
 *   Kg_r      = k_r * exp(b_r)                  gated keys (K-tilde)
 *   W         = T diag(beta) Kg                 C x dk
 *   U         = T diag(beta) V                  C x dv
 *   Vn        = U - W S                         new values
 *   Qg_r      = scale q_r * exp(b_r)            gated queries (GQ)
 *   O         = Qg S + Aqk Vn
 *   Kt_s      = k_s * exp(b_L - b_s)            keys carried to the chunk end
 *   S        <- diag(exp(b_L)) S + Kt^T Vn      (dec = exp(b_L))
 *
 * b_L is the cumulative gate at the chunk's last row.
 */
int gdn_oracle_chunked(const double *q, const double *k, const double *v,
                       const double *g, const double *beta, const double *h0,
                       double *o, double *hT, const int64_t *cu_seqlens,
                       int n_seqs, int H, int HV, int dk, int dv, double scale,
                       int gate_mode, int chunk) {
  if (check_common(cu_seqlens, n_seqs, H, HV, dk, dv, gate_mode)) return 1;
  if (!q || !k || !v || !g || !beta || !o || chunk < 1) return 1;
  const int group = HV / H;
  const int C = chunk;
  const int gw = (gate_mode == 0) ? 1 : dk; /* gate width per token */
  int failed = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int n = 0; n < n_seqs; n++) {
    for (int hv = 0; hv < HV; hv++) {
      const int hq = hv / group;
      const size_t SS = (size_t)dk * dv;
      double *S = (double *)malloc(sizeof(double) * SS);
      double *b = (double *)malloc(sizeof(double) * (size_t)C * gw);
      double *A = (double *)malloc(sizeof(double) * (size_t)C * C);
      double *Aqk = (double *)malloc(sizeof(double) * (size_t)C * C);
      double *T = (double *)malloc(sizeof(double) * (size_t)C * C);
      double *W = (double *)malloc(sizeof(double) * (size_t)C * dk);
      double *U = (double *)malloc(sizeof(double) * (size_t)C * dv);
      double *Vn = (double *)malloc(sizeof(double) * (size_t)C * dv);
      double *X = (double *)malloc(sizeof(double) * (size_t)C * dk);
      double *Snew = (double *)malloc(sizeof(double) * SS);
      if (!S || !b || !A || !Aqk || !T || !W || !U || !Vn || !X || !Snew) {
#pragma omp atomic write
        failed = 1;
        free(S); free(b); free(A); free(Aqk); free(T); free(W); free(U);
        free(Vn); free(X); free(Snew);
        continue;
      }
      if (h0) memcpy(S, h0 + ((size_t)n * HV + hv) * SS, sizeof(double) * SS);
      else memset(S, 0, sizeof(double) * SS);

      for (int64_t t0 = cu_seqlens[n]; t0 < cu_seqlens[n + 1]; t0 += C) {
        int L = C;
        if (cu_seqlens[n + 1] - t0 < C) L = (int)(cu_seqlens[n + 1] - t0);
#define QR(r) (q + ((size_t)(t0 + (r)) * H + hq) * dk)
#define KR(r) (k + ((size_t)(t0 + (r)) * H + hq) * dk)
#define VR(r) (v + ((size_t)(t0 + (r)) * HV + hv) * dv)
#define BETA(r) (beta[(size_t)(t0 + (r)) * HV + hv])
#define GR(r, c) (gate_mode == 0 ? g[(size_t)(t0 + (r)) * HV + hv] \
                                 : g[((size_t)(t0 + (r)) * HV + hv) * dk + (c)])
#define BC(r, c) (b[(size_t)(r) * gw + (gate_mode == 0 ? 0 : (c))])
        /* cumulative log-gates */
        for (int c = 0; c < gw; c++) {
          double run = 0.0;
          for (int r = 0; r < L; r++) {
            run += GR(r, c);
            b[(size_t)r * gw + c] = run;
          }
        }
        /* A (strictly lower) and Aqk (lower incl. diagonal), decays per pair */
        for (int r = 0; r < L; r++) {
          for (int s = 0; s < L; s++) {
            double a_rs = 0.0, p_rs = 0.0;
            if (s <= r) {
              const double *kr = KR(r), *ks = KR(s), *qr = QR(r);
              for (int c = 0; c < dk; c++) {
                const double d = exp(BC(r, c) - BC(s, c));
                a_rs += kr[c] * ks[c] * d;
                p_rs += qr[c] * ks[c] * d;
              }
            }
            A[(size_t)r * C + s] = (s < r) ? BETA(r) * a_rs : 0.0;
            Aqk[(size_t)r * C + s] = (s <= r) ? scale * p_rs : 0.0;
          }
        }
        /* T = (I + A)^-1 by forward substitution, one column at a time:
           T[r][j] = delta_rj - sum_{s<r} A[r][s] T[s][j] */
        for (int j = 0; j < L; j++) {
          for (int r = 0; r < L; r++) {
            double x = (r == j) ? 1.0 : 0.0;
            for (int s = 0; s < r; s++) x -= A[(size_t)r * C + s] * T[(size_t)s * C + j];
            T[(size_t)r * C + j] = x;
          }
        }
        /* W = T diag(beta) Kg  and  U = T diag(beta) V */
        for (int r = 0; r < L; r++) {
          for (int c = 0; c < dk; c++) W[(size_t)r * dk + c] = 0.0;
          for (int j = 0; j < dv; j++) U[(size_t)r * dv + j] = 0.0;
          for (int s = 0; s <= r; s++) {
            const double tb = T[(size_t)r * C + s] * BETA(s);
            const double *ks = KR(s), *vs = VR(s);
            for (int c = 0; c < dk; c++)
              W[(size_t)r * dk + c] += tb * ks[c] * exp(BC(s, c));
            for (int j = 0; j < dv; j++) U[(size_t)r * dv + j] += tb * vs[j];
          }
        }
        /* Vn = U - W S */
        for (int r = 0; r < L; r++) {
          for (int j = 0; j < dv; j++) Vn[(size_t)r * dv + j] = U[(size_t)r * dv + j];
          for (int c = 0; c < dk; c++) {
            const double w = W[(size_t)r * dk + c];
            const double *Sr = S + (size_t)c * dv;
            for (int j = 0; j < dv; j++) Vn[(size_t)r * dv + j] -= w * Sr[j];
          }
        }
        /* O = Qg S + Aqk Vn */
        for (int r = 0; r < L; r++) {
          double *orow = o + ((size_t)(t0 + r) * HV + hv) * dv;
          const double *qr = QR(r);
          for (int j = 0; j < dv; j++) orow[j] = 0.0;
          for (int c = 0; c < dk; c++) {
            const double qg = scale * qr[c] * exp(BC(r, c));
            const double *Sr = S + (size_t)c * dv;
            for (int j = 0; j < dv; j++) orow[j] += qg * Sr[j];
          }
          for (int s = 0; s <= r; s++) {
            const double p = Aqk[(size_t)r * C + s];
            for (int j = 0; j < dv; j++) orow[j] += p * Vn[(size_t)s * dv + j];
          }
        }
        /* S <- diag(exp(b_L)) S + Kt^T Vn */
        for (int c = 0; c < dk; c++) {
          const double dec = exp(BC(L - 1, c));
          for (int j = 0; j < dv; j++) Snew[(size_t)c * dv + j] = dec * S[(size_t)c * dv + j];
        }
        for (int s = 0; s < L; s++) {
          const double *ks = KR(s);
          for (int c = 0; c < dk; c++) X[(size_t)s * dk + c] = ks[c] * exp(BC(L - 1, c) - BC(s, c));
        }
        for (int s = 0; s < L; s++) {
          for (int c = 0; c < dk; c++) {
            const double kt = X[(size_t)s * dk + c];
            double *Sr = Snew + (size_t)c * dv;
            const double *vn = Vn + (size_t)s * dv;
            for (int j = 0; j < dv; j++) Sr[j] += kt * vn[j];
          }
        }
        memcpy(S, Snew, sizeof(double) * SS);
#undef QR
#undef KR
#undef VR
#undef BETA
#undef GR
#undef BC
      }
      if (hT) memcpy(hT + ((size_t)n * HV + hv) * SS, S, sizeof(double) * SS);
      free(S); free(b); free(A); free(Aqk); free(T); free(W); free(U);
      free(Vn); free(X); free(Snew);
    }
  }
  return failed;
}
