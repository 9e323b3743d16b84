/*
 * planted_walk.c -- NEGATIVE CONTROLS ONLY: deliberately wrong copies of the
 * token walk of gdn_oracle.c, built into a library of their own.
 *
 * TEST INFRASTRUCTURE ONLY.  The oracle's pin tests run their checks against
 * each variant below to show that every plausible mistake in the walk fails
 * at least one pin (the negative control of stratat pull #1296, "The parity
 * discipline").  Nothing else calls this file; gdn_oracle.c does not include
 * it, so the oracle's own walk carries no switch.
 *
 * `planted` selects the mistake (same arguments and layouts as
 * gdn_oracle_token_serial, one extra int):
 *   1  delta taken against the undecayed state (decay applied after the write)
 *   2  output read from the state before the rank-1 write
 *   3  sign of the prediction flipped (u = v + S^T k)
 *   4  beta dropped from the write (S += k u^T)
 *   5  decay applied per value column instead of per key row (KDA)
 *   6  output not scaled
 * Single-threaded; meant for the few-token cases of the pin tests.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static void decay_rows(double *S, const double *a, int dk, int dv) {
  for (int c = 0; c < dk; c++)
    for (int j = 0; j < dv; j++) S[(size_t)c * dv + j] *= a[c];
}

static void decay_columns(double *S, const double *a, int dk, int dv) {
  for (int c = 0; c < dk; c++)
    for (int j = 0; j < dv; j++) S[(size_t)c * dv + j] *= a[j % dk];
}

/* out[j] = sum_c S[c][j] x[c] */
static void read_state(const double *S, const double *x, double *out, int dk, int dv) {
  for (int j = 0; j < dv; j++) out[j] = 0.0;
  for (int c = 0; c < dk; c++)
    for (int j = 0; j < dv; j++) out[j] += S[(size_t)c * dv + j] * x[c];
}

int gdn_planted_token_serial(const double *q, const double *k, const double *v,
                             const double *g, const double *beta,
                             const double *h0, double *o, double *hT,
                             const int64_t *cu, int n_seqs, int H, int HV,
                             int dk, int dv, double scale, int gate_mode,
                             int planted) {
  if (planted < 1 || planted > 6) return 1;
  if (!cu || n_seqs < 0 || H <= 0 || HV <= 0 || HV % H || dk <= 0 || dv <= 0) return 1;
  if (gate_mode != 0 && gate_mode != 1) return 1;
  if (!q || !k || !v || !g || !beta || !o) return 1;
  const int group = HV / H;
  double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
  double *u = (double *)malloc(sizeof(double) * (size_t)dv);
  double *acc = (double *)malloc(sizeof(double) * (size_t)dv);
  double *a = (double *)malloc(sizeof(double) * (size_t)dk);
  if (!S || !u || !acc || !a) {
    free(S); free(u); free(acc); free(a);
    return 1;
  }
  for (int n = 0; n < n_seqs; n++) {
    for (int hv = 0; hv < HV; hv++) {
      const int hq = hv / group;
      if (h0)
        memcpy(S, h0 + ((size_t)n * HV + hv) * dk * dv, sizeof(double) * (size_t)dk * dv);
      else
        memset(S, 0, sizeof(double) * (size_t)dk * dv);
      for (int64_t t = cu[n]; t < cu[n + 1]; t++) {
        const double *kt = k + ((size_t)t * H + hq) * dk;
        const double *qt = q + ((size_t)t * H + hq) * dk;
        const double *vt = v + ((size_t)t * HV + hv) * dv;
        const double bt = beta[(size_t)t * HV + hv];
        double *ot = o + ((size_t)t * HV + hv) * dv;
        for (int c = 0; c < dk; c++)
          a[c] = exp(gate_mode == 0 ? g[(size_t)t * HV + hv] : g[((size_t)t * HV + hv) * dk + c]);
        if (planted == 5) decay_columns(S, a, dk, dv);
        else if (planted != 1) decay_rows(S, a, dk, dv);
        read_state(S, kt, acc, dk, dv);
        for (int j = 0; j < dv; j++) u[j] = planted == 3 ? vt[j] + acc[j] : vt[j] - acc[j];
        if (planted == 2) {
          read_state(S, qt, acc, dk, dv);
          for (int j = 0; j < dv; j++) ot[j] = scale * acc[j];
        }
        const double bw = planted == 4 ? 1.0 : bt;
        for (int c = 0; c < dk; c++)
          for (int j = 0; j < dv; j++) S[(size_t)c * dv + j] += bw * kt[c] * u[j];
        if (planted == 1) decay_rows(S, a, dk, dv);
        if (planted != 2) {
          read_state(S, qt, acc, dk, dv);
          for (int j = 0; j < dv; j++) ot[j] = (planted == 6 ? 1.0 : scale) * acc[j];
        }
      }
      if (hT) memcpy(hT + ((size_t)n * HV + hv) * dk * dv, S, sizeof(double) * (size_t)dk * dv);
    }
  }
  free(S); free(u); free(acc); free(a);
  return 0;
}
