/*
 * dualkv_oracle.c -- fp64 CPU oracle for DualKV shared-prompt attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the timed
 * CPU baseline of the benchmark may load this library.  The CUDA product path
 * shares no code with it and never calls it.
 *
 * What it computes (DualKV: Shared-Prompt Flash Attention for Efficient RL
 * Training with Large Rollouts and Long Contexts, abstract): DualKV is stated
 * to be mathematically identical to standard attention.  So this oracle is
 * the plain definition, written out with no blocking, fusion or reordering:
 *
 *   1. Unpack the packed micro-batch [prompt P][seg 0 R_0]...[seg N-1] into N
 *      replicated sequences X_n = prompt rows ++ segment-n rows, positions
 *      0..P+R_n-1 (the N(P+R) replicated tokens of the abstract).
 *   2. Per replica, per q-head h (kv-head g = h / (Hq/Hkv)), per row i:
 *      allowed keys A_i = { j <= i : window <= 0 or i - j < window },
 *      S_ij = scale * q_i . k_j,  m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i),
 *      P_ij = exp(S_ij - m_i) / l_i,  O_i = sum_j P_ij v_j,  LSE_i = m_i + ln l_i.
 *   3. Packed forward: response rows from their replica, prompt rows from
 *      replica 0.  Prompt rows of every replica are compared with replica 0
 *      (causal masking makes them identical: the abstract's invariance).
 *   4. Replica upstream gradient: response rows get the packed dO.  Prompt rows
 *      get the packed dO in replica 0 and zero elsewhere (dout_mode 0), or
 *      dO / N in every replica (dout_mode 1).  Gradients are linear in dO, so
 *      both splits give the same folded result.
 *   5. Analytic backward per replica: Delta_i = dO_i . O_i,
 *      dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - Delta_i),
 *      dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 *      dV_j = sum_i P_ij dO_i, with dK, dV summed over the q-heads of a group.
 *   6. Fold: packed prompt rows of dQ/dK/dV = sum over replicas n = 0..N-1 in
 *      that order; response rows are their replica's rows.
 *
 * Layouts (packed, contiguous): q, out, dout, dq [T, Hq, D]; k, v, dk, dv
 * [T, Hkv, D]; lse [Hq, T]; T = P + off[N].  Every array is fp64.  Only the
 * q-heads in [h_lo, h_hi) and their kv-heads are read or written; [h_lo, h_hi)
 * must cover whole GQA groups.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ENOMEM 2

typedef struct {
  int P, N;
  const int32_t *off;
  int Hq, Hkv, D;
  double scale;
  int window;
} orc_layout;

/* packed row of replicated position p in sequence n */
static int64_t rep_to_packed(const orc_layout *L, int n, int p) {
  return p < L->P ? (int64_t)p : (int64_t)L->P + L->off[n] + (p - L->P);
}

static int seq_len(const orc_layout *L, int n) { return L->P + (L->off[n + 1] - L->off[n]); }

/* first allowed key position of query position i (keys i-window+1 .. i) */
static int first_key(const orc_layout *L, int i) {
  if (L->window <= 0) return 0;
  int j = i - L->window + 1;
  return j < 0 ? 0 : j;
}

static double dot(const double *a, const double *b, int D) {
  double s = 0.0;
  for (int d = 0; d < D; ++d) s += a[d] * b[d];
  return s;
}

static int check_layout(const orc_layout *L, int h_lo, int h_hi) {
  if (L->P < 0 || L->N < 1 || L->Hq < 1 || L->Hkv < 1 || L->D < 1) return ORC_EINVAL;
  if (L->Hq % L->Hkv) return ORC_EINVAL;
  if (L->off[0] != 0) return ORC_EINVAL;
  for (int n = 0; n < L->N; ++n)
    if (L->off[n + 1] < L->off[n]) return ORC_EINVAL;
  int gs = L->Hq / L->Hkv;
  if (h_lo < 0 || h_hi > L->Hq || h_lo >= h_hi || h_lo % gs || h_hi % gs) return ORC_EINVAL;
  return ORC_OK;
}

/*
 * Forward of one query row (step 2): query at replicated position i of
 * sequence n, q-head h.  Writes m, l, the row's O (D values) and returns LSE.
 */
static double forward_row(const orc_layout *L, int n, int h, int i, const double *q, const double *k,
                          const double *v, double *o_row, double *m_out, double *l_out, double *sbuf) {
  const int D = L->D, Hq = L->Hq, Hkv = L->Hkv;
  const int g = h / (Hq / Hkv);
  const double *qi = q + (rep_to_packed(L, n, i) * Hq + h) * D;
  const int j0 = first_key(L, i);
  double m = -INFINITY;
  for (int j = j0; j <= i; ++j) {
    const double *kj = k + (rep_to_packed(L, n, j) * Hkv + g) * D;
    double s = L->scale * dot(qi, kj, D);
    sbuf[j - j0] = s;
    if (s > m) m = s;
  }
  double l = 0.0;
  for (int j = j0; j <= i; ++j) l += exp(sbuf[j - j0] - m);
  for (int d = 0; d < D; ++d) o_row[d] = 0.0;
  for (int j = j0; j <= i; ++j) {
    const double p = exp(sbuf[j - j0] - m) / l;
    const double *vj = v + (rep_to_packed(L, n, j) * Hkv + g) * D;
    for (int d = 0; d < D; ++d) o_row[d] += p * vj[d];
  }
  *m_out = m;
  *l_out = l;
  return m + log(l);
}

/* replica upstream gradient of row at replicated position i of sequence n (step 4) */
static void replica_dout(const orc_layout *L, int n, int h, int i, const double *dout, int dout_mode,
                         double *dst) {
  const int D = L->D;
  const double *src = dout + (rep_to_packed(L, n, i) * L->Hq + h) * D;
  if (i >= L->P) {
    for (int d = 0; d < D; ++d) dst[d] = src[d];
  } else if (dout_mode == 1) {
    for (int d = 0; d < D; ++d) dst[d] = src[d] / (double)L->N;
  } else {
    for (int d = 0; d < D; ++d) dst[d] = (n == 0) ? src[d] : 0.0;
  }
}

/*
 * Full oracle: forward (steps 1-3), backward (4-5) and fold (6).
 * Any of out/lse/dq/dk/dv may be NULL (dout may be NULL when dq, dk, dv are).
 * *prompt_invariant is set to 1 when every replica's prompt O and LSE equal
 * replica 0's bit for bit, else 0.
 */
int oracle_dualkv(int P, int N, const int32_t *off, int Hq, int Hkv, int D, double scale, int window,
                  int h_lo, int h_hi, const double *q, const double *k, const double *v,
                  const double *dout, int dout_mode, double *out, double *lse, double *dq, double *dk,
                  double *dv, int *prompt_invariant) {
  orc_layout L = {P, N, off, Hq, Hkv, D, scale, window};
  int rc = check_layout(&L, h_lo, h_hi);
  if (rc) return rc;
  const int gs = Hq / Hkv;
  const int g_lo = h_lo / gs, g_hi = h_hi / gs, ng = g_hi - g_lo;
  const int64_t T = (int64_t)P + off[N];
  const int want_bwd = (dq || dk || dv) && dout;
  int Lmax = P;
  for (int n = 0; n < N; ++n)
    if (seq_len(&L, n) > Lmax) Lmax = seq_len(&L, n);

  /* per-replica prompt results, folded afterwards in replica order */
  const size_t pro_o = (size_t)N * ng * gs * (size_t)P * D;
  const size_t pro_l = (size_t)N * ng * gs * (size_t)P;
  const size_t pro_kv = (size_t)N * ng * (size_t)P * D;
  double *rep_o = (double *)calloc(pro_o ? pro_o : 1, sizeof(double));
  double *rep_lse = (double *)calloc(pro_l ? pro_l : 1, sizeof(double));
  double *rep_dq = want_bwd ? (double *)calloc(pro_o ? pro_o : 1, sizeof(double)) : NULL;
  double *rep_dk = want_bwd ? (double *)calloc(pro_kv ? pro_kv : 1, sizeof(double)) : NULL;
  double *rep_dv = want_bwd ? (double *)calloc(pro_kv ? pro_kv : 1, sizeof(double)) : NULL;
  if (!rep_o || !rep_lse || (want_bwd && (!rep_dq || !rep_dk || !rep_dv))) {
    free(rep_o); free(rep_lse); free(rep_dq); free(rep_dk); free(rep_dv);
    return ORC_ENOMEM;
  }
  int fail = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int task = 0; task < N * ng; ++task) {
    const int n = task / ng, gi = task % ng, g = g_lo + gi;
    const int Ln = seq_len(&L, n);
    /* replica-local state for the gs q-heads of group g */
    double *O = (double *)malloc(sizeof(double) * (size_t)gs * Ln * D + 1);
    double *M = (double *)malloc(sizeof(double) * (size_t)gs * Ln + 1);
    double *Ls = (double *)malloc(sizeof(double) * (size_t)gs * Ln + 1);
    double *sbuf = (double *)malloc(sizeof(double) * (size_t)Lmax + 1);
    double *dKr = want_bwd ? (double *)calloc((size_t)Ln * D + 1, sizeof(double)) : NULL;
    double *dVr = want_bwd ? (double *)calloc((size_t)Ln * D + 1, sizeof(double)) : NULL;
    double *dQr = want_bwd ? (double *)calloc((size_t)gs * Ln * D + 1, sizeof(double)) : NULL;
    double *doi = (double *)malloc(sizeof(double) * (size_t)D + 1);
    if (!O || !M || !Ls || !sbuf || !doi || (want_bwd && (!dKr || !dVr || !dQr))) {
#pragma omp atomic write
      fail = 1;
      free(O); free(M); free(Ls); free(sbuf); free(dKr); free(dVr); free(dQr); free(doi);
      continue;
    }
    for (int hh = 0; hh < gs; ++hh) {
      const int h = g * gs + hh;
      for (int i = 0; i < Ln; ++i) {
        double lse_i = forward_row(&L, n, h, i, q, k, v, O + ((size_t)hh * Ln + i) * D, &M[hh * Ln + i],
                                   &Ls[hh * Ln + i], sbuf);
        if (i < P) {
          const size_t idx = (((size_t)n * ng + gi) * gs + hh) * P + i;
          rep_lse[idx] = lse_i;
          memcpy(rep_o + idx * D, O + ((size_t)hh * Ln + i) * D, sizeof(double) * D);
        } else {
          const int64_t row = rep_to_packed(&L, n, i);
          if (out) memcpy(out + (row * Hq + h) * D, O + ((size_t)hh * Ln + i) * D, sizeof(double) * D);
          if (lse) lse[(int64_t)h * T + row] = lse_i;
        }
      }
    }
    if (want_bwd) {
      for (int hh = 0; hh < gs; ++hh) {
        const int h = g * gs + hh;
        for (int i = 0; i < Ln; ++i) {
          replica_dout(&L, n, h, i, dout, dout_mode, doi);
          const double *Oi = O + ((size_t)hh * Ln + i) * D;
          const double delta = dot(doi, Oi, D);
          const double m = M[hh * Ln + i], l = Ls[hh * Ln + i];
          const double *qi = q + (rep_to_packed(&L, n, i) * Hq + h) * D;
          double *dqi = dQr + ((size_t)hh * Ln + i) * D;
          for (int j = first_key(&L, i); j <= i; ++j) {
            const int64_t rj = rep_to_packed(&L, n, j);
            const double *kj = k + (rj * Hkv + g) * D;
            const double *vj = v + (rj * Hkv + g) * D;
            const double s = scale * dot(qi, kj, D);
            const double p = exp(s - m) / l;
            const double dp = dot(doi, vj, D);
            const double ds = p * (dp - delta);
            for (int d = 0; d < D; ++d) {
              dqi[d] += scale * ds * kj[d];
              dKr[(size_t)j * D + d] += scale * ds * qi[d];
              dVr[(size_t)j * D + d] += p * doi[d];
            }
          }
        }
      }
      /* response rows are unique to this replica; prompt rows are kept for the fold */
      for (int i = 0; i < Ln; ++i) {
        if (i < P) {
          const size_t kvidx = (((size_t)n * ng + gi) * P + i) * D;
          memcpy(rep_dk + kvidx, dKr + (size_t)i * D, sizeof(double) * D);
          memcpy(rep_dv + kvidx, dVr + (size_t)i * D, sizeof(double) * D);
          for (int hh = 0; hh < gs; ++hh) {
            const size_t idx = ((((size_t)n * ng + gi) * gs + hh) * P + i) * D;
            memcpy(rep_dq + idx, dQr + ((size_t)hh * Ln + i) * D, sizeof(double) * D);
          }
        } else {
          const int64_t row = rep_to_packed(&L, n, i);
          if (dk) memcpy(dk + (row * Hkv + g) * D, dKr + (size_t)i * D, sizeof(double) * D);
          if (dv) memcpy(dv + (row * Hkv + g) * D, dVr + (size_t)i * D, sizeof(double) * D);
          for (int hh = 0; hh < gs; ++hh)
            if (dq) memcpy(dq + (row * Hq + g * gs + hh) * D, dQr + ((size_t)hh * Ln + i) * D, sizeof(double) * D);
        }
      }
    }
    free(O); free(M); free(Ls); free(sbuf); free(dKr); free(dVr); free(dQr); free(doi);
  }

  int invariant = 1;
  if (!fail) {
    /* step 3: prompt rows from replica 0; every replica must agree with it */
    for (int gi = 0; gi < ng; ++gi)
      for (int hh = 0; hh < gs; ++hh) {
        const int h = (g_lo + gi) * gs + hh;
        for (int i = 0; i < P; ++i) {
          const size_t idx0 = (((size_t)0 * ng + gi) * gs + hh) * P + i;
          for (int n = 1; n < N; ++n) {
            const size_t idxn = (((size_t)n * ng + gi) * gs + hh) * P + i;
            if (rep_lse[idxn] != rep_lse[idx0] ||
                memcmp(rep_o + idxn * D, rep_o + idx0 * D, sizeof(double) * D) != 0)
              invariant = 0;
          }
          if (out) memcpy(out + ((int64_t)i * Hq + h) * D, rep_o + idx0 * D, sizeof(double) * D);
          if (lse) lse[(int64_t)h * T + i] = rep_lse[idx0];
        }
      }
    /* step 6: fold prompt gradients over replicas n = 0..N-1 in order */
    if (want_bwd) {
      for (int gi = 0; gi < ng; ++gi) {
        const int g = g_lo + gi;
        for (int i = 0; i < P; ++i)
          for (int d = 0; d < D; ++d) {
            double sk = 0.0, sv = 0.0;
            for (int n = 0; n < N; ++n) {
              const size_t kvidx = (((size_t)n * ng + gi) * P + i) * D + d;
              sk += rep_dk[kvidx];
              sv += rep_dv[kvidx];
            }
            if (dk) dk[((int64_t)i * Hkv + g) * D + d] = sk;
            if (dv) dv[((int64_t)i * Hkv + g) * D + d] = sv;
          }
        for (int hh = 0; hh < gs; ++hh)
          for (int i = 0; i < P; ++i)
            for (int d = 0; d < D; ++d) {
              double s = 0.0;
              for (int n = 0; n < N; ++n) s += rep_dq[((((size_t)n * ng + gi) * gs + hh) * P + i) * D + d];
              if (dq) dq[((int64_t)i * Hq + g * gs + hh) * D + d] = s;
            }
      }
    }
  }
  if (prompt_invariant) *prompt_invariant = invariant;
  free(rep_o); free(rep_lse); free(rep_dq); free(rep_dk); free(rep_dv);
  return fail ? ORC_ENOMEM : ORC_OK;
}

/* replica and replicated position that a packed query row is read from (step 3) */
static void packed_to_rep(const orc_layout *L, int64_t row, int *n, int *pos) {
  if (row < L->P) {
    *n = 0;
    *pos = (int)row;
    return;
  }
  const int64_t r = row - L->P;
  /* segment s holds r when off[s] <= r < off[s+1]; empty segments are skipped */
  int s = 0;
  while (L->off[s + 1] <= r) ++s;
  *n = s;
  *pos = L->P + (int)(r - L->off[s]);
}

/*
 * Sampled query rows: O, LSE and dQ of the packed rows listed in `rows`, for
 * q-head h, by the same definition as oracle_dualkv (steps 2-6).  A prompt
 * row's dQ is the fold over replicas; with dout_mode 0 only replica 0 carries
 * its upstream gradient, with dout_mode 1 each replica carries dO/N.
 * Outputs are [nrows, D] (o_rows, dq_rows) and [nrows] (lse_rows); dq_rows
 * and dout may be NULL.
 */
int oracle_query_rows(int P, int N, const int32_t *off, int Hq, int Hkv, int D, double scale, int window,
                      int h, const int64_t *rows, int nrows, const double *q, const double *k,
                      const double *v, const double *dout, int dout_mode, double *o_rows, double *lse_rows,
                      double *dq_rows) {
  orc_layout L = {P, N, off, Hq, Hkv, D, scale, window};
  const int gs = Hq / Hkv;
  int rc = check_layout(&L, (h / gs) * gs, (h / gs) * gs + gs);
  if (rc) return rc;
  const int64_t T = (int64_t)P + off[N];
  int Lmax = P;
  for (int n = 0; n < N; ++n)
    if (seq_len(&L, n) > Lmax) Lmax = seq_len(&L, n);
  for (int r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= T) return ORC_EINVAL;
  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    double *sbuf = (double *)malloc(sizeof(double) * (size_t)Lmax + 1);
    double *oi = (double *)malloc(sizeof(double) * (size_t)D + 1);
    double *doi = (double *)malloc(sizeof(double) * (size_t)D + 1);
    if (!sbuf || !oi || !doi) {
#pragma omp atomic write
      fail = 1;
      free(sbuf); free(oi); free(doi);
      continue;
    }
    int n0, pos;
    packed_to_rep(&L, rows[r], &n0, &pos);
    double m, l;
    double lse_i = forward_row(&L, n0, h, pos, q, k, v, oi, &m, &l, sbuf);
    memcpy(o_rows + (size_t)r * D, oi, sizeof(double) * D);
    lse_rows[r] = lse_i;
    if (dq_rows && dout) {
      double *dqi = dq_rows + (size_t)r * D;
      for (int d = 0; d < D; ++d) dqi[d] = 0.0;
      const int g = h / gs;
      /* a prompt row appears in every replica; a response row in its own */
      const int nfirst = pos < P ? 0 : n0, nlast = pos < P ? N - 1 : n0;
      for (int n = nfirst; n <= nlast; ++n) {
        double mn, ln;
        forward_row(&L, n, h, pos, q, k, v, oi, &mn, &ln, sbuf);
        replica_dout(&L, n, h, pos, dout, dout_mode, doi);
        const double delta = dot(doi, oi, D);
        const double *qi = q + (rep_to_packed(&L, n, pos) * Hq + h) * D;
        for (int j = first_key(&L, pos); j <= pos; ++j) {
          const int64_t rj = rep_to_packed(&L, n, j);
          const double *kj = k + (rj * Hkv + g) * D;
          const double *vj = v + (rj * Hkv + g) * D;
          const double p = exp(scale * dot(qi, kj, D) - mn) / ln;
          const double ds = p * (dot(doi, vj, D) - delta);
          for (int d = 0; d < D; ++d) dqi[d] += scale * ds * kj[d];
        }
      }
    }
    free(sbuf); free(oi); free(doi);
  }
  return fail ? ORC_ENOMEM : ORC_OK;
}

/*
 * Sampled key rows: dK and dV of the packed key rows listed in `keys`, for
 * kv-head g, by the definition (steps 2-6): every replica that holds the key,
 * every q-head of the group, every query whose allowed set contains the key.
 * Each such query's m, l and O come from its own full forward row.  Partial
 * sums are folded over replicas n = 0..N-1 in order.  Outputs [nkeys, D].
 */
int oracle_key_rows(int P, int N, const int32_t *off, int Hq, int Hkv, int D, double scale, int window,
                    int g, const int64_t *keys, int nkeys, const double *q, const double *k, const double *v,
                    const double *dout, int dout_mode, double *dk_rows, double *dv_rows) {
  orc_layout L = {P, N, off, Hq, Hkv, D, scale, window};
  const int gs = Hq / Hkv;
  int rc = check_layout(&L, g * gs, g * gs + gs);
  if (rc) return rc;
  const int64_t T = (int64_t)P + off[N];
  for (int r = 0; r < nkeys; ++r)
    if (keys[r] < 0 || keys[r] >= T) return ORC_EINVAL;
  int Lmax = P;
  for (int n = 0; n < N; ++n)
    if (seq_len(&L, n) > Lmax) Lmax = seq_len(&L, n);
  /* partial[n][key][d] for dK and dV; folded in replica order below */
  double *pk = (double *)calloc((size_t)N * nkeys * D + 1, sizeof(double));
  double *pv = (double *)calloc((size_t)N * nkeys * D + 1, sizeof(double));
  if (!pk || !pv) {
    free(pk); free(pv);
    return ORC_ENOMEM;
  }
  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int n = 0; n < N; ++n) {
    const int Ln = seq_len(&L, n);
    double *sbuf = (double *)malloc(sizeof(double) * (size_t)Lmax + 1);
    double *oi = (double *)malloc(sizeof(double) * (size_t)D + 1);
    double *doi = (double *)malloc(sizeof(double) * (size_t)D + 1);
    int *kpos = (int *)malloc(sizeof(int) * (size_t)nkeys + 1);
    if (!sbuf || !oi || !doi || !kpos) {
#pragma omp atomic write
      fail = 1;
      free(sbuf); free(oi); free(doi); free(kpos);
      continue;
    }
    /* replicated position of each sampled key in this replica, or -1 */
    int minpos = Ln;
    for (int r = 0; r < nkeys; ++r) {
      kpos[r] = -1;
      for (int p = 0; p < Ln; ++p)
        if (rep_to_packed(&L, n, p) == keys[r]) {
          kpos[r] = p;
          break;
        }
      if (kpos[r] >= 0 && kpos[r] < minpos) minpos = kpos[r];
    }
    for (int hh = 0; hh < gs; ++hh) {
      const int h = g * gs + hh;
      for (int i = minpos; i < Ln; ++i) {
        const int j0 = first_key(&L, i);
        int sees = 0;
        for (int r = 0; r < nkeys; ++r)
          if (kpos[r] >= j0 && kpos[r] <= i) sees = 1;
        if (!sees) continue;
        /* Under the replica-0 split a prompt row of replica n >= 1 carries a zero
           upstream gradient, so its dV term p * 0 and its dK term scale * p * (0 - 0) * q
           are zeros: adding them changes no sum, and the row is skipped. */
        if (dout_mode == 0 && n > 0 && i < P) continue;
        double m, l;
        forward_row(&L, n, h, i, q, k, v, oi, &m, &l, sbuf);
        replica_dout(&L, n, h, i, dout, dout_mode, doi);
        const double delta = dot(doi, oi, D);
        const double *qi = q + (rep_to_packed(&L, n, i) * Hq + h) * D;
        for (int r = 0; r < nkeys; ++r) {
          const int j = kpos[r];
          if (j < j0 || j > i) continue;
          const double *kj = k + (keys[r] * Hkv + g) * D;
          const double *vj = v + (keys[r] * Hkv + g) * D;
          const double p = exp(scale * dot(qi, kj, D) - m) / l;
          const double ds = p * (dot(doi, vj, D) - delta);
          double *pkr = pk + ((size_t)n * nkeys + r) * D;
          double *pvr = pv + ((size_t)n * nkeys + r) * D;
          for (int d = 0; d < D; ++d) {
            pkr[d] += scale * ds * qi[d];
            pvr[d] += p * doi[d];
          }
        }
      }
    }
    free(sbuf); free(oi); free(doi); free(kpos);
  }
  if (!fail)
    for (int r = 0; r < nkeys; ++r)
      for (int d = 0; d < D; ++d) {
        double sk = 0.0, sv = 0.0;
        for (int n = 0; n < N; ++n) {
          sk += pk[((size_t)n * nkeys + r) * D + d];
          sv += pv[((size_t)n * nkeys + r) * D + d];
        }
        dk_rows[(size_t)r * D + d] = sk;
        dv_rows[(size_t)r * D + d] = sv;
      }
  free(pk); free(pv);
  return fail ? ORC_ENOMEM : ORC_OK;
}

/* number of OpenMP threads the oracle runs on */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
