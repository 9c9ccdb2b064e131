/*
 * CPU oracle for the target-side verify and commit of one GatedDeltaNet
 * (GDN) linear-attention layer in MTP speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file.  It shares no code, header
 * or constant with the CUDA library and must never be used as a fallback.
 *
 * What it computes (plain definition, fp64 throughout):
 *   A verify step scores the k+1 rows [pending, d1..dk] of each request in one
 *   pass, and speculative decoding is exact, so the rows must give what k+1
 *   sequential single-token decode steps give
 *   [LightLLM #1330 "Qwen3.5 / Qwen3.5-MoE MTP speculative decoding", Summary
 *    and Test Plan; FreeToken #828 "Speculative decoding: MTP and DFlash",
 *    Design].
 *   The GDN state is only read during the verify; the commit leaves each
 *   request's slot as a+1 decode steps would leave it, where a is the number
 *   of accepted drafts, with the conv window moved on over exactly the
 *   accepted rows [FreeToken #828, Design; FreeToken #844 "MTP drafts for
 *   Qwen3.5 family + Flash-Next", Design / Flash-Next target verify].
 *   The accept length those pages print counts committed tokens, a+1, at most
 *   k+1 [FreeToken #844, End-to-end].
 *
 * One decode step of a GDN layer, as this oracle writes it out.  The pages
 * name the layer but do not print its equations; this is the standard gated
 * delta rule with a width-W causal depthwise conv and SiLU in front of it:
 *   window_t[c] = last W entries of [conv_state[c][0..W-2], x_0[c] .. x_t[c]]
 *   y_t[c]      = SiLU(sum_j conv_w[c][j] * window_t[c][j]),  tap W-1 = newest
 *   q, k        = per-head  y / sqrt(sum y^2 + eps)   (q, k channel blocks)
 *   v           = the v channel block of y
 *   per value head h (q/k head h / (H_v/H_qk)):
 *     alpha = exp(g_t[h]);   S <- alpha * S
 *     u     = beta_t[h] * (v - S k)
 *     S     <- S + u k^T
 *     o_t   = scale * S q
 * which is S_t = alpha S_{t-1} + beta (v - alpha S_{t-1} k) k^T,  o_t = scale S_t q.
 *
 * Layouts (row-major, caller-owned):
 *   x [B][R][C], g/beta [B][R][H_v], conv_w [C][W], conv_state [P][C][W-1],
 *   ssm_state [P][H_v][d_v][d_k], o [B][R][H_v][d_v],
 *   snap_S [B][R][H_v][d_v][d_k], snap_cs [B][R][C][W-1],
 *   C = 2*H_qk*d_k + H_v*d_v, channel order [q heads | k heads | v heads].
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BAD_SLOT 1
#define ORACLE_BAD_NROWS 2
#define ORACLE_BAD_ACCEPT 4

/* Deliberate mistakes, switched on only by the tests that show each pin
 * catches one.  0 = the oracle as specified. */
enum {
  MUT_NONE = 0,
  MUT_CONV_COMMIT_EARLY = 1,   /* committed conv window one column early      */
  MUT_COMMIT_A_ROWS = 2,       /* commit after a rows instead of a+1          */
  MUT_VERIFY_WRITES_LIVE = 3,  /* verify-only writes the live slot state      */
  MUT_TAPS_REVERSED = 4,       /* tap 0 hits the newest row                   */
  MUT_GQA_MODULO = 5,          /* value head h uses q/k head h % H_qk         */
  MUT_O_BEFORE_UPDATE = 6,     /* o from the state before the rank-1 update   */
  MUT_NO_K_NORM = 7,           /* k not L2-normalised                         */
  MUT_NO_SCALE = 8,            /* o without the scale                         */
  MUT_DECAY_AFTER = 9,         /* decay applied after the delta update        */
  MUT_NO_BETA = 10,            /* write strength ignored                      */
  MUT_NO_SILU = 11             /* conv output not passed through SiLU         */
};

typedef struct {
  int B, R, H_qk, H_v, d_k, d_v, W, P;
  double scale;  /* o = scale * S q */
  double l2_eps; /* q, k <- y / sqrt(sum y^2 + l2_eps) */
} oracle_dims;

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Gating of a Qwen3.5-style GDN layer from its raw projections, per row and
 * value head h:  g = -exp(A_log[h]) * softplus(a),  beta = sigmoid(b), with
 * softplus(a) = log(1 + e^a) and sigmoid(b) = 1 / (1 + e^-b), written in the
 * overflow-free forms max(a, 0) + log1p(e^-|a|) and e^min(b,0) / (1 + e^-|b|).
 * a, b, g, beta are [n][Hv]; A_log is [Hv].  The pages feed the recurrence
 * these two per-head scalars without printing how they are formed; this is
 * the layer's standard recipe (decay always <= 0, strength in (0, 1)). */
void oracle_gdn_gating(long n, int Hv, const double* A_log, const double* a, const double* b,
                       double* g, double* beta) {
  for (long r = 0; r < n; ++r)
    for (int h = 0; h < Hv; ++h) {
      const double av = a[r * Hv + h], bv = b[r * Hv + h];
      const double softplus = (av > 0.0 ? av : 0.0) + log1p(exp(-fabs(av)));
      g[r * Hv + h] = -exp(A_log[h]) * softplus;
      beta[r * Hv + h] = exp(bv < 0.0 ? bv : 0.0) / (1.0 + exp(-fabs(bv)));
    }
}

/* Verify (and optionally commit) every request, one decode step per row.
 *
 * accept_len == NULL: verify only; conv_state and ssm_state are not written.
 * accept_len != NULL: request b's slot receives the state after rows
 *   0..accept_len[b], i.e. accept_len[b]+1 decode steps.
 * o, snap_S, snap_cs may each be NULL (not produced).  snap_* receive, per
 * row t, the state and conv window a commit at a = t would write.
 * Requests with n_rows == 0 are inactive and produce nothing.  A request with
 * a slot outside [0, P) or n_rows outside [0, R] produces nothing and sets a
 * status bit; an accept_len outside [0, n_rows-1] skips that request's commit
 * (its o is still produced) and sets a status bit.  Returns the OR of bits. */
int oracle_gdn_verify_commit(const oracle_dims* d, const double* x, const double* g,
                             const double* beta, const double* conv_w, double* conv_state,
                             double* ssm_state, const int* slot_ids, const int* n_rows,
                             const int* accept_len, double* o, double* snap_S,
                             double* snap_cs, int mutation) {
  const int B = d->B, R = d->R, Hq = d->H_qk, Hv = d->H_v, dk = d->d_k, dv = d->d_v;
  const int W = d->W, P = d->P, G = Hv / Hq;
  const long C = 2L * Hq * dk + (long)Hv * dv;
  const long headS = (long)dv * dk, slotS = (long)Hv * headS;
  const long qoff = 0, koff = (long)Hq * dk, voff = 2L * Hq * dk;
  int status = 0;

  double* S = (double*)malloc(sizeof(double) * slotS);       /* running state */
  double* S_commit = (double*)malloc(sizeof(double) * slotS);
  double* seq = (double*)malloc(sizeof(double) * C * (W - 1 + R)); /* [C][W-1+R] */
  double* cs_commit = (double*)malloc(sizeof(double) * C * (W - 1));
  double* y = (double*)malloc(sizeof(double) * C);
  double* r = (double*)malloc(sizeof(double) * dv);
  const long L = W - 1 + R; /* length of one channel's staged sequence */

  for (int b = 0; b < B; ++b) {
    const int n = n_rows[b];
    const int s = slot_ids[b];
    if (n == 0) continue;
    if (s < 0 || s >= P) { status |= ORACLE_BAD_SLOT; continue; }
    if (n < 0 || n > R) { status |= ORACLE_BAD_NROWS; continue; }
    int commit = accept_len != NULL;
    int a = commit ? accept_len[b] : -1;
    if (commit && (a < 0 || a >= n)) { status |= ORACLE_BAD_ACCEPT; commit = 0; }
    int a_eff = a;
    if (commit && mutation == MUT_COMMIT_A_ROWS) a_eff = a - 1;

    /* Work on copies: the live slot is never touched during the rows. */
    memcpy(S, ssm_state + (long)s * slotS, sizeof(double) * slotS);
    if (commit && a_eff < 0) memcpy(S_commit, S, sizeof(double) * slotS);
    /* Stage [live history | verify inputs] per channel. */
    for (long c = 0; c < C; ++c) {
      for (int j = 0; j < W - 1; ++j)
        seq[c * L + j] = conv_state[((long)s * C + c) * (W - 1) + j];
      for (int t = 0; t < n; ++t)
        seq[c * L + W - 1 + t] = x[((long)b * R + t) * C + c];
    }

    for (int t = 0; t < n; ++t) {
      /* causal conv over the window ending at row t, then SiLU */
      for (long c = 0; c < C; ++c) {
        double z = 0.0;
        for (int j = 0; j < W; ++j) {
          const int tap = mutation == MUT_TAPS_REVERSED ? W - 1 - j : j;
          z += conv_w[c * W + tap] * seq[c * L + t + j];
        }
        y[c] = mutation == MUT_NO_SILU ? z : silu(z);
      }
      /* per-head L2 normalisation of q and k */
      for (int hq = 0; hq < Hq; ++hq) {
        for (int which = 0; which < 2; ++which) {
          if (which == 1 && mutation == MUT_NO_K_NORM) continue;
          double* v0 = y + (which ? koff : qoff) + (long)hq * dk;
          double ss = 0.0;
          for (int j = 0; j < dk; ++j) ss += v0[j] * v0[j];
          const double inv = 1.0 / sqrt(ss + d->l2_eps);
          for (int j = 0; j < dk; ++j) v0[j] *= inv;
        }
      }
      /* gated delta rule, one value head at a time */
      for (int h = 0; h < Hv; ++h) {
        const int hq = mutation == MUT_GQA_MODULO ? h % Hq : h / G;
        const double* q = y + qoff + (long)hq * dk;
        const double* k = y + koff + (long)hq * dk;
        const double* v = y + voff + (long)h * dv;
        const double alpha = exp(g[((long)b * R + t) * Hv + h]);
        const double bt = mutation == MUT_NO_BETA ? 1.0 : beta[((long)b * R + t) * Hv + h];
        double* Sh = S + (long)h * headS;
        double* oh = o ? o + (((long)b * R + t) * Hv + h) * dv : NULL;

        if (mutation != MUT_DECAY_AFTER)
          for (long e = 0; e < headS; ++e) Sh[e] *= alpha;
        if (oh && mutation == MUT_O_BEFORE_UPDATE)
          for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += Sh[(long)i * dk + j] * q[j];
            oh[i] = d->scale * acc;
          }
        for (int i = 0; i < dv; ++i) {
          double acc = 0.0;
          for (int j = 0; j < dk; ++j) acc += Sh[(long)i * dk + j] * k[j];
          r[i] = bt * (v[i] - acc); /* u_i */
        }
        for (int i = 0; i < dv; ++i)
          for (int j = 0; j < dk; ++j) Sh[(long)i * dk + j] += r[i] * k[j];
        if (mutation == MUT_DECAY_AFTER)
          for (long e = 0; e < headS; ++e) Sh[e] *= alpha;
        if (oh && mutation != MUT_O_BEFORE_UPDATE)
          for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += Sh[(long)i * dk + j] * q[j];
            oh[i] = mutation == MUT_NO_SCALE ? acc : d->scale * acc;
          }
      }
      /* state and window as a commit at a = t would leave them */
      if (snap_S) memcpy(snap_S + ((long)b * R + t) * slotS, S, sizeof(double) * slotS);
      if (snap_cs)
        for (long c = 0; c < C; ++c)
          for (int j = 0; j < W - 1; ++j)
            snap_cs[(((long)b * R + t) * C + c) * (W - 1) + j] = seq[c * L + t + 1 + j];
      if (commit && t == a_eff) memcpy(S_commit, S, sizeof(double) * slotS);
    }

    if (commit) {
      /* window after rows 0..a: entries a+1 .. a+W-1 of the staged sequence */
      const int first = mutation == MUT_CONV_COMMIT_EARLY ? a : a + 1;
      for (long c = 0; c < C; ++c)
        for (int j = 0; j < W - 1; ++j)
          cs_commit[c * (W - 1) + j] = seq[c * L + first + j];
      memcpy(ssm_state + (long)s * slotS, S_commit, sizeof(double) * slotS);
      memcpy(conv_state + (long)s * C * (W - 1), cs_commit, sizeof(double) * C * (W - 1));
    } else if (accept_len == NULL && mutation == MUT_VERIFY_WRITES_LIVE) {
      memcpy(ssm_state + (long)s * slotS, S, sizeof(double) * slotS);
    }
  }

  free(S);
  free(S_commit);
  free(seq);
  free(cs_commit);
  free(y);
  free(r);
  return status;
}

/* Greedy acceptance, written out plainly.  For each request b with
 * 0 < n_rows[b] <= R: target[b][t] = index of the largest logits[b][t][v]
 * over v (scanning v upward, a later entry wins only if strictly larger, so
 * equal largest values keep the lowest index; NaN never compares larger), for
 * t < n_rows[b]; accept_len[b] = number of leading drafts equal to the target
 * token at the row before them: d_{i+1} = drafts[b][i] is kept while
 * drafts[b][i] == target[b][i], at most n_rows[b]-1 drafts.  Other requests
 * get accept_len 0 (a bad n_rows sets the returned status bit). */
int oracle_greedy_accept(int B, int R, long V, const double* logits, const int* drafts,
                         const int* n_rows, int* target, int* accept_len) {
  int status = 0;
  for (int b = 0; b < B; ++b) {
    const int n = n_rows[b];
    accept_len[b] = 0;
    if (n < 0 || n > R) {
      status |= ORACLE_BAD_NROWS;
      continue;
    }
    for (int t = 0; t < n; ++t) {
      const double* row = logits + ((long)b * R + t) * V;
      long best = 0;
      for (long v = 1; v < V; ++v)
        if (row[v] > row[best] || (row[best] != row[best] && row[v] == row[v])) best = v;
      target[(long)b * R + t] = (int)best;
    }
    int a = 0;
    while (a < n - 1 && drafts[(long)b * (R - 1) + a] == target[(long)b * R + a]) ++a;
    accept_len[b] = a;
  }
  return status;
}
