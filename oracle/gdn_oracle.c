/*
 * gdn_oracle.c -- plain, slow, fp64 CPU oracle of the Gated DeltaNet layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library: it has its own argument struct and reads every input as fp64
 * (bf16 and fp32 inputs convert to fp64 exactly before they get here).
 *
 * What the layer is.  The source pages name the layer and fix two of its
 * properties:
 *   - "Serving large language models on our own stack" (keilab.io), section
 *     "Qwen3.5-35B-A3B from a real GGUF": a hybrid Gated-DeltaNet /
 *     gated-attention model;
 *   - llmxabe README, architecture paragraph ("Three consequences drive most
 *     of the design"): three Gated DeltaNet layers per gated-attention layer,
 *     each holding a fixed-size recurrent state per sequence, constant
 *     regardless of position (~60 MiB over 30 layers = 2 MiB fp32 per layer
 *     at 32 value heads x 128 x 128);
 *   - "Our own inference runtime" (skindeep.ai), section "What it is": gated
 *     delta net is a linear-attention design with a state kept per sequence.
 * The pages print no formula.  The layer definition this library implements
 * (the standard gated delta rule) is, per token t of one sequence:
 *   (1) causal depthwise conv of width W over the mixed q|k|v channels, then
 *       SiLU:   y_t[c] = silu( sum_{j=0}^{W-1} w[c][j] * x_{t-W+1+j}[c] ),
 *       w[c][W-1] multiplies the current token, w[c][0] the oldest; inputs
 *       before the sequence start come from the carried conv state (its row
 *       0 is the oldest);
 *   (2) per key head: q^ = q / sqrt(sum q^2 + eps_l2) / sqrt(d_k),
 *       k^ = k / sqrt(sum k^2 + eps_l2);
 *   (3) per value head h: g = -exp(A_log[h]) * softplus(a + dt_bias[h]),
 *       beta = sigmoid(b);
 *   (4) S_t = exp(g) S_{t-1} (I - beta k^ k^T) + beta v k^T, written here as
 *       S <- exp(g) S;  u = beta (v - S k^);  S <- S + u k^T;
 *   (5) o_t = S_t q^   (the 1/sqrt(d_k) sits inside q^);
 *   (6) out = o / sqrt(mean(o^2) + eps_rms) * w_norm * silu(z)
 *       (normalise first, then gate).
 * Value head h reads key head floor(h / (h_v / h_k)).
 *
 * Besides the sequential definition the file holds two independent
 * re-derivations used only to check it: the chunked WY/UT form with any
 * chunk length, and the explicit product form for short sequences.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int h_k;        /* key (and query) heads */
  int h_v;        /* value heads; a multiple of h_k */
  int d_k;        /* key head dimension */
  int d_v;        /* value head dimension */
  int conv_w;     /* width of the causal conv */
  double l2_eps;  /* epsilon inside the q/k L2 norm */
  double rms_eps; /* epsilon inside the output RMSNorm */
} or_dims;

/* ---- scalar pieces (step 1, 3, 6) -------------------------------------- */

double or_silu(double x) { return x / (1.0 + exp(-x)); }

double or_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* softplus(x) = log(1 + e^x), in the overflow-free form
 * max(x, 0) + log1p(e^{-|x|}). */
double or_softplus(double x) {
  return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* Step (3): the decay (log-space, <= 0) and the write gate of one token of
 * one value head. */
void or_gates(double a, double b, double A_log, double dt_bias,
              double* g, double* beta) {
  *g = -exp(A_log) * or_softplus(a + dt_bias);
  *beta = or_sigmoid(b);
}

/* ---- step (1): conv + SiLU over one sequence --------------------------- */

/* Raw input of channel c at position tau of the sequence (tau may be
 * negative: then it comes from the carried conv state, row W-1+tau). */
static double conv_input(const double* x, long ld_x, const double* state,
                         int n_ch, int W, long tau, int c) {
  if (tau >= 0) return x[tau * ld_x + c];
  return state[(long)(W - 1 + tau) * n_ch + c];
}

/* y[t][c] for t in [0, T), all n_ch channels.  x: [T][ld_x] (the first n_ch
 * columns are used); w: [n_ch][W]; state: [W-1][n_ch] or NULL for zeros.
 * state_out (may alias nothing else): the last W-1 raw rows of
 * (state || x), oldest first. */
void or_conv_silu(long T, int n_ch, int W, const double* x, long ld_x,
                  const double* w, const double* state, double* y,
                  double* state_out) {
  double* zero = NULL;
  if (!state) {
    zero = (double*)calloc((size_t)(W > 1 ? W - 1 : 1) * n_ch, sizeof(double));
    state = zero;
  }
  for (long t = 0; t < T; ++t)
    for (int c = 0; c < n_ch; ++c) {
      double acc = 0.0;
      for (int j = 0; j < W; ++j)
        acc += w[(long)c * W + j] *
               conv_input(x, ld_x, state, n_ch, W, t - (W - 1) + j, c);
      y[t * n_ch + c] = or_silu(acc);
    }
  if (state_out)
    for (int r = 0; r < W - 1; ++r)
      for (int c = 0; c < n_ch; ++c)
        state_out[(long)r * n_ch + c] =
            conv_input(x, ld_x, state, n_ch, W, T - (W - 1) + r, c);
  free(zero);
}

/* ---- step (2): L2 normalisation of one head vector --------------------- */

/* out = v / sqrt(sum v^2 + eps) * scale */
void or_l2norm(int d, const double* v, double eps, double scale, double* out) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += v[i] * v[i];
  double r = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < d; ++i) out[i] = v[i] * r * scale;
}

/* ---- step (6): gated RMSNorm of one head vector ------------------------ */

void or_gated_rmsnorm(int d, const double* o, const double* z,
                      const double* w, double eps, double* out) {
  double ms = 0.0;
  for (int i = 0; i < d; ++i) ms += o[i] * o[i];
  ms /= d;
  double r = 1.0 / sqrt(ms + eps);
  for (int i = 0; i < d; ++i) out[i] = o[i] * r * w[i] * or_silu(z[i]);
}

/* ---- steps (4)-(5): the recurrence of one (sequence, value head) ------- */

/* One token.  S: [d_v][d_k] row-major (row i = output component i).
 * q, k already normalised.  o: [d_v]. */
void or_delta_step(int d_k, int d_v, double* S, const double* q,
                   const double* k, const double* v, double g, double beta,
                   double* o) {
  double decay = exp(g);
  for (long e = 0; e < (long)d_v * d_k; ++e) S[e] *= decay;
  for (int i = 0; i < d_v; ++i) {
    double sk = 0.0;
    for (int j = 0; j < d_k; ++j) sk += S[(long)i * d_k + j] * k[j];
    double u = beta * (v[i] - sk);
    for (int j = 0; j < d_k; ++j) S[(long)i * d_k + j] += u * k[j];
  }
  for (int i = 0; i < d_v; ++i) {
    double acc = 0.0;
    for (int j = 0; j < d_k; ++j) acc += S[(long)i * d_k + j] * q[j];
    o[i] = acc;
  }
}

/* Sequential recurrence over T tokens.  q,k: [T][d_k]; v,o: [T][d_v];
 * g, beta: [T]; S: [d_v][d_k] in/out. */
void or_recurrence_seq(long T, int d_k, int d_v, const double* q,
                       const double* k, const double* v, const double* g,
                       const double* beta, double* S, double* o) {
  for (long t = 0; t < T; ++t)
    or_delta_step(d_k, d_v, S, q + t * d_k, k + t * d_k, v + t * d_v, g[t],
                  beta[t], o + t * d_v);
}

/* Chunked WY/UT form of the same recurrence, chunk length C (any C >= 1).
 * Derivation: inside a chunk with cumulative log-decay gamma_i = sum_{s<=i}
 * g_s, the corrections u_i obey (I + A) U = diag(beta) V - diag(beta
 * e^gamma) K S0^T with A_ij = beta_i e^{gamma_i-gamma_j} k_i.k_j (j<i), so
 *   U_w  = (I+A)^{-1} diag(beta) V,   W = (I+A)^{-1} diag(beta e^gamma) K,
 *   Vn   = U_w - W S0^T,
 *   O    = diag(e^gamma) Q S0^T + (tril(Q K^T) o e^{gamma_i-gamma_j}) Vn,
 *   S    = e^{gamma_last} S0 + Vn^T diag(e^{gamma_last-gamma}) K.
 * Every decay is formed as exp(difference) with a non-positive difference. */
void or_recurrence_chunked(long T, int d_k, int d_v, int C, const double* q,
                           const double* k, const double* v, const double* g,
                           const double* beta, double* S, double* o) {
  double* gam = (double*)malloc(sizeof(double) * C);
  double* A = (double*)malloc(sizeof(double) * C * C);
  double* Uw = (double*)malloc(sizeof(double) * C * d_v);
  double* W = (double*)malloc(sizeof(double) * C * d_k);
  double* Vn = (double*)malloc(sizeof(double) * C * d_v);
  double* S0 = (double*)malloc(sizeof(double) * d_v * d_k);
  for (long c0 = 0; c0 < T; c0 += C) {
    int L = (int)((T - c0) < C ? (T - c0) : C);
    const double* Kc = k + c0 * d_k;
    const double* Qc = q + c0 * d_k;
    const double* Vc = v + c0 * d_v;
    double run = 0.0;
    for (int i = 0; i < L; ++i) { run += g[c0 + i]; gam[i] = run; }
    for (int i = 0; i < L; ++i)
      for (int j = 0; j < L; ++j) {
        double val = 0.0;
        if (j < i) {
          double kk = 0.0;
          for (int e = 0; e < d_k; ++e) kk += Kc[i * d_k + e] * Kc[j * d_k + e];
          val = beta[c0 + i] * exp(gam[i] - gam[j]) * kk;
        }
        A[i * C + j] = val;
      }
    /* forward substitution: (I + A) X = R, row by row */
    for (int i = 0; i < L; ++i) {
      double bi = beta[c0 + i];
      for (int e = 0; e < d_v; ++e) Uw[i * d_v + e] = bi * Vc[i * d_v + e];
      for (int e = 0; e < d_k; ++e)
        W[i * d_k + e] = bi * exp(gam[i]) * Kc[i * d_k + e];
      for (int j = 0; j < i; ++j) {
        double aij = A[i * C + j];
        for (int e = 0; e < d_v; ++e) Uw[i * d_v + e] -= aij * Uw[j * d_v + e];
        for (int e = 0; e < d_k; ++e) W[i * d_k + e] -= aij * W[j * d_k + e];
      }
    }
    memcpy(S0, S, sizeof(double) * d_v * d_k);
    for (int i = 0; i < L; ++i)
      for (int e = 0; e < d_v; ++e) {
        double ws = 0.0;
        for (int j = 0; j < d_k; ++j) ws += W[i * d_k + j] * S0[e * d_k + j];
        Vn[i * d_v + e] = Uw[i * d_v + e] - ws;
      }
    for (int i = 0; i < L; ++i)
      for (int e = 0; e < d_v; ++e) {
        double qs = 0.0;
        for (int j = 0; j < d_k; ++j) qs += Qc[i * d_k + j] * S0[e * d_k + j];
        double acc = exp(gam[i]) * qs;
        for (int s = 0; s <= i; ++s) {
          double qk = 0.0;
          for (int j = 0; j < d_k; ++j) qk += Qc[i * d_k + j] * Kc[s * d_k + j];
          acc += qk * exp(gam[i] - gam[s]) * Vn[s * d_v + e];
        }
        o[(c0 + i) * d_v + e] = acc;
      }
    double gl = gam[L - 1];
    for (int e = 0; e < d_v; ++e)
      for (int j = 0; j < d_k; ++j) {
        double acc = exp(gl) * S0[e * d_k + j];
        for (int s = 0; s < L; ++s)
          acc += Vn[s * d_v + e] * exp(gl - gam[s]) * Kc[s * d_k + j];
        S[e * d_k + j] = acc;
      }
  }
  free(gam); free(A); free(Uw); free(W); free(Vn); free(S0);
}

/* Explicit product form, for short sequences only.  With the per-token
 * transition A_t = e^{g_t} (I - beta_t k_t k_t^T) (d_k x d_k) and
 * P(a, b) = A_a A_{a+1} ... A_b (identity when a > b):
 *   S_t = S_0 P(1, t) + sum_{s<=t} beta_s v_s k_s^T P(s+1, t),
 *   o_t = S_t q_t.
 * Every S_t is built from scratch from this closed sum (no recursion on S),
 * so the cost is O(T^2 d^3): keep T and d small. */
void or_recurrence_products(long T, int d_k, int d_v, const double* q,
                            const double* k, const double* v, const double* g,
                            const double* beta, double* S, double* o) {
  long dd = (long)d_k * d_k;
  double* At = (double*)malloc(sizeof(double) * dd * (T > 0 ? T : 1));
  double* P = (double*)malloc(sizeof(double) * dd);
  double* tmp = (double*)malloc(sizeof(double) * dd);
  double* S0 = (double*)malloc(sizeof(double) * d_v * d_k);
  double* St = (double*)malloc(sizeof(double) * d_v * d_k);
  memcpy(S0, S, sizeof(double) * d_v * d_k);
  for (long t = 0; t < T; ++t) {
    double e = exp(g[t]);
    for (int r = 0; r < d_k; ++r)
      for (int c = 0; c < d_k; ++c)
        At[t * dd + r * d_k + c] =
            e * ((r == c ? 1.0 : 0.0) - beta[t] * k[t * d_k + r] * k[t * d_k + c]);
  }
  for (long t = 0; t < T; ++t) {
    /* term s = -1 stands for the initial state: S_0 P(0, t) */
    memset(St, 0, sizeof(double) * d_v * d_k);
    for (long s = -1; s <= t; ++s) {
      /* P = A_{s+1} ... A_t */
      for (int r = 0; r < d_k; ++r)
        for (int c = 0; c < d_k; ++c) P[r * d_k + c] = (r == c);
      for (long m = s + 1; m <= t; ++m) {
        for (int r = 0; r < d_k; ++r)
          for (int c = 0; c < d_k; ++c) {
            double acc = 0.0;
            for (int x = 0; x < d_k; ++x)
              acc += P[r * d_k + x] * At[m * dd + x * d_k + c];
            tmp[r * d_k + c] = acc;
          }
        memcpy(P, tmp, sizeof(double) * dd);
      }
      for (int i = 0; i < d_v; ++i)
        for (int c = 0; c < d_k; ++c) {
          double acc = 0.0;
          if (s < 0) {
            for (int x = 0; x < d_k; ++x) acc += S0[i * d_k + x] * P[x * d_k + c];
          } else {
            for (int x = 0; x < d_k; ++x)
              acc += beta[s] * v[s * d_v + i] * k[s * d_k + x] * P[x * d_k + c];
          }
          St[i * d_k + c] += acc;
        }
    }
    for (int i = 0; i < d_v; ++i) {
      double acc = 0.0;
      for (int c = 0; c < d_k; ++c) acc += St[i * d_k + c] * q[t * d_k + c];
      o[t * d_v + i] = acc;
    }
  }
  if (T > 0) memcpy(S, St, sizeof(double) * d_v * d_k);
  free(At); free(P); free(tmp); free(S0); free(St);
}

/* ---- the whole layer over cu_seqlens-packed sequences ------------------ */

/*
 * qkv:   [T_tot][Cc], Cc = 2 h_k d_k + h_v d_v, channel order q | k | v
 * z:     [T_tot][h_v][d_v];  a, b: [T_tot][h_v]
 * A_log, dt_bias: [h_v];  conv_w: [Cc][W];  norm_w: [d_v]
 * cu_seqlens: [n_seqs + 1], non-decreasing, cu_seqlens[0] = 0
 * conv_state: [n_seqs][W-1][Cc] in/out;  ssm_state: [n_seqs][h_v][d_v][d_k]
 * in/out;  out: [T_tot][h_v][d_v]
 * head_mask: NULL (all value heads) or [h_v] flags; unmasked heads leave
 *   their out and ssm_state untouched (used to sample large cases).
 * chunk: 0 runs the sequential recurrence, C > 0 the chunked form.
 * n_threads: OpenMP threads over independent (sequence, value head) units.
 * Returns 0, or -1 on an inconsistent argument.
 */
int or_layer(const or_dims* dm, const double* qkv, const double* z,
             const double* a, const double* b, const double* A_log,
             const double* dt_bias, const double* conv_w,
             const double* norm_w, const int64_t* cu_seqlens, int n_seqs,
             double* conv_state, double* ssm_state, double* out,
             const int32_t* head_mask, int chunk, int n_threads) {
  const int Hk = dm->h_k, Hv = dm->h_v, dk = dm->d_k, dv = dm->d_v,
            W = dm->conv_w;
  if (Hk <= 0 || Hv <= 0 || Hv % Hk || dk <= 0 || dv <= 0 || W < 1) return -1;
  const int G = Hv / Hk;
  const int Cc = 2 * Hk * dk + Hv * dv;
  const long n_units = (long)n_seqs * Hv;
  int bad = 0;
  for (int n = 0; n < n_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) bad = 1;
  if (bad || cu_seqlens[0] != 0) return -1;

#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (long unit = 0; unit < n_units; ++unit) {
    const int n = (int)(unit / Hv), h = (int)(unit % Hv), kh = h / G;
    if (head_mask && !head_mask[h]) continue;
    const long t0 = cu_seqlens[n], T = cu_seqlens[n + 1] - t0;
    /* the channels this unit reads: q and k of key head kh, v of head h */
    const int chq = kh * dk, chk = Hk * dk + kh * dk, chv = 2 * Hk * dk + h * dv;
    const double* state = conv_state + (long)n * (W - 1) * Cc;
    double* yq = (double*)malloc(sizeof(double) * (T > 0 ? T : 1) * dk);
    double* yk = (double*)malloc(sizeof(double) * (T > 0 ? T : 1) * dk);
    double* yv = (double*)malloc(sizeof(double) * (T > 0 ? T : 1) * dv);
    double* wq = (double*)malloc(sizeof(double) * dk * W);
    double* sq = (double*)malloc(sizeof(double) * (W > 1 ? W - 1 : 1) * dk);
    double* qn = (double*)malloc(sizeof(double) * (T > 0 ? T : 1) * dk);
    double* kn = (double*)malloc(sizeof(double) * (T > 0 ? T : 1) * dk);
    double* gv = (double*)malloc(sizeof(double) * (T > 0 ? T : 1));
    double* bv = (double*)malloc(sizeof(double) * (T > 0 ? T : 1));
    double* o = (double*)malloc(sizeof(double) * (T > 0 ? T : 1) * dv);
    double* wv = (double*)malloc(sizeof(double) * dv * W);
    double* sv = (double*)malloc(sizeof(double) * (W > 1 ? W - 1 : 1) * dv);
    /* step (1) on each channel group: gather that group's weights and carried
     * rows, then run the conv with the group's columns of qkv */
    struct { int ch, width; double* y; } grp[3] = {{chq, dk, yq}, {chk, dk, yk}, {chv, dv, yv}};
    for (int gi = 0; gi < 3; ++gi) {
      int c0 = grp[gi].ch, wd = grp[gi].width;
      double* wbuf = gi < 2 ? wq : wv;
      double* sbuf = gi < 2 ? sq : sv;
      for (int c = 0; c < wd; ++c)
        for (int j = 0; j < W; ++j) wbuf[c * W + j] = conv_w[(long)(c0 + c) * W + j];
      for (int r = 0; r < W - 1; ++r)
        for (int c = 0; c < wd; ++c) sbuf[r * wd + c] = state[(long)r * Cc + c0 + c];
      or_conv_silu(T, wd, W, qkv + t0 * Cc + c0, Cc, wbuf, sbuf, grp[gi].y, NULL);
    }
    /* steps (2)-(3) */
    for (long t = 0; t < T; ++t) {
      or_l2norm(dk, yq + t * dk, dm->l2_eps, 1.0 / sqrt((double)dk), qn + t * dk);
      or_l2norm(dk, yk + t * dk, dm->l2_eps, 1.0, kn + t * dk);
      or_gates(a[(t0 + t) * Hv + h], b[(t0 + t) * Hv + h], A_log[h], dt_bias[h],
               &gv[t], &bv[t]);
    }
    /* steps (4)-(5) */
    double* S = ssm_state + ((long)n * Hv + h) * dv * dk;
    if (chunk > 0)
      or_recurrence_chunked(T, dk, dv, chunk, qn, kn, yv, gv, bv, S, o);
    else
      or_recurrence_seq(T, dk, dv, qn, kn, yv, gv, bv, S, o);
    /* step (6) */
    for (long t = 0; t < T; ++t)
      or_gated_rmsnorm(dv, o + t * dv, z + ((t0 + t) * Hv + h) * dv, norm_w,
                       dm->rms_eps, out + ((t0 + t) * Hv + h) * dv);
    free(yq); free(yk); free(yv); free(wq); free(sq); free(qn); free(kn);
    free(gv); free(bv); free(o); free(wv); free(sv);
  }

  /* hand-off of the conv state: after every unit has read the old one */
  double* rows = (double*)malloc(sizeof(double) * (W > 1 ? W - 1 : 1) * Cc);
  for (int n = 0; n < n_seqs; ++n) {
    const long t0 = cu_seqlens[n], T = cu_seqlens[n + 1] - t0;
    double* st = conv_state + (long)n * (W - 1) * Cc;
    for (int r = 0; r < W - 1; ++r)
      for (int c = 0; c < Cc; ++c)
        rows[(long)r * Cc + c] =
            conv_input(qkv + t0 * Cc, Cc, st, Cc, W, T - (W - 1) + r, c);
    memcpy(st, rows, sizeof(double) * (W > 1 ? W - 1 : 0) * Cc);
  }
  free(rows);
  return 0;
}

/* ---- the dense projections around the layer ---------------------------
 *
 * In the hybrid models the pages run, every Gated DeltaNet layer sits between
 * two dense projections ("Serving large language models on our own stack",
 * section "Qwen3.5-35B-A3B from a real GGUF"; llmxabe README, architecture
 * paragraph): an input projection from the hidden state to the layer's
 * inputs q|k|v, z, a, b, and an output projection from the gated-norm output
 * back to the hidden size.  Both are y = x w^T with w stored output features
 * by input features.
 *
 * x: [M][K];  w: [N][K];  y: [M][N];  y[m][n] = sum_{k} x[m][k] w[n][k],
 * summed in increasing k in fp64.
 */
void or_linear(long M, long N, long K, const double* x, const double* w, double* y) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
  for (long m = 0; m < M; ++m)
    for (long n = 0; n < N; ++n) {
      double acc = 0.0;
      for (long k = 0; k < K; ++k) acc += x[m * K + k] * w[n * K + k];
      y[m * N + n] = acc;
    }
}

/* Storage of a value as bf16 (8 significant bits, round to nearest, ties to
 * even): the layer's activations, the projections' outputs, are bf16.  With
 * x = m 2^e, 1/2 <= |m| < 1, the bf16 value is round(m 2^8) 2^(e-8), the
 * rounding in the default nearest-even mode.  Zero, infinities and NaN pass
 * through; values below the bf16 normal range (2^-126) are not handled. */
void or_round_bf16(long n, const double* x, double* y) {
  for (long i = 0; i < n; ++i) {
    if (x[i] == 0.0 || !isfinite(x[i])) {
      y[i] = x[i];
      continue;
    }
    int e;
    const double m = frexp(x[i], &e);
    y[i] = ldexp(nearbyint(ldexp(m, 8)), e - 8);
  }
}

/* Threads the OpenMP runtime would use (reported beside the CPU timing). */
int or_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
