/*
 * hla_oracle.c — plain, slow, fp64 CPU oracle of the Lightning Attention RNN mixer
 * (and, at the end of the file, of the hybrid's softmax attention layer).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file.  The only legitimate users are the test suite, the smoke check in
 * __graft_entry__.py and the cpu_baseline / reference legs of bench.py.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (arXiv 2601.22156, "Hybrid Linear Attention Done Right",
 * Appendix A, Eq. 18 "RNN Layers" and Eq. 19 "Forget Gate"), per head, with
 * row vectors and S in R^{d_k x d_v}:
 *
 *   q_t  = Norm(q_raw_t)              k_t = Norm(k_raw_t)          (Eq. 12 / 18)
 *   q~_t = RoPE_t(q_t)                k~_t = RoPE_t(k_t) / sqrt(d)  (Eq. 18)
 *   S_t  = gamma * S_{t-1} + k~_t^T v_t                              (Eq. 18)
 *   o_t  = q~_t S_t                   (query after the update)       (Eq. 18)
 *   y_t  = Norm(o_t) * sigmoid(g_t)                                  (Eq. 14 / 18)
 *
 * The projections x W_q, x W_k, x W_v, x W_z and the output projection W_o sit
 * outside the mixer: q, k, v are the projected rows and g is the pre-sigmoid
 * gate logit x W_z.
 *
 * Readings where the paper leaves a step open:
 *   - Norm is RMSNorm x / sqrt(mean(x^2) + eps) with unit weight, eps a
 *     parameter (1e-6 in every workload).
 *   - RoPE is the rotate-half form: for i < d/2 the pair (x_i, x_{i+d/2}) is
 *     rotated by the angle p * base^(-2i/d); the angle is formed in fp64.
 *   - Positions are 0-based: token t of a call sits at p = pos_offset + t.
 *   - Head h (0-based) uses gamma_h = exp(-2^(-8(h+1)/H)) (Eq. 19 with the
 *     paper's 1-based head index h+1).
 *
 * Layouts: activations [B, T, H, d] row-major (d fastest); state [B, H, d, d]
 * with the d_v index fastest.  All arrays are fp64.  Every (b, h) recurrence is
 * independent; OpenMP spreads them over the host cores.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX(b, t, h, B_, T_, H_, d_) ((((size_t)(b) * (T_) + (t)) * (H_) + (h)) * (d_))

int hla_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads for the following oracle calls (for timing it on fewer cores). */
void hla_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Eq. 19: gamma_h = exp(-2^(-8h/H)) for the paper's h = 1..H. */
void hla_oracle_gamma(int H, double *gamma) {
  for (int h = 0; h < H; ++h) gamma[h] = exp(-pow(2.0, -8.0 * (double)(h + 1) / (double)H));
}

/* 1 / sqrt(mean(x^2) + eps): the RMSNorm scale (Zhang & Sennrich 2019). */
static double rms_scale(const double *x, int d, double eps) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += x[i] * x[i];
  return 1.0 / sqrt(ss / (double)d + eps);
}

/* Angle of RoPE pair i at position p: p * base^(-2i/d). */
static double rope_angle(int64_t p, int i, int d, double base) {
  return (double)p * pow(base, -2.0 * (double)i / (double)d);
}

/* RoPE_p applied to x (rotate-half pairing), written to out. */
static void rope_apply(const double *x, int d, int64_t p, double base, double *out) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double phi = rope_angle(p, i, d, base);
    double c = cos(phi), s = sin(phi);
    double a = x[i], b = x[i + half];
    out[i] = a * c - b * s;
    out[i + half] = a * s + b * c;
  }
}

/* Transpose of RoPE_p (its inverse), used by the backward pass. */
static void rope_apply_transpose(const double *x, int d, int64_t p, double base, double *out) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double phi = rope_angle(p, i, d, base);
    double c = cos(phi), s = sin(phi);
    double a = x[i], b = x[i + half];
    out[i] = a * c + b * s;
    out[i + half] = -a * s + b * c;
  }
}

/* q~ or k~ of Eq. 18: Norm, then RoPE at position p, then multiply by scale
 * (1 for queries, 1/sqrt(d) for keys).  Exposed so tests can pin it alone. */
void hla_oracle_feature(int d, const double *x, int64_t p, double base, double eps, double scale,
                        double *out) {
  double r = rms_scale(x, d, eps);
  double tmp[512];
  for (int i = 0; i < d; ++i) tmp[i] = x[i] * r;
  rope_apply(tmp, d, p, base, out);
  for (int i = 0; i < d; ++i) out[i] *= scale;
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* y = Norm(o) * sigmoid(g) (Eq. 18, last two lines, before W_o). */
static void gate_output(const double *o, const double *g, int d, double eps, double *y) {
  double r = rms_scale(o, d, eps);
  for (int j = 0; j < d; ++j) y[j] = o[j] * r * sigmoid(g[j]);
}

static int check_shape(int B, int T, int H, int d) {
  if (B < 1 || T < 1 || H < 1 || d < 2 || (d & 1) || d > 512) return 1;
  return 0;
}

/*
 * Per-timestep recurrence of Eq. 18 over T tokens, for every (b, h).
 * state_in may be NULL (zero initial state).  y, o, state_out may each be NULL.
 */
int hla_oracle_prefill(int B, int T, int H, int d, const double *q, const double *k,
                       const double *v, const double *g, const double *gamma,
                       const double *state_in, int64_t pos_offset, double base, double eps,
                       double *y, double *o, double *state_out) {
  if (check_shape(B, T, H, d)) return 1;
  const double kscale = 1.0 / sqrt((double)d);
  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int bh = 0; bh < B * H; ++bh) {
    int b = bh / H, h = bh % H;
    double gm = gamma[h];
    double *S = (double *)calloc((size_t)d * d, sizeof(double));
    double *qt = (double *)malloc(sizeof(double) * d * 4);
    if (!S || !qt) {
      fail = 1;
      free(S);
      free(qt);
      continue;
    }
    double *kt = qt + d, *ot = qt + 2 * d, *yt = qt + 3 * d;
    if (state_in) memcpy(S, state_in + (size_t)bh * d * d, sizeof(double) * d * d);
    for (int t = 0; t < T; ++t) {
      size_t base_idx = IDX(b, t, h, B, T, H, d);
      int64_t p = pos_offset + t;
      hla_oracle_feature(d, q + base_idx, p, base, eps, 1.0, qt);
      hla_oracle_feature(d, k + base_idx, p, base, eps, kscale, kt);
      const double *vt = v + base_idx;
      /* S_t = gamma S_{t-1} + k~_t^T v_t */
      for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) S[(size_t)i * d + j] = gm * S[(size_t)i * d + j] + kt[i] * vt[j];
      /* o_t = q~_t S_t */
      for (int j = 0; j < d; ++j) ot[j] = 0.0;
      for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) ot[j] += qt[i] * S[(size_t)i * d + j];
      if (o) memcpy(o + base_idx, ot, sizeof(double) * d);
      if (y) {
        gate_output(ot, g + base_idx, d, eps, yt);
        memcpy(y + base_idx, yt, sizeof(double) * d);
      }
    }
    if (state_out) memcpy(state_out + (size_t)bh * d * d, S, sizeof(double) * d * d);
    free(S);
    free(qt);
  }
  return fail ? 3 : 0;
}

/*
 * The same mixer evaluated chunk by chunk (the block form of the closed
 * recurrence S_t = sum_{s<=t} gamma^{t-s} k~_s^T v_s):
 *   o_i   = gamma^{i+1} q~_i S_n + sum_{j<=i} gamma^{i-j} (q~_i . k~_j) v_j
 *   S_n+1 = gamma^{c} S_n + sum_j gamma^{c-1-j} k~_j^T v_j
 * with i, j the in-chunk indices and c the chunk's true length.  Used only by
 * the tests that check chunked == recurrent.
 */
int hla_oracle_prefill_chunked(int B, int T, int H, int d, int chunk, const double *q,
                               const double *k, const double *v, const double *g,
                               const double *gamma, const double *state_in, int64_t pos_offset,
                               double base, double eps, double *y, double *o,
                               double *state_out) {
  if (check_shape(B, T, H, d) || chunk < 1) return 1;
  const double kscale = 1.0 / sqrt((double)d);
  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int bh = 0; bh < B * H; ++bh) {
    int b = bh / H, h = bh % H;
    double gm = gamma[h];
    double *S = (double *)calloc((size_t)d * d, sizeof(double));
    double *Qc = (double *)malloc(sizeof(double) * (size_t)chunk * d);
    double *Kc = (double *)malloc(sizeof(double) * (size_t)chunk * d);
    double *ot = (double *)malloc(sizeof(double) * d * 2);
    if (!S || !Qc || !Kc || !ot) {
      fail = 1;
      free(S); free(Qc); free(Kc); free(ot);
      continue;
    }
    double *yt = ot + d;
    if (state_in) memcpy(S, state_in + (size_t)bh * d * d, sizeof(double) * d * d);
    for (int n0 = 0; n0 < T; n0 += chunk) {
      int c = (T - n0 < chunk) ? (T - n0) : chunk;
      for (int i = 0; i < c; ++i) {
        size_t bi = IDX(b, n0 + i, h, B, T, H, d);
        hla_oracle_feature(d, q + bi, pos_offset + n0 + i, base, eps, 1.0, Qc + (size_t)i * d);
        hla_oracle_feature(d, k + bi, pos_offset + n0 + i, base, eps, kscale, Kc + (size_t)i * d);
      }
      for (int i = 0; i < c; ++i) {
        const double *qi = Qc + (size_t)i * d;
        double inter = pow(gm, (double)(i + 1));
        for (int j = 0; j < d; ++j) ot[j] = 0.0;
        for (int a = 0; a < d; ++a)
          for (int j = 0; j < d; ++j) ot[j] += inter * qi[a] * S[(size_t)a * d + j];
        for (int s = 0; s <= i; ++s) {
          double dot = 0.0;
          for (int a = 0; a < d; ++a) dot += qi[a] * Kc[(size_t)s * d + a];
          double w = pow(gm, (double)(i - s)) * dot;
          const double *vs = v + IDX(b, n0 + s, h, B, T, H, d);
          for (int j = 0; j < d; ++j) ot[j] += w * vs[j];
        }
        size_t bi = IDX(b, n0 + i, h, B, T, H, d);
        if (o) memcpy(o + bi, ot, sizeof(double) * d);
        if (y) {
          gate_output(ot, g + bi, d, eps, yt);
          memcpy(y + bi, yt, sizeof(double) * d);
        }
      }
      double carry = pow(gm, (double)c);
      for (size_t e = 0; e < (size_t)d * d; ++e) S[e] *= carry;
      for (int s = 0; s < c; ++s) {
        double w = pow(gm, (double)(c - 1 - s));
        const double *ks = Kc + (size_t)s * d;
        const double *vs = v + IDX(b, n0 + s, h, B, T, H, d);
        for (int a = 0; a < d; ++a)
          for (int j = 0; j < d; ++j) S[(size_t)a * d + j] += w * ks[a] * vs[j];
      }
    }
    if (state_out) memcpy(state_out + (size_t)bh * d * d, S, sizeof(double) * d * d);
    free(S); free(Qc); free(Kc); free(ot);
  }
  return fail ? 3 : 0;
}

/*
 * One decode step: Eq. 18 for a single token per sequence.  Inputs are
 * [B, 1, H, d]; pos[b] is the RoPE position of sequence b.  state_out may
 * equal state_in (in-place update).
 */
int hla_oracle_decode(int B, int H, int d, const double *q, const double *k, const double *v,
                      const double *g, const double *gamma, const int64_t *pos,
                      const double *state_in, double base, double eps, double *y, double *o,
                      double *state_out) {
  if (check_shape(B, 1, H, d)) return 1;
  const double kscale = 1.0 / sqrt((double)d);
  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int bh = 0; bh < B * H; ++bh) {
    int b = bh / H, h = bh % H;
    double gm = gamma[h];
    double *S = (double *)malloc(sizeof(double) * (size_t)d * d);
    double *qt = (double *)malloc(sizeof(double) * d * 4);
    if (!S || !qt) {
      fail = 1;
      free(S); free(qt);
      continue;
    }
    double *kt = qt + d, *ot = qt + 2 * d, *yt = qt + 3 * d;
    memcpy(S, state_in + (size_t)bh * d * d, sizeof(double) * d * d);
    size_t bi = IDX(b, 0, h, B, 1, H, d);
    hla_oracle_feature(d, q + bi, pos[b], base, eps, 1.0, qt);
    hla_oracle_feature(d, k + bi, pos[b], base, eps, kscale, kt);
    const double *vt = v + bi;
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < d; ++j) S[(size_t)i * d + j] = gm * S[(size_t)i * d + j] + kt[i] * vt[j];
    for (int j = 0; j < d; ++j) ot[j] = 0.0;
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < d; ++j) ot[j] += qt[i] * S[(size_t)i * d + j];
    if (o) memcpy(o + bi, ot, sizeof(double) * d);
    if (y) {
      gate_output(ot, g + bi, d, eps, yt);
      memcpy(y + bi, yt, sizeof(double) * d);
    }
    memcpy(state_out + (size_t)bh * d * d, S, sizeof(double) * d * d);
    free(S);
    free(qt);
  }
  return fail ? 3 : 0;
}

/*
 * Gradient of L = sum(dy * y) + sum(dstate_out * S_{T-1}) with respect to the
 * raw inputs q, k, v, g and the initial state, by the chain rule through
 * Eq. 18 (the paper trains through this mixer in its distillation stages but
 * prints no backward formulas; this is the plain chain rule).
 *
 * Forward sweep (t ascending), keeping S_t:
 *   n = o r,  r = (mean(o^2) + eps)^(-1/2),  z = sigmoid(g)
 *   dg   = dy * n * z (1 - z)
 *   dn   = dy * z
 *   do   = r (dn - n mean(dn * n))                (RMSNorm backward)
 *   dq~  = do S_t^T
 *   dq   = RMSNorm-backward(RoPE_t^T dq~)
 * Reverse sweep (t descending), with Sbar_t = dL/dS_t:
 *   Sbar_{T-1} = dstate_out + q~^T do,   Sbar_t = gamma Sbar_{t+1} + q~_t^T do_t
 *   dk~ = v Sbar^T,  dv = k~ Sbar
 *   dk  = RMSNorm-backward(RoPE_t^T dk~ / sqrt(d))
 *   dstate_in = gamma Sbar_0
 * The recurrence is never inverted (no division by gamma).
 */
int hla_oracle_backward(int B, int T, int H, int d, const double *q, const double *k,
                        const double *v, const double *g, const double *gamma,
                        const double *state_in, const double *dy, const double *dstate_out,
                        int64_t pos_offset, double base, double eps, double *dq, double *dk,
                        double *dv, double *dg, double *dstate_in) {
  if (check_shape(B, T, H, d)) return 1;
  const double kscale = 1.0 / sqrt((double)d);
  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int bh = 0; bh < B * H; ++bh) {
    int b = bh / H, h = bh % H;
    double gm = gamma[h];
    double *S = (double *)calloc((size_t)d * d, sizeof(double));
    double *Sb = (double *)calloc((size_t)d * d, sizeof(double));
    double *dO = (double *)malloc(sizeof(double) * (size_t)T * d);
    double *w = (double *)malloc(sizeof(double) * d * 8);
    if (!S || !Sb || !dO || !w) {
      fail = 1;
      free(S); free(Sb); free(dO); free(w);
      continue;
    }
    double *qt = w, *kt = w + d, *ot = w + 2 * d, *nt = w + 3 * d, *dn = w + 4 * d,
           *gv = w + 5 * d, *gr = w + 6 * d, *xn = w + 7 * d;
    if (state_in) memcpy(S, state_in + (size_t)bh * d * d, sizeof(double) * d * d);
    /* forward sweep */
    for (int t = 0; t < T; ++t) {
      size_t bi = IDX(b, t, h, B, T, H, d);
      int64_t p = pos_offset + t;
      hla_oracle_feature(d, q + bi, p, base, eps, 1.0, qt);
      hla_oracle_feature(d, k + bi, p, base, eps, kscale, kt);
      const double *vt = v + bi;
      for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) S[(size_t)i * d + j] = gm * S[(size_t)i * d + j] + kt[i] * vt[j];
      for (int j = 0; j < d; ++j) ot[j] = 0.0;
      for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) ot[j] += qt[i] * S[(size_t)i * d + j];
      double r = rms_scale(ot, d, eps);
      double m = 0.0;
      for (int j = 0; j < d; ++j) {
        double z = sigmoid(g[bi + j]);
        nt[j] = ot[j] * r;
        if (dg) dg[bi + j] = dy[bi + j] * nt[j] * z * (1.0 - z);
        dn[j] = dy[bi + j] * z;
        m += dn[j] * nt[j];
      }
      m /= (double)d;
      double *dot = dO + (size_t)t * d;
      for (int j = 0; j < d; ++j) dot[j] = r * (dn[j] - nt[j] * m);
      if (dq) {
        /* dq~ = do S^T */
        for (int i = 0; i < d; ++i) {
          double acc = 0.0;
          for (int j = 0; j < d; ++j) acc += dot[j] * S[(size_t)i * d + j];
          gv[i] = acc;
        }
        rope_apply_transpose(gv, d, p, base, gr);
        double rq = rms_scale(q + bi, d, eps), mm = 0.0;
        for (int i = 0; i < d; ++i) {
          xn[i] = q[bi + i] * rq;
          mm += gr[i] * xn[i];
        }
        mm /= (double)d;
        for (int i = 0; i < d; ++i) dq[bi + i] = rq * (gr[i] - xn[i] * mm);
      }
    }
    /* reverse sweep */
    if (dstate_out) memcpy(Sb, dstate_out + (size_t)bh * d * d, sizeof(double) * d * d);
    for (int t = T - 1; t >= 0; --t) {
      size_t bi = IDX(b, t, h, B, T, H, d);
      int64_t p = pos_offset + t;
      if (t != T - 1)
        for (size_t e = 0; e < (size_t)d * d; ++e) Sb[e] *= gm;
      hla_oracle_feature(d, q + bi, p, base, eps, 1.0, qt);
      hla_oracle_feature(d, k + bi, p, base, eps, kscale, kt);
      const double *dot = dO + (size_t)t * d;
      for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) Sb[(size_t)i * d + j] += qt[i] * dot[j];
      const double *vt = v + bi;
      if (dv)
        for (int j = 0; j < d; ++j) {
          double acc = 0.0;
          for (int i = 0; i < d; ++i) acc += kt[i] * Sb[(size_t)i * d + j];
          dv[bi + j] = acc;
        }
      if (dk) {
        for (int i = 0; i < d; ++i) {
          double acc = 0.0;
          for (int j = 0; j < d; ++j) acc += Sb[(size_t)i * d + j] * vt[j];
          gv[i] = acc * kscale;
        }
        rope_apply_transpose(gv, d, p, base, gr);
        double rk = rms_scale(k + bi, d, eps), mm = 0.0;
        for (int i = 0; i < d; ++i) {
          xn[i] = k[bi + i] * rk;
          mm += gr[i] * xn[i];
        }
        mm /= (double)d;
        for (int i = 0; i < d; ++i) dk[bi + i] = rk * (gr[i] - xn[i] * mm);
      }
    }
    if (dstate_in)
      for (size_t e = 0; e < (size_t)d * d; ++e) dstate_in[(size_t)bh * d * d + e] = gm * Sb[e];
    free(S); free(Sb); free(dO); free(w);
  }
  return fail ? 3 : 0;
}

/*
 * NoPE softmax attention of the hybrid's attention layers (arXiv 2601.22156,
 * Section 5.1 "Attention Logits Scaling", Eq. 11, and Appendix A "Attention
 * Layers", Eq. 17), per query head h, whose keys and values are those of
 * key/value head h / (Hq / Hkv) (grouped-query attention):
 *
 *   s_t  = log_a(t + a)          t the paper's 1-based query position
 *   q~_t = s_t q_t / sqrt(d)
 *   o_t  = sum_{i <= t} exp(q~_t . k_i) v_i / sum_{j <= t} exp(q~_t . k_j)
 *   y_t  = Norm(o_t) * sigmoid(g_t)
 *
 * Readings: the printed denominator's exp(q~_j k_j) is the softmax's own
 * normalisation over the same keys, exp(q~_t k_j); token t of a call sits at
 * the 0-based position p = pos_offset + t, so s = ln(p + 1 + a) / ln(a); the
 * keys are this call's tokens 0..t; no positional encoding and no QK-norm.
 * The softmax subtracts the row's largest logit before exp (the same value in
 * exact arithmetic, and no overflow in fp64).
 * Layouts: q, g, y, o [B, T, Hq, d]; k, v [B, T, Hkv, d].  o may be NULL.
 * Returns 0, or non-zero on a bad shape or an allocation failure.
 */
int hla_oracle_attention(int B, int T, int Hq, int Hkv, int d, const double *q, const double *k,
                         const double *v, const double *g, double a, int64_t pos_offset,
                         double eps, double *y, double *o) {
  if (B < 0 || T < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || d < 1 || !(a > 1.0)) return 1;
  const int group = Hq / Hkv;
  const double la = log(a);
  int fail = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h) {
      double *w = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
      double *ot = (double *)malloc(sizeof(double) * (size_t)d);
      if (!w || !ot) {
#pragma omp atomic write
        fail = 1;
        free(w); free(ot);
        continue;
      }
      const int hk = h / group;
      for (int t = 0; t < T; ++t) {
        const size_t qi = (((size_t)b * T + t) * Hq + h) * d;
        const double s = log((double)(pos_offset + t) + 1.0 + a) / la;
        const double qs = s / sqrt((double)d);
        double m = -HUGE_VAL;
        for (int i = 0; i <= t; ++i) {
          const size_t ki = (((size_t)b * T + i) * Hkv + hk) * d;
          double dot = 0.0;
          for (int e = 0; e < d; ++e) dot += q[qi + e] * k[ki + e];
          w[i] = qs * dot;
          if (w[i] > m) m = w[i];
        }
        double z = 0.0;
        for (int i = 0; i <= t; ++i) {
          w[i] = exp(w[i] - m);
          z += w[i];
        }
        for (int e = 0; e < d; ++e) ot[e] = 0.0;
        for (int i = 0; i <= t; ++i) {
          const size_t vi = (((size_t)b * T + i) * Hkv + hk) * d;
          for (int e = 0; e < d; ++e) ot[e] += w[i] * v[vi + e];
        }
        for (int e = 0; e < d; ++e) ot[e] /= z;
        if (o) memcpy(o + qi, ot, sizeof(double) * (size_t)d);
        gate_output(ot, g + qi, d, eps, y + qi);
      }
      free(w); free(ot);
    }
  return fail ? 2 : 0;
}

/*
 * The projections around the RNN mixer, arXiv 2601.22156, Appendix A, Eq. 18
 * ("RNN Layers"): q_t = Norm(x_t W_q), k_t = Norm(x_t W_k), v_t = x_t W_v,
 * z_t = sigmoid(x_t W_z) take the projected rows x_t W (before the norm and
 * the sigmoid), and y_t = (Norm(o_t) . z_t) W_o^T maps the gated rows back.
 * Both are products of a row-major matrix with a transposed one:
 *   out[m, n] = sum_k a[m, k] w[n, k]     (a [M, K], w [N, K], out [M, N])
 * With w = W^T of the paper's W in R^{d x d_h} this is x_t W; with w = W_o
 * itself it is u_t W_o^T.  Plain fp64 loops, OpenMP over the rows m.
 */
int hla_oracle_matmul_nt(int M, int N, int K, const double *a, const double *w, double *out) {
  if (M < 0 || N < 0 || K < 0) return 1;
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      double s = 0.0;
      for (int k = 0; k < K; ++k) s += a[(size_t)m * K + k] * w[(size_t)n * K + k];
      out[(size_t)m * N + n] = s;
    }
  return 0;
}
