/*
 * ssm_oracle.c -- plain, slow, fp64 CPU oracle of the selective state-space (S6)
 * hot path: the causal depthwise conv1d + SiLU prologue, the selective scan
 * forward with its skip term and SiLU gate, the chunk-carry composition and the
 * single-token recurrent (decode) update.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. It shares no code, header, table or
 * helper with the CUDA library and includes none of it; the product path never
 * calls it.
 *
 * Every routine is the definition written out in double precision, in the order
 * the pages state it, with one loop per index and no blocking, fusion or
 * reordering. The only parallelism is an optional OpenMP loop over independent
 * (batch, channel) pairs, which does not change any arithmetic.
 *
 * Sources (page title, section / equation):
 *  - "Mamba" (ai360xpert.com, core ML), "The selection mechanism":
 *      Delta_t = softplus(W_Delta x_t + b_Delta); Abar_t = exp(Delta_t A); Bbar_t ~ Delta_t B.
 *  - "Mamba (Selective State-Space Model)" (gunjandhanuka.github.io), "Key math":
 *      B_t = s_B(x_t), C_t = s_C(x_t), Delta_t = softplus(s_Delta(x_t)), Abar_t = exp(Delta_t A).
 *  - "Mamba" (ozercemkelahmet.com/tools/mamba), "How it works" steps 1-3 and
 *      "A minimal selective scan in PyTorch": per-channel Delta, Euler Bbar = Delta B,
 *      h_t = Abar_t * h_{t-1} + Bbar_t u_t, y_t = C_t . h_t, zero initial state;
 *      "Deployment notes": long prompts are processed in chunks that pass the state on.
 *  - "Overview of Mamba (SSM) Model" (bembew.net), "How the Mamba Block Works":
 *      depthwise causal conv + SiLU before the SSM, a SiLU gate multiplying the output.
 * The skip term D*u and the returned final state follow the problem statement of
 * this library (y_t = C_t . h_t + D_d u_t, gated by silu(z_t)).
 *
 * Readings taken where the pages are silent (stated once here, used throughout):
 *  - Bbar is the Euler form Delta*B by default. With the zoh flag it is the zero-order-hold
 *    form (Abar - 1)/A * B = expm1(Delta A)/A * B ("Mamba", ai360xpert.com, "Show Me the
 *    Code": B_bar = (1 - A_bar)/(-A) B; "Mamba", inferensys.com: a zero-order hold rule
 *    discretizes the continuous system), whose limit as A -> 0 is the Euler form.
 *  - Delta, B and C are per token; A is a fixed parameter A[d, n].
 *  - B and C are shared by every channel: B[b, n, t], C[b, n, t].
 *  - The conv is a cross-correlation with K-1 zeros (or a supplied window) on
 *    the left: w[d, K-1] multiplies the current input.
 *  - out = (C.h + D*u) * silu(z); u is the post-conv, post-SiLU value.
 *  - The decode window holds the last K-1 raw inputs, oldest first.
 *
 * Layouts (all contiguous, row-major):
 *   u/x, delta, z, out : [batch, dim, seqlen]      B, C : [batch, dstate, seqlen]
 *   A : [dim, dstate]   D, delta_bias, conv_b : [dim]   conv_w : [dim, d_conv]
 *   h0, h_last : [batch, dim, dstate]   conv windows : [batch, dim, d_conv-1]
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* softplus(x) = log(1 + e^x), written in the overflow-free form max(x,0) + log1p(e^-|x|). */
static double softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

/* Input factor of Bbar = factor * B: Delta (Euler), or expm1(Delta A) / A (zero-order hold;
 * Delta when A = 0, its limit). */
static double bbar_factor(double Delta, double A, int zoh) {
  if (!zoh) return Delta;
  return A != 0.0 ? expm1(Delta * A) / A : Delta;
}

/* silu(x) = x * sigmoid(x) = x / (1 + e^-x). */
static double silu(double x) { return x / (1.0 + exp(-x)); }

void oracle_softplus(const double* x, double* y, long n) {
  for (long i = 0; i < n; ++i) y[i] = softplus(x[i]);
}

void oracle_silu(const double* x, double* y, long n) {
  for (long i = 0; i < n; ++i) y[i] = silu(x[i]);
}

/*
 * Causal depthwise conv1d of one channel:
 *   out[t] = sum_{k=0}^{K-1} w[k] * x[t - (K-1) + k] + bias, x[s < 0] = window[K-1+s] (or 0),
 * then out[t] = silu(out[t]) when apply_silu is set.
 */
static void conv_channel(const double* x, const double* w, double bias, const double* window,
                         double* out, long L, int K, int apply_silu) {
  for (long t = 0; t < L; ++t) {
    double acc = 0.0;
    for (int k = 0; k < K; ++k) {
      long s = t - (K - 1) + k;
      double xs;
      if (s >= 0) xs = x[s];
      else xs = window ? window[(K - 1) + s] : 0.0;
      acc += w[k] * xs;
    }
    acc += bias;
    out[t] = apply_silu ? silu(acc) : acc;
  }
}

void oracle_causal_conv1d(const double* x, const double* w, const double* bias, const double* window,
                          double* out, long batch, long dim, long seqlen, int d_conv, int apply_silu,
                          int nthreads) {
  long nch = batch * dim;
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
  for (long c = 0; c < nch; ++c) {
    long d = c % dim;
    conv_channel(x + c * seqlen, w + d * d_conv, bias ? bias[d] : 0.0,
                 window ? window + c * (d_conv - 1) : NULL, out + c * seqlen, seqlen, d_conv, apply_silu);
  }
}

/*
 * Selective scan forward over every (batch b, channel d):
 *   u_t      = x_t, or silu(causal conv of x)_t when conv_w is given
 *   Delta_t  = softplus(delta_t + delta_bias[d])   (delta_t + delta_bias[d] when delta_softplus == 0)
 *   h_t[n]   = exp(Delta_t A[d,n]) h_{t-1}[n] + Delta_t B[b,n,t] u_t,     h_{-1} = h0 or 0
 *   y_t      = sum_n C[b,n,t] h_t[n] + D[d] u_t
 *   out_t    = y_t * silu(z_t)   (y_t when z is NULL)
 * Optional outputs: h_last = h_{L-1}; conv_state_out = the last K-1 raw inputs
 * (taken from the window when seqlen < K-1); h_trace[b,d,t,n] = h_t[n].
 */
void oracle_selective_scan(const double* x, const double* delta, const double* A, const double* Bm,
                           const double* Cm, const double* Dskip, const double* z, const double* delta_bias,
                           int delta_softplus, const double* conv_w, const double* conv_b, int d_conv,
                           const double* conv_init, const double* h0, double* out, double* h_last,
                           double* conv_state_out, double* h_trace, long batch, long dim, long seqlen,
                           long dstate, int nthreads, int zoh) {
  long nch = batch * dim;
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
  for (long c = 0; c < nch; ++c) {
    long b = c / dim, d = c % dim;
    const double* xc = x + c * seqlen;
    double* u = (double*)malloc(sizeof(double) * (size_t)(seqlen > 0 ? seqlen : 1));
    double* h = (double*)malloc(sizeof(double) * (size_t)dstate);
    if (conv_w) {
      conv_channel(xc, conv_w + d * d_conv, conv_b ? conv_b[d] : 0.0,
                   conv_init ? conv_init + c * (d_conv - 1) : NULL, u, seqlen, d_conv, 1);
    } else {
      for (long t = 0; t < seqlen; ++t) u[t] = xc[t];
    }
    for (long n = 0; n < dstate; ++n) h[n] = h0 ? h0[c * dstate + n] : 0.0;
    for (long t = 0; t < seqlen; ++t) {
      double v = delta[c * seqlen + t] + (delta_bias ? delta_bias[d] : 0.0);
      double Delta = delta_softplus ? softplus(v) : v;
      for (long n = 0; n < dstate; ++n) {
        double Abar = exp(Delta * A[d * dstate + n]);
        double Bbar = bbar_factor(Delta, A[d * dstate + n], zoh) * Bm[(b * dstate + n) * seqlen + t];
        h[n] = Abar * h[n] + Bbar * u[t];
        if (h_trace) h_trace[(c * seqlen + t) * dstate + n] = h[n];
      }
      double y = 0.0;
      for (long n = 0; n < dstate; ++n) y += Cm[(b * dstate + n) * seqlen + t] * h[n];
      if (Dskip) y += Dskip[d] * u[t];
      if (z) y *= silu(z[c * seqlen + t]);
      out[c * seqlen + t] = y;
    }
    if (h_last)
      for (long n = 0; n < dstate; ++n) h_last[c * dstate + n] = h[n];
    if (conv_state_out && d_conv > 1) {
      /* raw input stream = [window (K-1 values, or zeros), x_0 .. x_{L-1}]; keep its last K-1 */
      long K1 = d_conv - 1;
      for (long j = 0; j < K1; ++j) {
        long s = seqlen - K1 + j; /* index into x; negative means the window */
        double v;
        if (s >= 0) v = xc[s];
        else v = conv_init ? conv_init[c * K1 + (K1 + s)] : 0.0;
        conv_state_out[c * K1 + j] = v;
      }
    }
    free(u);
    free(h);
  }
}

/*
 * Backward of oracle_causal_conv1d: given dout = dL/dout [b,d,t], the chain rule on
 *   acc_t = sum_k w[k] xs(t - (K-1) + k) + bias,  out_t = silu(acc_t) (or acc_t),
 * where xs(s) = x[s] for s >= 0 and window[K-1+s] for s < 0, gives
 *   dacc_t = dout_t silu'(acc_t) (or dout_t),  silu'(a) = s(a) (1 + a (1 - s(a)))
 *   dx[s] = sum_k w[k] dacc_{s + (K-1) - k} over t = s + (K-1) - k in [0, L)
 *   dwindow[j] (position s = j - (K-1)) likewise;  dw[d,k] = sum_{b,t} dacc_t xs(t - (K-1) + k)
 *   dbias[d] = sum_{b,t} dacc_t
 * Outputs: dx [b,d,L]; dwindow [b,d,K-1] (NULL: not wanted); dw [d,K]; dbias [d] (NULL: not
 * wanted). All are written, not accumulated into.
 */
void oracle_causal_conv1d_bwd(const double* x, const double* w, const double* bias, const double* window,
                              const double* dout, double* dx, double* dwindow, double* dw, double* dbias,
                              long batch, long dim, long seqlen, int d_conv, int apply_silu, int nthreads) {
  long nch = batch * dim;
  int K = d_conv;
  double* cw = (double*)calloc((size_t)(nch * K), sizeof(double));
  double* cb = (double*)calloc((size_t)nch, sizeof(double));
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
  for (long c = 0; c < nch; ++c) {
    long d = c % dim;
    const double* xc = x + c * seqlen;
    const double* wc = w + d * K;
    const double* win = window ? window + c * (K - 1) : NULL;
    double* dacc = (double*)malloc(sizeof(double) * (size_t)(seqlen > 0 ? seqlen : 1));
    for (long t = 0; t < seqlen; ++t) {
      double acc = bias ? bias[d] : 0.0;
      for (int k = 0; k < K; ++k) {
        long s = t - (K - 1) + k;
        double xs = s >= 0 ? xc[s] : (win ? win[(K - 1) + s] : 0.0);
        acc += wc[k] * xs;
      }
      double g = dout[c * seqlen + t];
      if (apply_silu) {
        double sg = 1.0 / (1.0 + exp(-acc));
        g *= sg * (1.0 + acc * (1.0 - sg));
      }
      dacc[t] = g;
      cb[c] += g;
      for (int k = 0; k < K; ++k) {
        long s = t - (K - 1) + k;
        double xs = s >= 0 ? xc[s] : (win ? win[(K - 1) + s] : 0.0);
        cw[c * K + k] += g * xs;
      }
    }
    /* dx[s] and dwindow: every (t, k) with t - (K-1) + k = s */
    for (long s = -(K - 1); s < seqlen; ++s) {
      double v = 0.0;
      for (int k = 0; k < K; ++k) {
        long t = s + (K - 1) - k;
        if (t >= 0 && t < seqlen) v += wc[k] * dacc[t];
      }
      if (s >= 0) dx[c * seqlen + s] = v;
      else if (dwindow) dwindow[c * (K - 1) + (K - 1) + s] = v;
    }
    free(dacc);
  }
  for (long d = 0; d < dim; ++d) {
    for (int k = 0; k < K; ++k) {
      double sw = 0.0;
      for (long b = 0; b < batch; ++b) sw += cw[(b * dim + d) * K + k];
      dw[d * K + k] = sw;
    }
    if (dbias) {
      double sb = 0.0;
      for (long b = 0; b < batch; ++b) sb += cb[b * dim + d];
      dbias[d] = sb;
    }
  }
  free(cw);
  free(cb);
}

/*
 * Composition of two affine maps h -> a*h + b (first (a1,b1), then (a2,b2)):
 *   (a1, b1) o (a2, b2) = (a1*a2, a2*b1 + b2).
 * This is the associative operator of the parallel scan ("Mamba", ai360xpert.com,
 * "Why this breaks the parallel form"; "Mamba" ozercemkelahmet.com, "Step 4").
 */
void oracle_compose(const double* a1, const double* b1, const double* a2, const double* b2, double* a,
                    double* b, long n) {
  for (long i = 0; i < n; ++i) {
    double aa = a1[i] * a2[i];
    double bb = a2[i] * b1[i] + b2[i];
    a[i] = aa;
    b[i] = bb;
  }
}

/*
 * Chunk aggregates: split time into chunks of chunk_len steps (the last one ragged).
 * For chunk q of channel (b, d), the aggregate (a, b)[n] is the composition, in
 * time order, of the per-step maps h -> Abar_t[n] h + Bbar_t[n] u_t over the
 * chunk, starting from the identity (1, 0). So b is the state at the chunk's end
 * when the chunk starts from zero, and a = prod_t Abar_t[n].
 * Layout of agg_a, agg_b: [batch, dim, nchunks, dstate].
 */
void oracle_chunk_aggregates(const double* x, const double* delta, const double* A, const double* Bm,
                             const double* delta_bias, int delta_softplus, const double* conv_w,
                             const double* conv_b, int d_conv, const double* conv_init, long chunk_len,
                             double* agg_a, double* agg_b, long batch, long dim, long seqlen, long dstate,
                             int nthreads, int zoh) {
  long nchunks = (seqlen + chunk_len - 1) / chunk_len;
  long nch = batch * dim;
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
  for (long c = 0; c < nch; ++c) {
    long b = c / dim, d = c % dim;
    const double* xc = x + c * seqlen;
    double* u = (double*)malloc(sizeof(double) * (size_t)(seqlen > 0 ? seqlen : 1));
    if (conv_w) {
      conv_channel(xc, conv_w + d * d_conv, conv_b ? conv_b[d] : 0.0,
                   conv_init ? conv_init + c * (d_conv - 1) : NULL, u, seqlen, d_conv, 1);
    } else {
      for (long t = 0; t < seqlen; ++t) u[t] = xc[t];
    }
    for (long q = 0; q < nchunks; ++q) {
      long t0 = q * chunk_len, t1 = t0 + chunk_len < seqlen ? t0 + chunk_len : seqlen;
      for (long n = 0; n < dstate; ++n) {
        double a = 1.0, bb = 0.0;
        for (long t = t0; t < t1; ++t) {
          double v = delta[c * seqlen + t] + (delta_bias ? delta_bias[d] : 0.0);
          double Delta = delta_softplus ? softplus(v) : v;
          double step_a = exp(Delta * A[d * dstate + n]);
          double step_b = bbar_factor(Delta, A[d * dstate + n], zoh) * Bm[(b * dstate + n) * seqlen + t] * u[t];
          double na, nb;
          oracle_compose(&a, &bb, &step_a, &step_b, &na, &nb, 1);
          a = na;
          bb = nb;
        }
        agg_a[((c * nchunks) + q) * dstate + n] = a;
        agg_b[((c * nchunks) + q) * dstate + n] = bb;
      }
    }
    free(u);
  }
}

/*
 * One recurrent (decode) step for every (batch b, channel d), in place:
 *   window  = [conv_state[b,d,0..K-2], x[b,d]]   (oldest first)
 *   u       = silu(sum_k conv_w[d,k] window[k] + conv_b[d]);  conv_state <- window[1..K-1]
 *             (u = x[b,d] when conv_w is NULL)
 *   Delta   = softplus(delta[b,d] + delta_bias[d])
 *   state[n]= exp(Delta A[d,n]) state[n] + Delta B[b,n] u
 *   y[b,d]  = (sum_n C[b,n] state[n] + D[d] u) * silu(z[b,d])
 * x, delta, z, y : [batch, dim]; B, C : [batch, dstate].
 */
void oracle_state_update(double* state, double* conv_state, const double* x, const double* delta,
                         const double* A, const double* Bm, const double* Cm, const double* Dskip,
                         const double* z, const double* delta_bias, int delta_softplus, const double* conv_w,
                         const double* conv_b, int d_conv, double* y, long batch, long dim, long dstate,
                         int nthreads, int zoh) {
  long nch = batch * dim;
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(static)
  for (long c = 0; c < nch; ++c) {
    long b = c / dim, d = c % dim;
    double u;
    if (conv_w) {
      int K = d_conv;
      double acc = 0.0;
      for (int k = 0; k < K; ++k) {
        double wk = (k < K - 1) ? conv_state[c * (K - 1) + k] : x[c];
        acc += conv_w[d * K + k] * wk;
      }
      acc += conv_b ? conv_b[d] : 0.0;
      u = silu(acc);
      for (int k = 0; k < K - 1; ++k) {
        double next = (k + 1 < K - 1) ? conv_state[c * (K - 1) + k + 1] : x[c];
        conv_state[c * (K - 1) + k] = next;
      }
    } else {
      u = x[c];
    }
    double v = delta[c] + (delta_bias ? delta_bias[d] : 0.0);
    double Delta = delta_softplus ? softplus(v) : v;
    double yy = 0.0;
    for (long n = 0; n < dstate; ++n) {
      double Abar = exp(Delta * A[d * dstate + n]);
      double Bbar = bbar_factor(Delta, A[d * dstate + n], zoh) * Bm[b * dstate + n];
      state[c * dstate + n] = Abar * state[c * dstate + n] + Bbar * u;
    }
    for (long n = 0; n < dstate; ++n) yy += Cm[b * dstate + n] * state[c * dstate + n];
    if (Dskip) yy += Dskip[d] * u;
    if (z) yy *= silu(z[c]);
    y[c] = yy;
  }
}

/*
 * Backward pass of the selective scan (training): the gradients of a scalar loss L through
 * oracle_selective_scan with the scan input u given directly (no conv) and the Euler rule,
 * given dout = dL/dout [b,d,t] and dh_last = dL/dh_last [b,d,n] (NULL: 0). The backward pass
 * is the adjoint of the recurrence ("Mamba (Selective State-Space Model)",
 * gunjandhanuka.github.io, "Cost of selectivity": training runs through the parallel scan); every line
 * below is the chain rule applied to one line of the forward definition.
 *   forward:  Delta_t = softplus(v_t), v_t = delta_t + bias;  Abar_t[n] = exp(Delta_t A[n]);
 *             h_t[n] = Abar_t[n] h_{t-1}[n] + Delta_t B_t[n] u_t;  y_t = sum_n C_t[n] h_t[n] + D u_t;
 *             out_t = y_t silu(z_t)
 *   adjoint:  g_t[n] = dL/dh_t[n] = Abar_{t+1}[n] g_{t+1}[n] + C_t[n] dy_t,  g_L = dh_last
 *   dy_t = dout_t silu(z_t);  dz_t = dout_t y_t silu'(z_t),  silu'(z) = s(z) (1 + z (1 - s(z)))
 *   dC_t[n] += dy_t h_t[n];  dB_t[n] += g_t[n] Delta_t u_t      (summed over channels d)
 *   du_t = D dy_t + sum_n g_t[n] Delta_t B_t[n]
 *   dDelta_t = sum_n g_t[n] (A[n] Abar_t[n] h_{t-1}[n] + B_t[n] u_t)
 *   dA[n] += g_t[n] Delta_t Abar_t[n] h_{t-1}[n];  dD += dy_t u_t   (summed over b and t)
 *   ddelta_t = dDelta_t sigmoid(v_t) (softplus on) or dDelta_t;  ddelta_bias += ddelta_t
 *   dh0[n] = Abar_0[n] g_0[n]
 * Outputs: du, ddelta [b,d,t]; dz [b,d,t] (when z is given); dA [d,n]; dB, dC [b,n,t];
 * dD, ddelta_bias [d]; dh0 [b,d,n]. All are written (not accumulated into).
 */
void oracle_selective_scan_bwd(const double* u, const double* delta, const double* A, const double* Bm,
                               const double* Cm, const double* Dskip, const double* z, const double* delta_bias,
                               int delta_softplus, const double* h0, const double* dout, const double* dh_last,
                               double* du, double* ddelta, double* dz, double* dA, double* dB, double* dC,
                               double* dD, double* ddelta_bias, double* dh0, long batch, long dim, long seqlen,
                               long dstate, int nthreads) {
  long nch = batch * dim;
  long NL = dstate * seqlen;
  /* per-channel contributions, summed below in a fixed order */
  double* cA = (double*)calloc((size_t)(nch * dstate), sizeof(double));
  double* cD = (double*)calloc((size_t)nch, sizeof(double));
  double* cbias = (double*)calloc((size_t)nch, sizeof(double));
  double* cB = (double*)calloc((size_t)(nch * NL > 0 ? nch * NL : 1), sizeof(double));
  double* cC = (double*)calloc((size_t)(nch * NL > 0 ? nch * NL : 1), sizeof(double));
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
  for (long c = 0; c < nch; ++c) {
    long b = c / dim, d = c % dim;
    const double* uc = u + c * seqlen;
    double* hs = (double*)malloc(sizeof(double) * (size_t)((seqlen + 1) * dstate)); /* h_{-1} .. h_{L-1} */
    double* Dl = (double*)malloc(sizeof(double) * (size_t)(seqlen > 0 ? seqlen : 1));
    double* sg = (double*)malloc(sizeof(double) * (size_t)(seqlen > 0 ? seqlen : 1));
    double* g = (double*)malloc(sizeof(double) * (size_t)dstate);
    /* forward, keeping every state */
    for (long n = 0; n < dstate; ++n) hs[n] = h0 ? h0[c * dstate + n] : 0.0;
    for (long t = 0; t < seqlen; ++t) {
      double v = delta[c * seqlen + t] + (delta_bias ? delta_bias[d] : 0.0);
      Dl[t] = delta_softplus ? softplus(v) : v;
      sg[t] = delta_softplus ? 1.0 / (1.0 + exp(-v)) : 1.0; /* dDelta/dv */
      for (long n = 0; n < dstate; ++n) {
        double Abar = exp(Dl[t] * A[d * dstate + n]);
        hs[(t + 1) * dstate + n] = Abar * hs[t * dstate + n] + Dl[t] * Bm[(b * dstate + n) * seqlen + t] * uc[t];
      }
    }
    /* backward */
    for (long n = 0; n < dstate; ++n) g[n] = dh_last ? dh_last[c * dstate + n] : 0.0;
    for (long t = seqlen - 1; t >= 0; --t) {
      const double* ht = hs + (t + 1) * dstate;
      const double* hp = hs + t * dstate;
      double y = 0.0;
      for (long n = 0; n < dstate; ++n) y += Cm[(b * dstate + n) * seqlen + t] * ht[n];
      if (Dskip) y += Dskip[d] * uc[t];
      double dy = dout[c * seqlen + t];
      if (z) {
        double zz = z[c * seqlen + t];
        double s = 1.0 / (1.0 + exp(-zz));
        dz[c * seqlen + t] = dout[c * seqlen + t] * y * s * (1.0 + zz * (1.0 - s));
        dy = dout[c * seqlen + t] * zz * s;
      }
      double dut = Dskip ? Dskip[d] * dy : 0.0;
      double dDel = 0.0;
      for (long n = 0; n < dstate; ++n) {
        double Bt = Bm[(b * dstate + n) * seqlen + t];
        double Ct = Cm[(b * dstate + n) * seqlen + t];
        double An = A[d * dstate + n];
        double Abar = exp(Dl[t] * An);
        g[n] += Ct * dy;
        cC[c * NL + n * seqlen + t] = dy * ht[n];
        cB[c * NL + n * seqlen + t] = g[n] * Dl[t] * uc[t];
        dut += g[n] * Dl[t] * Bt;
        dDel += g[n] * (An * Abar * hp[n] + Bt * uc[t]);
        cA[c * dstate + n] += g[n] * Dl[t] * Abar * hp[n];
        g[n] = Abar * g[n];
      }
      du[c * seqlen + t] = dut;
      ddelta[c * seqlen + t] = dDel * sg[t];
      cbias[c] += dDel * sg[t];
      if (Dskip) cD[c] += dy * uc[t];
    }
    for (long n = 0; n < dstate; ++n) dh0[c * dstate + n] = g[n];
    free(hs);
    free(Dl);
    free(sg);
    free(g);
  }
  /* reductions: over b for the per-channel parameters, over d for B and C */
  for (long d = 0; d < dim; ++d) {
    double sD = 0.0, sb = 0.0;
    for (long b = 0; b < batch; ++b) {
      sD += cD[b * dim + d];
      sb += cbias[b * dim + d];
    }
    if (dD) dD[d] = sD;
    if (ddelta_bias) ddelta_bias[d] = sb;
    for (long n = 0; n < dstate; ++n) {
      double sA = 0.0;
      for (long b = 0; b < batch; ++b) sA += cA[(b * dim + d) * dstate + n];
      dA[d * dstate + n] = sA;
    }
  }
  for (long b = 0; b < batch; ++b)
    for (long i = 0; i < NL; ++i) {
      double sB = 0.0, sC = 0.0;
      for (long d = 0; d < dim; ++d) {
        sB += cB[(b * dim + d) * NL + i];
        sC += cC[(b * dim + d) * NL + i];
      }
      dB[b * NL + i] = sB;
      dC[b * NL + i] = sC;
    }
  free(cA);
  free(cD);
  free(cbias);
  free(cB);
  free(cC);
}

/*
 * Multi-head selective SSM with one scalar decay per head: the layer of the structured
 * state-space duality ("Mamba" (inferensys.com / ai360xpert.com pages), "Mamba-2 introduces the
 * Structured State Space Duality": multi-head SSM, every head with its own selective parameters;
 * the state dimension treated like a head dimension; "Mamba" (ozercemkelahmet.com), "Mamba-2 and
 * the dual view": the same layer written as a masked matrix product with a decaying mask). A
 * single decay per head and step is what makes that mask one matrix per head. For every batch
 * element b and head h, with a state H of P x N (head dim x state dim):
 *   Delta_t   = softplus(dt[b,t,h] + dt_bias[h])       (the raw sum when dt_softplus == 0)
 *   H_t[p][n] = exp(Delta_t A[h]) H_{t-1}[p][n] + Delta_t x[b,t,h,p] B[b,t,n],   H_{-1} = h0 or 0
 *   y[b,t,h,p] = sum_n C[b,t,n] H_t[p][n] + D[h] x[b,t,h,p]
 * B and C are shared by all heads (one group). Layouts: x, y [batch, L, H, P]; dt [batch, L, H];
 * B, C [batch, L, N]; A, D, dt_bias [H]; h0, h_last [batch, H, P, N]. With d = h*P + p this is the
 * selective scan above with A[d,n] = A[h], delta[b,d,t] = dt[b,t,h] and B, C transposed.
 */
void oracle_ssd(const double* x, const double* dt, const double* A, const double* Bm, const double* Cm,
                const double* Dskip, const double* dt_bias, int dt_softplus, const double* h0, double* y,
                double* h_last, long batch, long seqlen, long nheads, long headdim, long dstate, int nthreads) {
  long npairs = batch * nheads;
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
  for (long c = 0; c < npairs; ++c) {
    long b = c / nheads, h = c % nheads;
    double* H = (double*)malloc(sizeof(double) * (size_t)(headdim * dstate));
    for (long i = 0; i < headdim * dstate; ++i) H[i] = h0 ? h0[c * headdim * dstate + i] : 0.0;
    for (long t = 0; t < seqlen; ++t) {
      double v = dt[(b * seqlen + t) * nheads + h] + (dt_bias ? dt_bias[h] : 0.0);
      double Delta = dt_softplus ? softplus(v) : v;
      double a = exp(Delta * A[h]);
      const double* xt = x + ((b * seqlen + t) * nheads + h) * headdim;
      const double* Bt = Bm + (b * seqlen + t) * dstate;
      const double* Ct = Cm + (b * seqlen + t) * dstate;
      double* yt = y + ((b * seqlen + t) * nheads + h) * headdim;
      for (long p = 0; p < headdim; ++p) {
        double acc = 0.0;
        for (long n = 0; n < dstate; ++n) {
          double* hp = H + p * dstate + n;
          *hp = a * (*hp) + Delta * xt[p] * Bt[n];
          acc += Ct[n] * (*hp);
        }
        if (Dskip) acc += Dskip[h] * xt[p];
        yt[p] = acc;
      }
    }
    if (h_last)
      for (long i = 0; i < headdim * dstate; ++i) h_last[c * headdim * dstate + i] = H[i];
    free(H);
  }
}

int oracle_version(void) { return 1; }
