/*
 * ssm_oracle.c -- the fp64 sequential oracle declared in ssm_oracle.h.
 *
 * TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU-baseline leg of the bench).
 * Written from the definition, step by step in the pages' order, with no blocking,
 * fusion or reordering: one (batch, channel) recurrence at a time, t ascending,
 * states n ascending. Threads only split independent (batch, channel) recurrences.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -o libssm_oracle.so ssm_oracle.c -lm -lpthread
 *
 * SSM_ORACLE_PLANT=k (compile-time, tests only) plants one deliberate mistake so the
 * pin tests can show that each kind of mistake is caught; the default build plants none.
 */
#include "ssm_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <unistd.h>

#ifndef SSM_ORACLE_PLANT
#define SSM_ORACLE_PLANT 0
#endif

/* Softplus: log(1 + exp(r)), the positivity map for the step size ("Mamba and State
 * Space Models", "Discretization and initialization details"). Written in the
 * overflow-free form; both branches equal log(1 + exp(r)) exactly in real arithmetic. */
double ssm_oracle_softplus(double r) {
  if (r > 0.0) return r + log1p(exp(-r));
  return log1p(exp(r));
}

/* SiLU / swish gate z * sigmoid(z) ("8.7 State Space Models (Mamba)", section 6;
 * "Mamba and State Space Models", "The Mamba Block": multiply by SiLU of the z branch). */
double ssm_oracle_silu(double z) {
#if SSM_ORACLE_PLANT == 5
  return 1.0 / (1.0 + exp(-z)); /* planted: sigmoid instead of SiLU */
#else
  return z / (1.0 + exp(-z));
#endif
}

/* B-bar factor of the exact zero-order hold for one diagonal entry a of A:
 * (delta a)^-1 (exp(delta a) - 1) delta = (exp(delta a) - 1) / a ("Arch 02: Mamba SSM",
 * zero-order-hold discretisation; "8.7 State Space Models (Mamba)", section 3), with
 * its limit delta at a = 0. */
static double zoh_factor(double dt, double a) {
#if SSM_ORACLE_PLANT == 16
  return a != 0.0 ? expm1(dt * a) : dt; /* planted: the 1 / a of the hold dropped */
#else
  return a != 0.0 ? expm1(dt * a) / a : dt;
#endif
}

typedef struct {
  int64_t batch, L, D, N;
  const double *u, *delta, *A, *B, *C, *Dskip, *z, *delta_bias, *h0;
  int delta_softplus, zoh;
  double *y, *last_state;
  int64_t ch_begin, ch_end; /* flattened channel range b*D + d */
} fwd_job_t;

/* One channel's recurrence, exactly the sequential definition:
 *   "Mamba and State Space Models", "Selective scan pseudo-code" (loop over t:
 *   dA = exp(delta*A); dB = delta*B; h = dA*h + dB*x; y = sum_n h*C), plus the
 *   D skip of the continuous form y = Cx + Du ("Arch 02: Mamba SSM") and the
 *   SiLU(z) output gate ("8.7 State Space Models (Mamba)", section 6). */
static void fwd_channel(const fwd_job_t* j, int64_t b, int64_t d, double* h) {
  const int64_t L = j->L, D = j->D, N = j->N;
  for (int64_t n = 0; n < N; ++n) h[n] = j->h0 ? j->h0[(b * D + d) * N + n] : 0.0; /* h(0) = 0 */
  for (int64_t t = 0; t < L; ++t) {
    const int64_t ix = (b * L + t) * D + d;  /* (batch, L, D) */
    const int64_t ixn = (b * L + t) * N;     /* (batch, L, N) */
    double r = j->delta[ix];
#if SSM_ORACLE_PLANT == 4
    double dt = j->delta_softplus ? ssm_oracle_softplus(r) : r; /* planted: bias after softplus */
    if (j->delta_bias) dt += j->delta_bias[d];
#else
    if (j->delta_bias) r += j->delta_bias[d];
#if SSM_ORACLE_PLANT == 9
    double dt = r; /* planted: softplus skipped */
#else
    double dt = j->delta_softplus ? ssm_oracle_softplus(r) : r;
#endif
#endif
    const double x = j->u[ix];
    double acc = 0.0;
    for (int64_t n = 0; n < N; ++n) {
#if SSM_ORACLE_PLANT == 8
      const double An = j->A[n * D + d]; /* planted: A indexed (n, d) instead of (d, n) */
#else
      const double An = j->A[d * N + n];
#endif
#if SSM_ORACLE_PLANT == 2
      const double dA = exp(-dt * An);              /* planted: wrong sign in the exponent */
#else
      const double dA = exp(dt * An);               /* A-bar = exp(Delta * A) */
#endif
#if SSM_ORACLE_PLANT == 6
      const double dB = j->B[ixn + n];              /* planted: B-bar = B (Delta dropped) */
#elif SSM_ORACLE_PLANT == 3
      const double dB = dt * j->C[ixn + n];         /* planted: B and C swapped */
#else
      const double dB = j->zoh ? zoh_factor(dt, An) * j->B[ixn + n]  /* B-bar, exact ZOH */
                               : dt * j->B[ixn + n];                 /* B-bar = Delta * B */
#endif
#if SSM_ORACLE_PLANT == 7
      acc += j->C[ixn + n] * h[n];                  /* planted: read out before the update */
      h[n] = dA * h[n] + dB * x;
#elif SSM_ORACLE_PLANT == 3
      h[n] = dA * h[n] + dB * x;
      acc += j->B[ixn + n] * h[n];
#else
      h[n] = dA * h[n] + dB * x;                    /* h_t = A-bar h_{t-1} + B-bar u_t */
      acc += j->C[ixn + n] * h[n];                  /* y_t = C_t . h_t */
#endif
    }
#if SSM_ORACLE_PLANT == 1
    double v = acc;                                 /* planted: D skip dropped */
#else
    double v = acc + (j->Dskip ? j->Dskip[d] * x : 0.0);
#endif
    j->y[ix] = j->z ? v * ssm_oracle_silu(j->z[ix]) : v;
  }
  if (j->last_state)
    for (int64_t n = 0; n < N; ++n) j->last_state[(b * D + d) * N + n] = h[n];
}

static void* fwd_worker(void* arg) {
  const fwd_job_t* j = (const fwd_job_t*)arg;
  double* h = (double*)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
  if (!h) return (void*)1;
  for (int64_t c = j->ch_begin; c < j->ch_end; ++c) fwd_channel(j, c / j->D, c % j->D, h);
  free(h);
  return NULL;
}

static int resolve_threads(int nthreads, int64_t work) {
  if (nthreads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = n > 0 ? (int)n : 1;
  }
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > work) nthreads = work > 0 ? (int)work : 1;
  return nthreads;
}

int ssm_oracle_fwd(int64_t batch, int64_t L, int64_t D, int64_t N,
                   const double* u, const double* delta, const double* A,
                   const double* B, const double* C, const double* Dskip,
                   const double* z, const double* delta_bias, int delta_softplus,
                   const double* h0, double* y, double* last_state, int nthreads) {
  return ssm_oracle_fwd_ex(batch, L, D, N, u, delta, A, B, C, Dskip, z, delta_bias, delta_softplus, 0, h0, y,
                           last_state, nthreads);
}

int ssm_oracle_fwd_ex(int64_t batch, int64_t L, int64_t D, int64_t N,
                      const double* u, const double* delta, const double* A,
                      const double* B, const double* C, const double* Dskip,
                      const double* z, const double* delta_bias, int delta_softplus, int zoh,
                      const double* h0, double* y, double* last_state, int nthreads) {
  if (batch < 0 || L < 0 || D < 0 || N <= 0) return -1;
  const int64_t nch = batch * D;
  if (nch == 0) return 0;
  if ((L > 0 && (!u || !delta || !B || !C || !y)) || !A) return -1;
  fwd_job_t base = {batch, L, D, N, u, delta, A, B, C, Dskip, z, delta_bias, h0,
                    delta_softplus, zoh, y, last_state, 0, 0};
  int nt = resolve_threads(nthreads, nch);
  if (nt == 1) {
    base.ch_begin = 0;
    base.ch_end = nch;
    return fwd_worker(&base) ? -1 : 0;
  }
  pthread_t tid[256];
  fwd_job_t jobs[256];
  int started = 0, rc = 0;
  for (int i = 0; i < nt; ++i) {
    jobs[i] = base;
    jobs[i].ch_begin = nch * i / nt;
    jobs[i].ch_end = nch * (i + 1) / nt;
    if (pthread_create(&tid[i], NULL, fwd_worker, &jobs[i]) != 0) {
      rc = -1;
      break;
    }
    ++started;
  }
  for (int i = 0; i < started; ++i) {
    void* ret = NULL;
    pthread_join(tid[i], &ret);
    if (ret) rc = -1;
  }
  return rc;
}

/* One recurrent step per (batch, channel): the O(1)-per-token inference update
 * ("8.7 State Space Models (Mamba)", section 5; "Mamba and State Space Models",
 * "Selective scan pseudo-code" body for a single t), continuing from a given state. */
int ssm_oracle_state_update_ex(int64_t batch, int64_t D, int64_t N, double* state,
                               const double* x, const double* delta, const double* A,
                               const double* B, const double* C, const double* Dskip,
                               const double* z, const double* delta_bias, int delta_softplus,
                               int zoh, double* y) {
  if (batch < 0 || D < 0 || N <= 0) return -1;
  if (batch * D == 0) return 0;
  if (!state || !x || !delta || !A || !B || !C || !y) return -1;
  for (int64_t b = 0; b < batch; ++b) {
    for (int64_t d = 0; d < D; ++d) {
      /* the forward pass's step-size map, when asked: dt = softplus(delta + bias) */
      const double r = delta[b * D + d] + (delta_bias ? delta_bias[d] : 0.0);
      const double dt = delta_softplus ? ssm_oracle_softplus(r) : r;
      const double xv = x[b * D + d];
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        double* s = &state[(b * D + d) * N + n];
        const double dA = exp(dt * A[d * N + n]);
        const double dB = (zoh ? zoh_factor(dt, A[d * N + n]) : dt) * B[b * N + n];
        *s = dA * (*s) + dB * xv;
        acc += C[b * N + n] * (*s);
      }
      double v = acc + (Dskip ? Dskip[d] * xv : 0.0);
      y[b * D + d] = z ? v * ssm_oracle_silu(z[b * D + d]) : v;
    }
  }
  return 0;
}

int ssm_oracle_state_update(int64_t batch, int64_t D, int64_t N, double* state,
                            const double* x, const double* delta, const double* A,
                            const double* B, const double* C, const double* Dskip,
                            const double* z, double* y) {
  return ssm_oracle_state_update_ex(batch, D, N, state, x, delta, A, B, C, Dskip, z, NULL, 0, 0, y);
}

/* Causal depthwise convolution of width 4 followed by SiLU: the step before the SSM in
 * the Mamba block ("Mamba and State Space Models", "The Mamba Block": depthwise Conv1d,
 * kernel 4, then SiLU; "Mamba and State Space Models" model card: d_conv = 4). For every
 * (b, t, d):  u = silu(bias[d] + sum_{k=0..3} w[d,k] * x[b, t-3+k, d]), where an input
 * before t = 0 is conv_state[b, d, 3 + (t-3+k)] (the three inputs that preceded the
 * sequence, oldest first), or 0 when conv_state is NULL. */
int ssm_oracle_conv1d_silu(int64_t batch, int64_t L, int64_t D, const double* x, const double* w,
                           const double* bias, const double* conv_state, double* u) {
  if (batch < 0 || L < 0 || D < 0) return -1;
  if (batch * L * D == 0) return 0;
  if (!x || !w || !u) return -1;
  for (int64_t b = 0; b < batch; ++b)
    for (int64_t t = 0; t < L; ++t)
      for (int64_t d = 0; d < D; ++d) {
        double acc = bias ? bias[d] : 0.0;
        for (int64_t k = 0; k < 4; ++k) {
          const int64_t s = t - 3 + k;
          double xv;
          if (s >= 0)
            xv = x[(b * L + s) * D + d];
          else
            xv = conv_state ? conv_state[(b * D + d) * 3 + (3 + s)] : 0.0;
#if SSM_ORACLE_PLANT == 15
          acc += w[d * 4 + (3 - k)] * xv; /* planted: taps in reverse order */
#else
          acc += w[d * 4 + k] * xv;
#endif
        }
        u[(b * L + t) * D + d] = ssm_oracle_silu(acc);
      }
  return 0;
}

/* d silu(z) / dz = sigma(z) (1 + z (1 - sigma(z))). */
static double silu_grad(double z) {
  const double sg = 1.0 / (1.0 + exp(-z));
  return sg * (1.0 + z * (1.0 - sg));
}

/* Backward pass of ssm_oracle_fwd (Delta * B discretisation), the chain rule applied to
 * the recurrence in reverse time with every h_t kept from a forward sweep. For one
 * channel, with g = dL/dh_t (starting from dlast at t = L-1):
 *   dv   = dy_t silu(z_t)              dz_t = dy_t v_t silu'(z_t)      dD += dv u_t
 *   g   += dv C_t                      dC_t += dv h_t
 *   dB_t += g dt u_t                   du_t  = dv D + sum_n g dt B_t
 *   d(dt) = sum_n g (B_t u_t + A a_t h_{t-1})      dA += g a_t h_{t-1} dt
 *   ddelta_t = d(dt) * (softplus ? sigmoid(r_t) : 1)                  dbias += ddelta_t
 *   g   *= a_t                          (dL/dh_{t-1}; after t = 0 it is dL/dh0)
 * dA, dB, dC, dD, dbias accumulate over channels and batch rows and are zeroed here. */
int ssm_oracle_bwd(int64_t batch, int64_t L, int64_t D, int64_t N,
                   const double* u, const double* delta, const double* A,
                   const double* B, const double* C, const double* Dskip,
                   const double* z, const double* delta_bias, int delta_softplus,
                   const double* h0, const double* dy, const double* dlast,
                   double* du, double* ddelta, double* dA, double* dB, double* dC,
                   double* dD, double* dz, double* dbias, double* dh0) {
  if (batch < 0 || L < 0 || D < 0 || N <= 0) return -1;
  if (!A || !dA) return -1;
  if (L > 0 && (!u || !delta || !B || !C || !dy || !du || !ddelta || !dB || !dC)) return -1;
  for (int64_t i = 0; i < D * N; ++i) dA[i] = 0.0;
  for (int64_t i = 0; i < batch * L * N; ++i) dB[i] = dC[i] = 0.0;
  if (dD) for (int64_t i = 0; i < D; ++i) dD[i] = 0.0;
  if (dbias) for (int64_t i = 0; i < D; ++i) dbias[i] = 0.0;
  double* hs = (double*)malloc(sizeof(double) * (size_t)((L + 1) * N)); /* h_{-1} .. h_{L-1} */
  double* dts = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  double* rs = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  double* g = (double*)malloc(sizeof(double) * (size_t)N);
  if (!hs || !dts || !rs || !g) {
    free(hs); free(dts); free(rs); free(g);
    return -1;
  }
  for (int64_t b = 0; b < batch; ++b) {
    for (int64_t d = 0; d < D; ++d) {
      /* forward sweep, keeping every state */
      for (int64_t n = 0; n < N; ++n) hs[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;
      for (int64_t t = 0; t < L; ++t) {
        const int64_t ix = (b * L + t) * D + d, ixn = (b * L + t) * N;
        const double r = delta[ix] + (delta_bias ? delta_bias[d] : 0.0);
        const double dt = delta_softplus ? ssm_oracle_softplus(r) : r;
        rs[t] = r;
        dts[t] = dt;
        for (int64_t n = 0; n < N; ++n)
          hs[(t + 1) * N + n] = exp(dt * A[d * N + n]) * hs[t * N + n] + dt * B[ixn + n] * u[ix];
      }
      /* reverse sweep */
      for (int64_t n = 0; n < N; ++n) g[n] = dlast ? dlast[(b * D + d) * N + n] : 0.0;
      for (int64_t t = L - 1; t >= 0; --t) {
        const int64_t ix = (b * L + t) * D + d, ixn = (b * L + t) * N;
        const double dt = dts[t], x = u[ix];
        const double* ht = &hs[(t + 1) * N];
        const double* hp = &hs[t * N];
        double v = Dskip ? Dskip[d] * x : 0.0;
        for (int64_t n = 0; n < N; ++n) v += C[ixn + n] * ht[n];
        double dv = dy[ix];
        if (z) {
          dz[ix] = dy[ix] * v * silu_grad(z[ix]);
          dv = dy[ix] * ssm_oracle_silu(z[ix]);
        }
        if (dD) dD[d] += dv * x;
        double dux = Dskip ? dv * Dskip[d] : 0.0, ddt = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          const double An = A[d * N + n];
          const double a = exp(dt * An);
          g[n] += dv * C[ixn + n];
#if SSM_ORACLE_PLANT == 11
          g[n] *= a; /* planted: g carried to step t-1 before its use at step t */
#endif
#if SSM_ORACLE_PLANT == 12
          dC[ixn + n] += dv * hp[n]; /* planted: dC from h_{t-1} instead of h_t */
#else
          dC[ixn + n] += dv * ht[n];
#endif
          dB[ixn + n] += g[n] * dt * x;
          dux += g[n] * dt * B[ixn + n];
#if SSM_ORACLE_PLANT == 10
          ddt += g[n] * (B[ixn + n] * x); /* planted: the A a h_{t-1} term of d(dt) dropped */
#else
          ddt += g[n] * (B[ixn + n] * x + An * a * hp[n]);
#endif
          dA[d * N + n] += g[n] * a * hp[n] * dt;
#if SSM_ORACLE_PLANT != 11
          g[n] *= a;
#endif
        }
        du[ix] = dux;
        const double dr = delta_softplus ? ddt / (1.0 + exp(-rs[t])) : ddt;
        ddelta[ix] = dr;
        if (dbias) dbias[d] += dr;
      }
      if (dh0)
        for (int64_t n = 0; n < N; ++n) dh0[(b * D + d) * N + n] = g[n];
    }
  }
  free(hs); free(dts); free(rs); free(g);
  return 0;
}

/* Mamba-2 SSD recurrence (scalar decay per head): for every batch row b and head h, with
 * the (P x N) state S starting at h0 (or 0) and g = h / (H / G) the B/C group:
 *   dt  = delta[b,t,h] + dt_bias[h], then softplus when dt_softplus
 *   S   = exp(dt A[h]) S + dt x[b,t,h,:] B[b,t,g,:]^T
 *   y[b,t,h,:] = S C[b,t,g,:] + D[h] x[b,t,h,:]
 * ("8.7 State Space Models (Mamba)" and "Mamba and State Space Models", "Mamba-2 and
 * State Space Duality": A-bar_t = a_t I per head; B-bar = Delta B as in Mamba). */
int ssm_oracle_ssd_fwd(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G,
                       const double* x, const double* delta, const double* A, const double* B,
                       const double* C, const double* Dskip, const double* dt_bias, int dt_softplus,
                       const double* h0, double* y, double* last_state) {
  if (batch < 0 || L < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0) return -1;
  if (batch * H == 0) return 0;
  if (!A || (L > 0 && (!x || !delta || !B || !C || !y))) return -1;
  double* S = (double*)malloc(sizeof(double) * (size_t)(P * N));
  if (!S) return -1;
  for (int64_t b = 0; b < batch; ++b) {
    for (int64_t h = 0; h < H; ++h) {
#if SSM_ORACLE_PLANT == 13
      const int64_t g = h % G; /* planted: heads assigned to groups round-robin */
#else
      const int64_t g = h / (H / G);
#endif
      for (int64_t i = 0; i < P * N; ++i) S[i] = h0 ? h0[(b * H + h) * P * N + i] : 0.0;
      for (int64_t t = 0; t < L; ++t) {
        double r = delta[(b * L + t) * H + h] + (dt_bias ? dt_bias[h] : 0.0);
        const double dt = dt_softplus ? ssm_oracle_softplus(r) : r;
        const double a = exp(dt * A[h]);
        const double* xt = &x[((b * L + t) * H + h) * P];
        const double* Bt = &B[((b * L + t) * G + g) * N];
        const double* Ct = &C[((b * L + t) * G + g) * N];
        double* yt = &y[((b * L + t) * H + h) * P];
        for (int64_t p = 0; p < P; ++p) {
          double acc = 0.0;
          for (int64_t n = 0; n < N; ++n) {
#if SSM_ORACLE_PLANT == 14
            S[p * N + n] = a * (S[p * N + n] + dt * xt[p] * Bt[n]); /* planted: input decayed too */
#else
            S[p * N + n] = a * S[p * N + n] + dt * xt[p] * Bt[n];
#endif
            acc += S[p * N + n] * Ct[n];
          }
          yt[p] = acc + (Dskip ? Dskip[h] * xt[p] : 0.0);
        }
      }
      if (last_state)
        for (int64_t i = 0; i < P * N; ++i) last_state[(b * H + h) * P * N + i] = S[i];
    }
  }
  free(S);
  return 0;
}
