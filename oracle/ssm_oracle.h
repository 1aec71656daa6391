/*
 * ssm_oracle.h -- plain, slow, sequential fp64 CPU oracle for the Mamba selective
 * scan (forward) and the single-token recurrent state update.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link, load or
 * call this code: only the tests, the smoke check and the bench's CPU-baseline leg
 * use it. It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (all arrays fp64, dense, row-major, channel index fastest):
 *
 *   for every batch row b and channel d, starting from h = h0 (or 0):
 *     for t = 0 .. L-1:
 *       r     = delta[b,t,d] + delta_bias[d]                  (bias 0 if absent)
 *       dt    = delta_softplus ? log(1 + exp(r)) : r
 *       for n: h[n] = exp(dt * A[d,n]) * h[n] + dt * B[b,t,n] * u[b,t,d]
 *       v     = sum_n C[b,t,n] * h[n] + Dskip[d] * u[b,t,d]   (skip 0 if absent)
 *       y     = z present ? v * z / (1 + exp(-z[b,t,d])) : v
 *     last_state[b,d,:] = h
 *
 * Sources (page title, section):
 *  - "Mamba and State Space Models" (vanos001 placement-prep chapter), section
 *    "Selective scan pseudo-code": the sequential loop over t with
 *    dA = exp(delta*A), dB = delta*B, h = dA*h + dB*x, y = (h*C).sum over N.
 *  - same chapter, "Discretization and initialization details": A-bar = exp(Delta*A)
 *    with B-bar simplified to Delta*B; Delta = softplus(W x + b_Delta), the bias
 *    added before the softplus.
 *  - "Arch 02: Mamba SSM" deck, continuous form y = Cx + Du (the D skip) and the
 *    selective-SSM block (B, C per token (B,L,N); Delta per token and channel).
 *  - "8.7 State Space Models (Mamba)", section 6 "The block": the SSM output is
 *    multiplied elementwise by SiLU of the other half (the z gate); section 2.1: h(0)=0.
 *  - "Mamba and State Space Models", "Common Pitfalls": the state after a prefix is
 *    reusable (h0 argument / last_state output; decode continues from it).
 */
#ifndef SSM_ORACLE_H
#define SSM_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Softplus in a numerically stable form: r + log1p(exp(-r)) for r > 0, else log1p(exp(r)). */
double ssm_oracle_softplus(double r);
/* SiLU (swish): z * sigmoid(z) = z / (1 + exp(-z)). */
double ssm_oracle_silu(double z);

/*
 * Forward selective scan.
 *   u, delta, z, y : (batch, L, D)      B, C : (batch, L, N)
 *   A : (D, N)     Dskip, delta_bias : (D)     h0, last_state : (batch, D, N)
 * Nullable: Dskip, z, delta_bias, h0, last_state. y must not alias an input.
 * nthreads <= 0 uses every online CPU. Returns 0 on success, -1 on bad arguments.
 */
int ssm_oracle_fwd(int64_t batch, int64_t L, int64_t D, int64_t N,
                   const double* u, const double* delta, const double* A,
                   const double* B, const double* C, const double* Dskip,
                   const double* z, const double* delta_bias, int delta_softplus,
                   const double* h0, double* y, double* last_state, int nthreads);

/*
 * The same with a choice of B-bar: zoh = 0 takes Delta * B (as above); zoh = 1 the exact
 * zero-order hold of the continuous system, B-bar[n] = (exp(Delta A[d,n]) - 1) / A[d,n]
 * * B[b,t,n] (Delta * B[b,t,n] where A[d,n] = 0).
 */
int ssm_oracle_fwd_ex(int64_t batch, int64_t L, int64_t D, int64_t N,
                      const double* u, const double* delta, const double* A,
                      const double* B, const double* C, const double* Dskip,
                      const double* z, const double* delta_bias, int delta_softplus, int zoh,
                      const double* h0, double* y, double* last_state, int nthreads);

/*
 * One recurrent decode step, in place on state (batch, D, N):
 *   x, delta, z, y : (batch, D)   B, C : (batch, N)   A : (D, N)   Dskip : (D)
 * delta is the final step size (no bias, no softplus). Nullable: Dskip, z.
 * Returns 0 on success, -1 on bad arguments.
 */
int ssm_oracle_state_update(int64_t batch, int64_t D, int64_t N, double* state,
                            const double* x, const double* delta, const double* A,
                            const double* B, const double* C, const double* Dskip,
                            const double* z, double* y);

/*
 * The same step with the forward pass's step-size map applied first:
 *   dt = delta[b,d] + delta_bias[d] (bias 0 if absent), then log(1 + exp(dt)) when
 *   delta_softplus is 1; and B-bar chosen as in ssm_oracle_fwd_ex (zoh).
 */
int ssm_oracle_state_update_ex(int64_t batch, int64_t D, int64_t N, double* state,
                               const double* x, const double* delta, const double* A,
                               const double* B, const double* C, const double* Dskip,
                               const double* z, const double* delta_bias, int delta_softplus,
                               int zoh, double* y);

/*
 * Causal depthwise convolution (width 4) + SiLU, the step before the SSM in the block:
 *   u[b,t,d] = silu(bias[d] + sum_{k=0..3} w[d,k] * x[b,t-3+k,d])
 * x, u : (batch, L, D)   w : (D, 4)   bias : (D), nullable
 * conv_state : (batch, D, 3), nullable -- the three inputs before x[b,0,d], oldest first
 * (zeros if NULL). Returns 0 on success, -1 on bad arguments.
 */
int ssm_oracle_conv1d_silu(int64_t batch, int64_t L, int64_t D, const double* x, const double* w,
                           const double* bias, const double* conv_state, double* u);

/*
 * Backward pass of ssm_oracle_fwd (Delta * B discretisation): given dy (batch, L, D) and
 * dlast (batch, D, N, nullable = 0), the gradients of sum(dy * y) + sum(dlast * last_state)
 * with respect to every input: du, ddelta, dz (batch, L, D); dB, dC (batch, L, N);
 * dA (D, N); dD, dbias (D); dh0 (batch, D, N). dD, dz, dbias, dh0 are nullable (needed
 * only when Dskip, z, delta_bias, h0 are given). Single-threaded; keeps every state of a
 * channel, so it is meant for small problems. Returns 0, or -1 on bad arguments.
 */
int ssm_oracle_bwd(int64_t batch, int64_t L, int64_t D, int64_t N,
                   const double* u, const double* delta, const double* A,
                   const double* B, const double* C, const double* Dskip,
                   const double* z, const double* delta_bias, int delta_softplus,
                   const double* h0, const double* dy, const double* dlast,
                   double* du, double* ddelta, double* dA, double* dB, double* dC,
                   double* dD, double* dz, double* dbias, double* dh0);

/*
 * Mamba-2 SSD (scalar decay per head, P x N state per head), sequential:
 *   x, y : (batch, L, H, P)   delta : (batch, L, H)   A, Dskip, dt_bias : (H)
 *   B, C : (batch, L, G, N), head h uses group h / (H / G)
 *   h0, last_state : (batch, H, P, N), nullable
 * Returns 0, or -1 on bad arguments.
 */
int ssm_oracle_ssd_fwd(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G,
                       const double* x, const double* delta, const double* A, const double* B,
                       const double* C, const double* Dskip, const double* dt_bias, int dt_softplus,
                       const double* h0, double* y, double* last_state);

#ifdef __cplusplus
}
#endif
#endif
