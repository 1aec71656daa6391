// state_update.cuh -- single-token recurrent decode step, fp32 state updated in place.
//
// For each (b, d):  dt = delta[b,d] (+ bias[d], then softplus, when asked)
//                   state[n] = exp(dt A[d,n]) state[n] + dt B[b,n] x
//                   y = (sum_n C[b,n] state[n] + D[d] x) * silu(z)
// ("8.7 State Space Models (Mamba)", section 5: O(1) work per generated token on a
//  fixed d*n state; "Mamba and State Space Models", "Selective scan pseudo-code",
//  one iteration of the loop body.)
//
// The step streams the whole state once (read + write, 16-byte vectors); it is bound
// by memory bandwidth, not arithmetic. Each thread keeps two 16-byte state vectors (8
// states) in flight: twice the bytes in flight per SM of one vector per thread, with
// every warp still reading one contiguous 1 KB run.
#pragma once

#include "common.cuh"

namespace ssm {

struct DecodeParams {
  float* state;
  const void* x;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* Dskip;  // nullable
  const void* z;       // nullable
  void* y;
  const float* delta_bias;  // nullable: added to delta
  int delta_softplus;       // 1: dt = softplus(delta + bias)
  int zoh;                  // 1: B-bar = (exp(dt A) - 1) / A B instead of dt B
  // Conv prologue (nullable conv_w = none): x is the conv input; the SSM input is
  // silu(conv_b + w0 cs0 + w1 cs1 + w2 cs2 + w3 x) with conv_state (batch, D, 3), I/O
  // type, the previous three inputs oldest first, shifted in place to (cs1, cs2, x).
  const float* conv_w;
  const float* conv_b;
  void* conv_state;
  int64_t batch, D;
};

// One thread per (b, d, group of 8 states; 4 for N = 4); the lanes of a channel are adjacent
// in the warp and combine their partial C.h with xor-shuffles.
// kExt: the step-size map, the zero-order hold and the conv prologue are compiled in;
// the plain step (all of them off) keeps the lean kernel (fewer registers, more resident
// threads for this latency-bound update).
template <typename T, typename TY, int N, bool kExt>
__global__ void __launch_bounds__(256) state_update_kernel(const DecodeParams p) {
  constexpr int SPT = N >= 8 ? 8 : 4;  // states per thread: two 16-byte vectors where N allows
  constexpr int LPC = N / SPT;
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t bd = gt / LPC;
  const int g = (int)(gt % LPC);
  const int64_t nbd = p.batch * p.D;
  const bool v = bd < nbd;
  const int64_t b = v ? bd / p.D : 0, d = v ? bd % p.D : 0;

  float acc = 0.f, x = 0.f;
  if (v) {
    const T* xp = static_cast<const T*>(p.x);
    const T* dp = static_cast<const T*>(p.delta);
    const T* Bp = static_cast<const T*>(p.B) + b * N + g * SPT;
    const T* Cp = static_cast<const T*>(p.C) + b * N + g * SPT;
    x = to_f32(xp[bd]);
    if (kExt && p.conv_w) {  // the block's causal conv + SiLU over (cs0, cs1, cs2, x)
      const T* cs = static_cast<const T*>(p.conv_state) + bd * 3;
      const float* w = p.conv_w + d * 4;
      float c = p.conv_b ? p.conv_b[d] : 0.f;
      c = fmaf(w[0], to_f32(cs[0]), c);
      c = fmaf(w[1], to_f32(cs[1]), c);
      c = fmaf(w[2], to_f32(cs[2]), c);
      c = fmaf(w[3], x, c);
      x = silu_precise(c);
    }
    float dt = to_f32(dp[bd]);
    if (kExt && p.delta_bias) dt += p.delta_bias[d];
    if (kExt && p.delta_softplus) dt = softplus_precise(dt);
    const float dx = dt * x;
    float4* sp = reinterpret_cast<float4*>(p.state + bd * N + g * SPT);
    const float4* ap = reinterpret_cast<const float4*>(p.A + d * N + g * SPT);
    float sv[SPT], av[SPT];
#pragma unroll
    for (int q = 0; q < SPT / 4; ++q) {
      const float4 s4 = sp[q], a4 = ap[q];
      sv[4 * q] = s4.x; sv[4 * q + 1] = s4.y; sv[4 * q + 2] = s4.z; sv[4 * q + 3] = s4.w;
      av[4 * q] = a4.x; av[4 * q + 1] = a4.y; av[4 * q + 2] = a4.z; av[4 * q + 3] = a4.w;
    }
#pragma unroll
    for (int k = 0; k < SPT; ++k) {
      const float a = decay<sizeof(T) == 4>(dt, av[k], av[k] * kLog2e);
      const float bx = (kExt && p.zoh) ? zoh_factor<sizeof(T) == 4>(dt, av[k]) * x : dx;  // B-bar u = bx B
      sv[k] = fmaf(a, sv[k], bx * to_f32(Bp[k]));
      acc = fmaf(to_f32(Cp[k]), sv[k], acc);
    }
#pragma unroll
    for (int q = 0; q < SPT / 4; ++q) sp[q] = make_float4(sv[4 * q], sv[4 * q + 1], sv[4 * q + 2], sv[4 * q + 3]);
  }
#pragma unroll
  for (int off = LPC / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (kExt) __syncwarp();  // every lane of a channel has read the conv state before it is shifted
  if (kExt && v && g == 0 && p.conv_w) {
    T* cs = static_cast<T*>(p.conv_state) + bd * 3;
    const T c1 = cs[1], c2 = cs[2];
    cs[0] = c1;
    cs[1] = c2;
    cs[2] = static_cast<const T*>(p.x)[bd];
  }
  if (v && g == 0) {
    float out = acc;
    if (p.Dskip) out = fmaf(p.Dskip[d], x, out);
    if (p.z) out *= silu_precise(to_f32(static_cast<const T*>(p.z)[bd]));
    static_cast<TY*>(p.y)[bd] = from_f32<TY>(out);
  }
}

}  // namespace ssm
