// scan_fwd.cuh -- fused selective-scan forward kernels.
//
// Per (batch b, channel d), from h = 0, for t = 0 .. L-1:
//   dt   = softplus(delta + bias)           (or delta + bias)
//   h[n] = exp(dt * A[d,n]) * h[n] + dt * u * B[t,n]
//   y    = (sum_n C[t,n] h[n] + D[d] u) * silu(z)
// ("Mamba and State Space Models", "Selective scan pseudo-code" and
//  "Discretization and initialization details"; "Arch 02: Mamba SSM", y = Cx + Du;
//  "8.7 State Space Models (Mamba)", section 6, the SiLU(z) gate.)
//
// The state h lives in fp32 registers for the whole sequence and never reaches
// global memory; only y and the final state are written ("Mamba and State Space
// Models", "Hardware-Aware Parallel Scan": kernel fusion, no intermediate h in HBM).
#pragma once

#include "common.cuh"

namespace ssm {

struct FwdParams {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* Dskip;       // nullable
  const void* z;            // nullable
  const float* delta_bias;  // nullable
  int delta_softplus;
  void* y;
  float* last_state;        // nullable
  const float* h0;          // nullable: start state (batch, D, N); zeros when null
  int zoh;                  // 1: B-bar = (exp(dt A) - 1) / A B (general kernel only)
  // Conv prologue (nullable conv_w = none): u then holds the conv input x and the SSM
  // input is silu(conv_b + sum_k conv_w[d,k] x[t-3+k]); conv_state (batch, D, 3), I/O
  // type, nullable: the three inputs before t = 0 (zeros when null).
  const float* conv_w;
  const float* conv_b;
  const void* conv_state;
  int64_t batch, L, D;
  // Sequence segments (channel kernel only): CTA z covers steps [z*seg_len, (z+1)*seg_len).
  // seg_len == L means one segment. seg_h0 (nullable): start state of each segment,
  // laid out [segment][batch][D][N]. seg_E / seg_P: outputs of the aggregate pass, same
  // layout: end state from a zero start and the decay product exp(A * sum of dt).
  int64_t seg_len;
  const float* seg_h0;
  float* seg_E;
  float* seg_P;
  // Segment scratch kept in the output (channel kernel): when seg_y is set, seg_h0 /
  // seg_E / seg_P are not used; the start state, end state and decay product of segment
  // s for channel d live in y itself, in column d of the segment's first rows (see
  // seg_slot), which the segment's own full pass overwrites with y afterwards.
  void* seg_y;
  int seg_y_bf16;
  // Failure detection (channel kernel): the limit of every bounded wait in cycles (0: the
  // default of about one second), and a fault-injection switch for tests: when set, the
  // TMA issuer issues no copy, so every wait for data runs out and reports its code.
  long long wait_cycles;
  int fault_skip_loads;
  // State checkpoints (channel kernel: the aggregate pass over one segment, or the full
  // pass of a training forward): when set, the state before every
  // kCkSteps-step chunk c of the sequence is written to ck[b][c][D][N] (f32), c < ck_nc.
  // The backward pass recomputes each chunk's states from these.
  float* ck;
  int64_t ck_nc;
};

// Segment scratch inside y: value `kind` (0 start state H, 1 end state E, 2 decay product
// P) of state n, channel d, batch row b, segment s sits in column d of y at rows
// s * seg_len + kind * N + n (fp32 y), or as two bf16-sized halves (high, low 16 bits of
// the fp32 value) at rows s * seg_len + 2 (kind * N + n) + {0, 1} (bf16 y). Every value
// of a channel stays in that channel's own column and segment, which only the CTA that
// owns both touches, so no two CTAs of a pass share scratch. Needs seg_len >= 6 N rows.
struct SegY {
  void* y;
  int bf16;
  int64_t L, D, seg_len;
  int N;
};
__device__ __forceinline__ void seg_slot_store(const SegY& q, int kind, int64_t s, int64_t b, int64_t d, int n,
                                               float v) {
  const int64_t r = s * q.seg_len + (int64_t)(kind * q.N + n) * (q.bf16 ? 2 : 1);
  if (q.bf16) {
    unsigned short* y = static_cast<unsigned short*>(q.y) + (b * q.L + r) * q.D + d;
    const uint32_t w = __float_as_uint(v);
    y[0] = (unsigned short)(w >> 16);
    y[q.D] = (unsigned short)(w & 0xffffu);
  } else {
    static_cast<float*>(q.y)[(b * q.L + r) * q.D + d] = v;
  }
}
__device__ __forceinline__ float seg_slot_load(const SegY& q, int kind, int64_t s, int64_t b, int64_t d, int n) {
  const int64_t r = s * q.seg_len + (int64_t)(kind * q.N + n) * (q.bf16 ? 2 : 1);
  if (q.bf16) {
    const unsigned short* y = static_cast<const unsigned short*>(q.y) + (b * q.L + r) * q.D + d;
    return __uint_as_float(((uint32_t)y[0] << 16) | (uint32_t)y[q.D]);
  }
  return static_cast<const float*>(q.y)[(b * q.L + r) * q.D + d];
}

// ------------------------------------------------------------------------------------
// Generic kernel: any D, any L, fp32 or bf16 I/O. Channel-parallel: a group of
// LPC = N / SPL adjacent lanes owns one channel, SPL states each, and walks the
// sequence in chunks of TC steps staged through shared memory:
//   stage  : u, z, (dt, dt*u) per (t, d) and B, C per (t, n) -> smem (fp32)
//   scan   : each lane updates its SPL states for every t, writes its partial C.h
//   finish : y = sum of partials + D u, gated, stored
// ------------------------------------------------------------------------------------
// kZOH: B-bar = (exp(dt A) - 1) / A B (zero-order hold) instead of dt B.
// kAgg: the aggregate pass of a segmented scan over CTA z's sequence segment (end state
// from zero and decay product into y's segment rows, see SegY; no outputs).
// Segments: blockIdx.z covers steps [z * seg_len, (z + 1) * seg_len); with seg_y set the
// full pass starts each segment from the start state the carry scan left in y.
template <typename T, typename TY, int N, int SPL, int DT, int TC, bool kZOH, bool kAgg = false>
__global__ void __launch_bounds__(DT*(N / SPL))
scan_fwd_generic(const FwdParams p) {
  constexpr int LPC = N / SPL;
  constexpr int NT = DT * LPC;
  __shared__ float sU[TC][DT];
  __shared__ float sZ[TC][DT];
  __shared__ float2 sDD[TC][DT];
  __shared__ float sB[TC][N];
  __shared__ float sC[TC][N];
  __shared__ float sP[TC][NT];

  const int tid = threadIdx.x;
  const int64_t b = blockIdx.y;
  const int64_t L = p.L, D = p.D;
  const int64_t d0 = (int64_t)blockIdx.x * DT;
  const int j = tid / LPC, g = tid % LPC;
  const int64_t dj = d0 + j;
  const bool vj = dj < D;

  const T* __restrict__ u = static_cast<const T*>(p.u) + b * L * D;
  const T* __restrict__ dl = static_cast<const T*>(p.delta) + b * L * D;
  const T* __restrict__ zp = p.z ? static_cast<const T*>(p.z) + b * L * D : nullptr;
  const T* __restrict__ Bp = static_cast<const T*>(p.B) + b * L * N;
  const T* __restrict__ Cp = static_cast<const T*>(p.C) + b * L * N;
  TY* __restrict__ y = static_cast<TY*>(p.y) + b * L * D;

  constexpr bool kAccurate = sizeof(T) == 4;  // fp32 I/O: near-correctly-rounded decay
  const int64_t seg = blockIdx.z;
  const int64_t seg_len = p.seg_y ? p.seg_len : L;
  const int64_t t_begin = seg * seg_len;
  const int64_t t_end = (t_begin + seg_len) < L ? (t_begin + seg_len) : L;
  const SegY sy{p.seg_y, p.seg_y_bf16, L, D, seg_len, N};
  double sdt = 0.0;  // kAgg: sum of dt over the segment
  float Av[SPL], A2[SPL], h[SPL];
#pragma unroll
  for (int k = 0; k < SPL; ++k) {
    Av[k] = vj ? p.A[dj * N + g * SPL + k] : 0.f;
    A2[k] = Av[k] * kLog2e;
    if (kAgg) h[k] = 0.f;
    else if (p.seg_y) h[k] = vj ? seg_slot_load(sy, 0, seg, b, dj, g * SPL + k) : 0.f;
    else h[k] = (vj && p.h0) ? p.h0[(b * D + dj) * N + g * SPL + k] : 0.f;
  }

  for (int64_t t0 = t_begin; t0 < t_end; t0 += TC) {
    const int tc = (int)((t_end - t0) < TC ? (t_end - t0) : TC);
    for (int i = tid; i < TC * DT; i += NT) {
      const int t = i / DT, jj = i % DT;
      const int64_t d = d0 + jj;
      float uu = 0.f, zz = 0.f, dt = 0.f;
      if (t < tc && d < D) {
        const int64_t ix = (t0 + t) * D + d;
        if (p.conv_w) {  // causal width-4 conv + SiLU of the input x (the block's prologue)
          float acc = p.conv_b ? p.conv_b[d] : 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int64_t s = t0 + t - 3 + k;
            float xv = 0.f;
            if (s >= 0)
              xv = to_f32(u[s * D + d]);
            else if (p.conv_state)
              xv = to_f32(static_cast<const T*>(p.conv_state)[(b * D + d) * 3 + 3 + s]);
            acc = fmaf(p.conv_w[d * 4 + k], xv, acc);
          }
          uu = silu_precise(acc);
        } else {
          uu = to_f32(u[ix]);
        }
        float r = to_f32(dl[ix]);
        if (p.delta_bias) r += p.delta_bias[d];
        dt = p.delta_softplus ? softplus_precise(r) : r;
        if (zp) zz = to_f32(zp[ix]);
      }
      sU[t][jj] = uu;
      sZ[t][jj] = zz;
      sDD[t][jj] = make_float2(dt, dt * uu);
    }
    for (int i = tid; i < TC * N; i += NT) {
      const int t = i / N, n = i % N;
      float bb = 0.f, cc = 0.f;
      if (t < tc) {
        const int64_t ix = (t0 + t) * N + n;
        bb = to_f32(Bp[ix]);
        cc = to_f32(Cp[ix]);
      }
      sB[t][n] = bb;
      sC[t][n] = cc;
    }
    __syncthreads();

    for (int t = 0; t < tc; ++t) {
      const float2 dd = sDD[t][j];
      if (kAgg) sdt += (double)dd.x;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < SPL; ++k) {
        const int n = g * SPL + k;
        const float a = decay<kAccurate>(dd.x, Av[k], A2[k]);  // A-bar = exp(dt * A)
        const float bu = kZOH ? zoh_factor<kAccurate>(dd.x, Av[k]) * sU[t][j] : dd.y;
        h[k] = fmaf(a, h[k], bu * sB[t][n]);               // h = A-bar h + (dt u) B
        acc = fmaf(sC[t][n], h[k], acc);                   // C . h (this lane's states)
      }
      sP[t][tid] = acc;
    }
    __syncthreads();

    for (int i = tid; i < TC * DT; i += NT) {
      const int t = i / DT, jj = i % DT;
      const int64_t d = d0 + jj;
      if (!kAgg && t < tc && d < D) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < LPC; ++q) v += sP[t][jj * LPC + q];
        if (p.Dskip) v = fmaf(p.Dskip[d], sU[t][jj], v);
        if (zp) v *= silu_precise(sZ[t][jj]);
        y[(t0 + t) * D + d] = from_f32<TY>(v);
      }
    }
    __syncthreads();
  }

  if (kAgg) {  // end state from zero and decay product exp(A * sum dt) of the segment
    if (vj) {
#pragma unroll
      for (int k = 0; k < SPL; ++k) {
        seg_slot_store(sy, 1, seg, b, dj, g * SPL + k, h[k]);
        seg_slot_store(sy, 2, seg, b, dj, g * SPL + k,
                       kAccurate ? (float)exp((double)Av[k] * sdt) : ex2(A2[k] * (float)sdt));
      }
    }
    return;
  }
  if (vj && p.last_state && seg == (int64_t)gridDim.z - 1) {
#pragma unroll
    for (int k = 0; k < SPL; ++k) p.last_state[(b * D + dj) * N + g * SPL + k] = h[k];
  }
}

// The conv state after a sequence: the three inputs before step L, oldest first, from
// the old state where the sequence is shorter than three. One thread per (b, d); it
// reads before it writes, so the state is updated in place.
template <typename T>
__global__ void __launch_bounds__(256) conv_state_next_kernel(const T* __restrict__ x, T* cs, int64_t batch, int64_t L,
                                                              int64_t D) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= batch * D) return;
  const int64_t b = i / D, d = i % D;
  const T old[3] = {cs[i * 3], cs[i * 3 + 1], cs[i * 3 + 2]};
  T nw[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int64_t s = L - 3 + j;
    nw[j] = s >= 0 ? x[(b * L + s) * D + d] : old[j + L];
  }
#pragma unroll
  for (int j = 0; j < 3; ++j) cs[i * 3 + j] = nw[j];
}

}  // namespace ssm
