// scan_bwd.cuh -- backward pass of the selective scan (Delta * B discretisation), sm_103a.
//
// For the loss sum(dy * y) + sum(dlast * last_state), per channel, in reverse time with
// g = dL/dh_t (starting from dlast):
//   dv = dy silu(z)          dz = dy v silu'(z)          dD += dv u
//   g += dv C_t              dC_t += dv h_t
//   dB_t += g dt u           du = dv D + sum_n g dt B_t
//   d(dt) = sum_n g (B_t u + A a h_{t-1})                 dA += g a h_{t-1} dt
//   ddelta = d(dt) sigmoid(r) with softplus (else d(dt))   dbias += ddelta
//   g *= a                   (after t = 0: dh0 = g)
// The chain rule through the recurrence of "Mamba and State Space Models", "Selective
// scan pseudo-code"; the reverse sweep is the backward of the scan with recomputation
// of the states that "Hardware-Aware Parallel Scan" describes ("8.7 State Space Models
// (Mamba)", section 4.1: the same (a, b) recurrence run backwards).
//
// Layout: two lanes per channel, each holding half of its N states in registers (a warp
// covers 16 channels; one warp per CTA, several CTAs per SM), so that twice as many warps
// hide the latency of the per-step dependency chains. A forward sweep stores the state before every
// chunk of kBwdK steps (checkpoints); the reverse sweep recomputes a chunk's states into
// shared memory, then walks it backwards. Each chunk's inputs are staged into shared
// memory with asynchronous copies (cp.async), double-buffered: the next chunk streams
// in while the current one is computed, and B, C are read as shared-memory broadcasts.
// dB and dC are sums over channels: each warp
// reduces its 16 channels with a transpose-reduce butterfly (shuffles) and writes one
// partial per (b, t, warp, n); scan_bwd_reduce then sums the partials over warps, and
// dA, dD, dbias over batch rows, in a fixed order (deterministic, no atomics).
#pragma once

#include "common.cuh"

namespace ssm {

struct BwdParams {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* Dskip;       // nullable
  const void* z;            // nullable
  const float* delta_bias;  // nullable
  int delta_softplus;
  const float* h0;          // nullable
  const void* dy;           // gradient type TG
  const float* dlast;       // nullable
  void* du;                 // TG
  void* ddelta;             // TG
  void* dz;                 // TG, nullable (iff z)
  float* dh0;               // nullable
  // workspace
  float* ck;          // [b][nc][D][N]: state before each chunk
  float* part;        // [b][L][W][2][N]: per-warp partials of dB (0) and dC (1)
  float* dA_part;     // [b][D][N]
  float* dD_part;     // [b][D]
  float* dbias_part;  // [b][D]
  int64_t batch, L, D;
  int nc, W;          // chunks of kBwdK steps; warps along D
  bool async_ok;      // every staged row starts 16-byte aligned: stage with cp.async
};

constexpr int kBwdK = 16;
constexpr int kBwdCh = 16;  // channels per warp (two lanes per channel)

// Sum over the warp's 16 channels (lanes of equal parity: lane = 2 * channel + half) of
// each of v[0..NH-1]; lane l ends with the sum of v[(l >> (5 - log2 NH)) & (NH - 1)] of
// its half. Each round halves the values a lane holds: the lanes with the round's bit set
// keep the upper half and send the lower, the others the reverse; bit 0 (the half) is
// never summed.
template <int NH>
__device__ __forceinline__ float pair_transpose_reduce(float (&v)[NH], int lane) {
  constexpr int kLog = NH == 8 ? 3 : NH == 4 ? 2 : 1;
  int m = NH;
#pragma unroll
  for (int r = 0; r < kLog; ++r) {
    const int o = 16 >> r;
    const bool upper = (lane & o) != 0;
    const int half = m / 2;
#pragma unroll
    for (int i = 0; i < NH / 2; ++i) {
      if (i < half) {
        const float send = upper ? v[i] : v[i + half];
        const float keep = upper ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    m = half;
  }
  float s = v[0];
#pragma unroll
  for (int o = 16 >> kLog; o >= 2; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// ---- chunk staging: global -> shared memory, asynchronous (cp.async) ----
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Raw inputs of one chunk of kBwdK steps for the 32 channels of this warp.
template <typename T, typename TG, int N>
struct BwdStage {
  T u[kBwdK][kBwdCh];
  T dl[kBwdK][kBwdCh];
  T z[kBwdK][kBwdCh];
  TG dy[kBwdK][kBwdCh];
  T B[kBwdK * N];
  T C[kBwdK * N];
};

// One (kBwdK x kBwdCh) tile of a (batch, L, D) tensor into smem. Asynchronous 16-byte copies
// when every row start is 16-byte aligned (zero-filled past L and D), else plain loads.
template <typename E>
__device__ __forceinline__ void stage_rows(E (*dst)[kBwdCh], const E* src, int64_t b, int64_t t0, int64_t L,
                                           int64_t D, int64_t d0, bool async_ok, int lane) {
  if (async_ok) {
    constexpr int kPieces = kBwdCh * (int)sizeof(E) / 16;  // 16-byte pieces per row
    const int64_t valid_row = (D - d0) * (int64_t)sizeof(E);
    for (int q = lane; q < kBwdK * kPieces; q += 32) {
      const int k = q / kPieces, j = q % kPieces;
      const int64_t t = t0 + k;
      int64_t nb = t < L ? valid_row - j * 16 : 0;
      nb = nb < 0 ? 0 : (nb > 16 ? 16 : nb);
      const E* g = nb > 0 ? src + ((b * L + t) * D + d0) + j * (16 / (int)sizeof(E)) : src;
      cp_async16(reinterpret_cast<unsigned char*>(&dst[k][0]) + j * 16, g, (int)nb);
    }
  } else {
    for (int i = lane; i < kBwdK * kBwdCh; i += 32) {
      const int k = i / kBwdCh, cc = i % kBwdCh;
      const int64_t t = t0 + k, d = d0 + cc;
      dst[k][cc] = (t < L && d < D) ? src[(b * L + t) * D + d] : E(0.f);
    }
  }
}

// The chunk's (kBwdK x N) block of a (batch, L, N) tensor.
template <typename E, int N>
__device__ __forceinline__ void stage_bc(E* dst, const E* src, int64_t b, int64_t t0, int64_t L, bool async_ok,
                                         int lane) {
  constexpr int kBytes = kBwdK * N * (int)sizeof(E);
  if (async_ok) {
    const int64_t valid = (L - t0) * N * (int64_t)sizeof(E);
    for (int j = lane; j < kBytes / 16; j += 32) {
      int64_t nb = valid - j * 16;
      nb = nb < 0 ? 0 : (nb > 16 ? 16 : nb);
      const E* g = nb > 0 ? src + (b * L + t0) * N + j * (16 / (int)sizeof(E)) : src;
      cp_async16(reinterpret_cast<unsigned char*>(dst) + j * 16, g, (int)nb);
    }
  } else {
    for (int i = lane; i < kBwdK * N; i += 32) {
      const int64_t t = t0 + i / N;
      dst[i] = t < L ? src[(b * L + t0) * N + i] : E(0.f);
    }
  }
}

template <typename T, typename TG, int N>
__device__ __forceinline__ void stage_chunk(BwdStage<T, TG, N>& sg, const BwdParams& p, int64_t b, int c, int64_t d0,
                                            bool reverse, int lane) {
  const int64_t t0 = (int64_t)c * kBwdK;
  stage_rows<T>(sg.u, static_cast<const T*>(p.u), b, t0, p.L, p.D, d0, p.async_ok, lane);
  stage_rows<T>(sg.dl, static_cast<const T*>(p.delta), b, t0, p.L, p.D, d0, p.async_ok, lane);
  stage_bc<T, N>(sg.B, static_cast<const T*>(p.B), b, t0, p.L, p.async_ok, lane);
  if (reverse) {
    stage_rows<TG>(sg.dy, static_cast<const TG*>(p.dy), b, t0, p.L, p.D, d0, p.async_ok, lane);
    if (p.z) stage_rows<T>(sg.z, static_cast<const T*>(p.z), b, t0, p.L, p.D, d0, p.async_ok, lane);
    stage_bc<T, N>(sg.C, static_cast<const T*>(p.C), b, t0, p.L, p.async_ok, lane);
  }
  cp_async_commit();
}

// The P2 state pairs of this lane's half of a B or C row; 16-byte loads when P2 is even
// (the row and the half then start 16-byte aligned).
template <int P2>
__device__ __forceinline__ void load_pairs(const float* row, float2 (&v)[P2]) {
  if constexpr (P2 % 2 == 0) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll
    for (int i = 0; i < P2 / 2; ++i) {
      const float4 t = r4[i];
      v[2 * i] = make_float2(t.x, t.y);
      v[2 * i + 1] = make_float2(t.z, t.w);
    }
  } else {
    const float2* r2 = reinterpret_cast<const float2*>(row);
#pragma unroll
    for (int i = 0; i < P2; ++i) v[i] = r2[i];
  }
}

// Decay factors of two states: 2^(dt A log2 e) on the SFU, or exp in double on the
// fp32 I/O path (as the forward kernels).
template <bool kAccurate>
__device__ __forceinline__ float2 decay2(float2 dt2, float2 A, float2 A2) {
  if (kAccurate) return make_float2(decay<true>(dt2.x, A.x, A2.x), decay<true>(dt2.y, A.y, A2.y));
  const float2 x = __fmul2_rn(dt2, A2);
  return make_float2(ex2(x.x), ex2(x.y));
}

// grid (W = ceil(D / 16), batch), block 32 (one warp: 16 channels x two halves of the
// states); dynamic shared memory:
//   hs  [kBwdK + 1][N/4][32] f32x2 each lane's state pairs h_{t0-1} .. h_{t0+K-1} of the chunk
//   bc  [kBwdK][2N]          f32  the chunk's B | C rows
//   dts [kBwdK][32]          f32  step sizes (both lanes of a channel hold the same)
//   vs  [kBwdK][32]          f32  read-outs C.h + D u (before the gate)
//   stage[2]                      raw inputs of the current and the next chunk
template <typename T, typename TG, int N>
constexpr int bwd_smem_bytes() {
  return ((kBwdK + 1) * (N / 2) * 32 + kBwdK * 2 * N + 2 * kBwdK * 32) * 4 + 2 * (int)sizeof(BwdStage<T, TG, N>);
}

template <typename T, typename TG, int N>
__global__ void __launch_bounds__(32) scan_bwd_kernel(const BwdParams p) {
  constexpr int NH = N / 2;   // states per lane
  constexpr int P2 = NH / 2;  // packed pairs per lane
  extern __shared__ __align__(16) float sm[];
  float* hs = sm;  // [kBwdK + 1][P2][32] float2: state pairs of each lane
  float2* hs2 = reinterpret_cast<float2*>(hs);
  float* bc = hs + (kBwdK + 1) * NH * 32;
  float* dts = bc + kBwdK * 2 * N;
  float* vs = dts + kBwdK * 32;
  BwdStage<T, TG, N>* stg = reinterpret_cast<BwdStage<T, TG, N>*>(vs + kBwdK * 32);
  const int lane = threadIdx.x, ch = lane >> 1, half = lane & 1, nb = half * NH;
  const int w = blockIdx.x;
  const int64_t b = blockIdx.y;
  const int64_t L = p.L, D = p.D;
  const int64_t d0 = (int64_t)w * kBwdCh, d = d0 + ch;
  const bool vd = d < D;
  constexpr bool kAccurate = sizeof(T) == 4;
  const float bias = (vd && p.delta_bias) ? p.delta_bias[d] : 0.f;

  float2 Av[P2], A2[P2], h[P2];
#pragma unroll
  for (int q = 0; q < P2; ++q) {
    Av[q] = vd ? make_float2(p.A[d * N + nb + 2 * q], p.A[d * N + nb + 2 * q + 1]) : make_float2(0.f, 0.f);
    A2[q] = __fmul2_rn(Av[q], make_float2(kLog2e, kLog2e));
    h[q] = (vd && p.h0) ? make_float2(p.h0[(b * D + d) * N + nb + 2 * q], p.h0[(b * D + d) * N + nb + 2 * q + 1])
                        : make_float2(0.f, 0.f);
  }
  auto convert_bc = [&](const BwdStage<T, TG, N>& sg, bool with_c) {
    for (int i = lane; i < kBwdK * N; i += 32) {
      const int k = i / N, n = i % N;
      bc[k * 2 * N + n] = to_f32(sg.B[i]);
      if (with_c) bc[k * 2 * N + N + n] = to_f32(sg.C[i]);
    }
    __syncwarp();
  };
  auto step_dt = [&](const BwdStage<T, TG, N>& sg, int k, float* r_out) {
    const float r = to_f32(sg.dl[k][ch]) + bias;
    if (r_out) *r_out = r;
    if (!p.delta_softplus) return r;
    if (kAccurate) return softplus_precise(r);
    return fmaxf(r, 0.f) + kLn2 * lg2(1.f + ex2(fabsf(r) * -kLog2e));  // SFU form, as the forward
  };
  // the bf16 path divides with the fast approximate reciprocal (~2 ulp), well inside its
  // tolerance; the fp32 path keeps the correctly rounded one
  auto sigmoid = [&](float x) {
    return kAccurate ? __frcp_rn(1.f + __expf(-x)) : __fdividef(1.f, 1.f + __expf(-x));
  };

  // ---- forward sweep: the state before every chunk ----
  if (p.nc > 1) stage_chunk<T, TG, N>(stg[0], p, b, 0, d0, false, lane);
  for (int c = 0; c < p.nc; ++c) {
    if (vd) {
      float2* ckp = reinterpret_cast<float2*>(p.ck + (((int64_t)b * p.nc + c) * D + d) * N + nb);
#pragma unroll
      for (int q = 0; q < P2; ++q) ckp[q] = h[q];
    }
    if (c == p.nc - 1) break;  // the state after the last chunk is not needed
    cp_async_wait_all();
    __syncwarp();
    const BwdStage<T, TG, N>& sg = stg[c & 1];
    convert_bc(sg, false);
    if (c + 1 < p.nc - 1) stage_chunk<T, TG, N>(stg[(c + 1) & 1], p, b, c + 1, d0, false, lane);
    for (int k = 0; k < kBwdK; ++k) {  // chunks before the last are full
      const float dt = vd ? step_dt(sg, k, nullptr) : 0.f;
      const float dx = dt * to_f32(sg.u[k][ch]);
      const float2 dt2 = make_float2(dt, dt), dx2 = make_float2(dx, dx);
      float2 b2[P2];
      load_pairs<P2>(bc + k * 2 * N + nb, b2);
#pragma unroll
      for (int q = 0; q < P2; ++q)
        h[q] = __ffma2_rn(decay2<kAccurate>(dt2, Av[q], A2[q]), h[q], __fmul2_rn(dx2, b2[q]));
    }
    __syncwarp();
  }

  // ---- reverse sweep ----
  float2 g[P2], dA_acc[P2];
#pragma unroll
  for (int q = 0; q < P2; ++q) {
    g[q] = (vd && p.dlast) ? make_float2(p.dlast[(b * D + d) * N + nb + 2 * q], p.dlast[(b * D + d) * N + nb + 2 * q + 1])
                           : make_float2(0.f, 0.f);
    dA_acc[q] = make_float2(0.f, 0.f);
  }
  float dD_acc = 0.f, dbias_acc = 0.f;
  const float Dk = (vd && p.Dskip) ? p.Dskip[d] : 0.f;
  constexpr int kLog = NH == 8 ? 3 : NH == 4 ? 2 : 1;
  const int n_red = nb + ((lane >> (5 - kLog)) & (NH - 1));
  const bool writer = (lane & (((1 << (5 - kLog)) - 1) & ~1)) == 0;
  const bool lead = half == 0 && vd;  // writes the channel's per-step outputs
  TG* du = static_cast<TG*>(p.du) + b * L * D + d;
  TG* ddl = static_cast<TG*>(p.ddelta) + b * L * D + d;
  TG* dzp = p.dz ? static_cast<TG*>(p.dz) + b * L * D + d : nullptr;
  float* part = p.part + ((b * L) * p.W + w) * 2 * N;  // + t * W * 2N

  stage_chunk<T, TG, N>(stg[(p.nc - 1) & 1], p, b, p.nc - 1, d0, true, lane);
  for (int c = p.nc - 1; c >= 0; --c) {
    const int64_t t0 = (int64_t)c * kBwdK;
    const int kc = (int)((L - t0) < kBwdK ? (L - t0) : kBwdK);
    cp_async_wait_all();
    __syncwarp();
    const BwdStage<T, TG, N>& sg = stg[c & 1];
    convert_bc(sg, true);
    if (c > 0) stage_chunk<T, TG, N>(stg[(c - 1) & 1], p, b, c - 1, d0, true, lane);
    // recompute the chunk's states and read-outs
    {
      const float2* ckp = reinterpret_cast<const float2*>(p.ck + (((int64_t)b * p.nc + c) * D + d) * N + nb);
#pragma unroll
      for (int q = 0; q < P2; ++q) {
        h[q] = vd ? ckp[q] : make_float2(0.f, 0.f);
        hs2[q * 32 + lane] = h[q];
      }
      for (int k = 0; k < kc; ++k) {
        const float dt = vd ? step_dt(sg, k, nullptr) : 0.f;
        const float x = to_f32(sg.u[k][ch]);
        const float dx = dt * x;
        dts[k * 32 + lane] = dt;
        const float2 dt2 = make_float2(dt, dt), dx2 = make_float2(dx, dx);
        float2 b2[P2], c2[P2];
        load_pairs<P2>(bc + k * 2 * N + nb, b2);
        load_pairs<P2>(bc + k * 2 * N + N + nb, c2);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < P2; ++q) {
          h[q] = __ffma2_rn(decay2<kAccurate>(dt2, Av[q], A2[q]), h[q], __fmul2_rn(dx2, b2[q]));
          acc = __ffma2_rn(c2[q], h[q], acc);
          hs2[((k + 1) * P2 + q) * 32 + lane] = h[q];
        }
        const float vp = acc.x + acc.y;
        vs[k * 32 + lane] = fmaf(Dk, x, vp + __shfl_xor_sync(0xffffffffu, vp, 1));
      }
    }
    // walk it backwards; h[] holds h_t of the current step (the chunk's last state first)
    for (int k = kc - 1; k >= 0; --k) {
      const int64_t t = t0 + k;
      const float dt = dts[k * 32 + lane];
      float r = 0.f;
      if (vd) step_dt(sg, k, &r);
      const float x = to_f32(sg.u[k][ch]), dyv = to_f32(sg.dy[k][ch]);
      const float v = vs[k * 32 + lane];
      float dv = dyv;
      if (dzp) {
        const float zz = to_f32(sg.z[k][ch]);
        const float sgm = sigmoid(zz);
        if (lead) dzp[t * D] = from_f32<TG>(dyv * v * (sgm * (1.f + zz * (1.f - sgm))));
        dv = dyv * zz * sgm;
      }
      dD_acc = fmaf(dv, x, dD_acc);
      const float2 dv2 = make_float2(dv, dv), dt2 = make_float2(dt, dt), x2 = make_float2(x, x);
      float2 b2[P2], c2[P2];
      load_pairs<P2>(bc + k * 2 * N + nb, b2);
      load_pairs<P2>(bc + k * 2 * N + N + nb, c2);
      float2 dux2 = make_float2(0.f, 0.f), ddt2 = make_float2(0.f, 0.f);
      float vb[NH], vc[NH];
#pragma unroll
      for (int q = 0; q < P2; ++q) {
        const float2 hp = hs2[(k * P2 + q) * 32 + lane];
        const float2 a = decay2<kAccurate>(dt2, Av[q], A2[q]);
        const float2 B2 = b2[q];
        g[q] = __ffma2_rn(dv2, c2[q], g[q]);                 // g = dL/dh_t
        const float2 cv = __fmul2_rn(dv2, h[q]);             // dC_t contribution: dv h_t
        const float2 gdt = __fmul2_rn(g[q], dt2);
        const float2 bv = __fmul2_rn(gdt, x2);               // dB_t contribution: g dt u
        dux2 = __ffma2_rn(gdt, B2, dux2);
        const float2 ah = __fmul2_rn(a, hp);
        ddt2 = __ffma2_rn(g[q], __ffma2_rn(B2, x2, __fmul2_rn(Av[q], ah)), ddt2);
        dA_acc[q] = __ffma2_rn(__fmul2_rn(g[q], ah), dt2, dA_acc[q]);
        g[q] = __fmul2_rn(g[q], a);                          // dL/dh_{t-1} (through the recurrence)
        h[q] = hp;                                           // h_t of step t-1
        vb[2 * q] = bv.x;
        vb[2 * q + 1] = bv.y;
        vc[2 * q] = cv.x;
        vc[2 * q + 1] = cv.y;
      }
      float dux = dux2.x + dux2.y, ddt = ddt2.x + ddt2.y;
      dux += __shfl_xor_sync(0xffffffffu, dux, 1);          // the channel's other half
      ddt += __shfl_xor_sync(0xffffffffu, ddt, 1);
      dux = fmaf(dv, Dk, dux);
      const float dr = p.delta_softplus ? ddt * sigmoid(r) : ddt;
      dbias_acc += dr;
      if (lead) {
        du[t * D] = from_f32<TG>(dux);
        ddl[t * D] = from_f32<TG>(dr);
      }
      const float sb = pair_transpose_reduce<NH>(vb, lane);
      const float sc = pair_transpose_reduce<NH>(vc, lane);
      if (writer) {
        float* pp = part + t * p.W * 2 * N;
        pp[n_red] = sb;
        pp[N + n_red] = sc;
      }
    }
    __syncwarp();
  }

  if (vd) {
#pragma unroll
    for (int q = 0; q < P2; ++q) {
      p.dA_part[(b * D + d) * N + nb + 2 * q] = dA_acc[q].x;
      p.dA_part[(b * D + d) * N + nb + 2 * q + 1] = dA_acc[q].y;
    }
    if (half == 0) {
      p.dD_part[b * D + d] = dD_acc;
      p.dbias_part[b * D + d] = dbias_acc;
    }
    if (p.dh0) {
#pragma unroll
      for (int q = 0; q < P2; ++q) {
        p.dh0[(b * D + d) * N + nb + 2 * q] = g[q].x;
        p.dh0[(b * D + d) * N + nb + 2 * q + 1] = g[q].y;
      }
    }
  }
}

// Fixed-order sums of the partials: dB, dC (batch, L, N) over the W warps along D;
// dA (D, N), dD (D), dbias (D) over the batch rows. One thread per output element.
template <typename TG>
__global__ void __launch_bounds__(256) scan_bwd_reduce(const float* __restrict__ part, const float* __restrict__ dA_part,
                                                       const float* __restrict__ dD_part,
                                                       const float* __restrict__ dbias_part, TG* dB, TG* dC, float* dA,
                                                       float* dD, float* dbias, int64_t batch, int64_t L, int64_t D,
                                                       int N, int W) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nbc = batch * L * N, na = D * N;
  if (i < nbc) {
    const int64_t n = i % N, bt = i / N;
    float sb = 0.f, sc = 0.f;
    for (int w = 0; w < W; ++w) {
      const float* pp = part + ((bt * W + w) * 2) * N;
      sb += pp[n];
      sc += pp[N + n];
    }
    dB[i] = from_f32<TG>(sb);
    dC[i] = from_f32<TG>(sc);
  } else if (i < nbc + na) {
    const int64_t j = i - nbc;
    float s = 0.f;
    for (int64_t b = 0; b < batch; ++b) s += dA_part[b * na + j];
    dA[j] = s;
  } else if (i < nbc + na + D) {
    const int64_t j = i - nbc - na;
    float s = 0.f, sb = 0.f;
    for (int64_t b = 0; b < batch; ++b) {
      s += dD_part[b * D + j];
      sb += dbias_part[b * D + j];
    }
    if (dD) dD[j] = s;
    if (dbias) dbias[j] = sb;
  }
}

}  // namespace ssm
