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
// hide the latency of the per-step dependency chains. The state before every chunk of
// kBwdK steps (a checkpoint) comes from the channel kernel's forward sweep (ck_ready), or
// from a forward sweep here when that kernel does not apply. Per chunk, in reverse order:
// the raw inputs, staged into shared memory by asynchronous copies (cp.async), become
// per-(step, channel) scalars in a prologue (each computed once), the buffer is refilled
// with the previous chunk at once, the chunk's states are recomputed into shared memory
// from its checkpoint, and the chunk is walked backwards; the read-out C.h + D u that the
// gate's gradient needs is recomputed in that walk. dB and dC are sums over channels:
// each warp sums its 16 channels once per step (column sums in shared memory for N = 16,
// a shuffle transpose-reduce below) and writes one partial per (b, t, warp, n); scan_bwd_reduce then sums the partials over
// warps, and dA, dD, dbias over batch rows, in a fixed order (deterministic, no atomics).
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
  int ck_ready;       // 1: ck already holds the checkpoints (no forward sweep here)
};

constexpr int kBwdK = kCkSteps;
constexpr int kBwdCh = 16;  // channels per warp (two lanes per channel)

// Sums over the warp's 16 channels (lane = 2 * channel + half) of the 2 NH values v[]
// of every lane (its half's dB contributions, then its dC contributions): a transpose-
// reduce. Each round halves what a lane holds: the lanes with the round's bit set keep
// the upper half and send the lower, the others the reverse. After the rounds over lane
// bits 4..1 (2 NH = 16) lane l holds the sum for value index (l >> 1) & 15 of its half,
// i.e. kind (l >> 4) & 1 (0 = dB, 1 = dC) and state half * NH + ((l >> 1) & 7).
// N = 8 / 4 (2 NH = 8 / 4 values) stop after 3 / 2 rounds; lane bits 2 / 3..1 left over
// still separate channels, so those lanes finish with plain xor-shuffle sums.
template <int NV>
__device__ __forceinline__ float bwd_transpose_reduce(float (&v)[NV], int lane) {
  constexpr int kLog = NV == 16 ? 4 : NV == 8 ? 3 : 2;
  int m = NV;
#pragma unroll
  for (int r = 0; r < kLog; ++r) {
    const int o = 16 >> r;
    const bool upper = (lane & o) != 0;
    const int half = m / 2;
#pragma unroll
    for (int i = 0; i < NV / 2; ++i) {
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
  if constexpr (sizeof(T) == 2 && sizeof(TG) == 2 && N == 16) {
    // a whole chunk of a whole channel block: no clamping; lane l copies the 16 bytes at row
    // l / 2, half l % 2 of each (step x channel) tile, and piece l of the B and C blocks
    if (p.async_ok && t0 + kBwdK <= p.L && d0 + kBwdCh <= p.D) {
      const int64_t off = (b * p.L + t0 + (lane >> 1)) * p.D + d0 + (lane & 1) * 8;
      const int64_t offbc = (b * p.L + t0) * N + lane * 8;
      cp_async16(&sg.u[0][0] + lane * 8, static_cast<const T*>(p.u) + off, 16);
      cp_async16(&sg.dl[0][0] + lane * 8, static_cast<const T*>(p.delta) + off, 16);
      cp_async16(&sg.B[0] + lane * 8, static_cast<const T*>(p.B) + offbc, 16);
      if (reverse) {
        cp_async16(&sg.dy[0][0] + lane * 8, static_cast<const TG*>(p.dy) + off, 16);
        if (p.z) cp_async16(&sg.z[0][0] + lane * 8, static_cast<const T*>(p.z) + off, 16);
        cp_async16(&sg.C[0] + lane * 8, static_cast<const T*>(p.C) + offbc, 16);
      }
      cp_async_commit();
      return;
    }
  }
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

// 16 bytes of T (8 bf16 or 4 fp32) from shared memory to fp32 in shared memory.
template <typename T>
__device__ __forceinline__ void vec_to_f32(float* dst, const T* src) {
  const uint4 v = *reinterpret_cast<const uint4*>(src);
  float4* d4 = reinterpret_cast<float4*>(dst);
  if constexpr (sizeof(T) == 4) {
    d4[0] = make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
  } else {
    // bf16 -> fp32 is the 16 bits moved to the top half
    d4[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u), __uint_as_float(v.y << 16),
                        __uint_as_float(v.y & 0xffff0000u));
    d4[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u), __uint_as_float(v.w << 16),
                        __uint_as_float(v.w & 0xffff0000u));
  }
}

// Two adjacent elements of T (bf16 or fp32) from shared memory as floats.
template <typename T>
__device__ __forceinline__ float2 ld_pair(const T* src) {
  if constexpr (sizeof(T) == 4) {
    return *reinterpret_cast<const float2*>(src);
  } else {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(src);
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
  }
}
// Softplus and sigmoid of two values on the bf16 path (2^x, log2 and the reciprocal on the
// SFU, the rest as packed f32x2 ops): max(r, 0) + ln2 log2(1 + 2^(-|r| log2 e)), and
// 1 / (1 + 2^(-x log2 e)) (the denominator is at least 1, so the SFU's reciprocal is used
// as it stands).
__device__ __forceinline__ float2 softplus2_bwd(float2 r) {
  const float2 a = __fmul2_rn(make_float2(fabsf(r.x), fabsf(r.y)), make_float2(-kLog2e, -kLog2e));
  const float2 op = __fadd2_rn(make_float2(ex2(a.x), ex2(a.y)), make_float2(1.f, 1.f));
  return __ffma2_rn(make_float2(lg2(op.x), lg2(op.y)), make_float2(kLn2, kLn2),
                    make_float2(fmaxf(r.x, 0.f), fmaxf(r.y, 0.f)));
}
__device__ __forceinline__ float2 sigmoid2_bwd(float2 x) {
  const float2 a = __fmul2_rn(x, make_float2(-kLog2e, -kLog2e));
  const float2 den = __fadd2_rn(make_float2(ex2(a.x), ex2(a.y)), make_float2(1.f, 1.f));
  float rx, ry;  // den >= 1: the approximate reciprocal needs no range handling
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rx) : "f"(den.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(ry) : "f"(den.y));
  return make_float2(rx, ry);
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
//   hs  [kBwdK][N/4][32]     f32x2 each lane's state pairs h_{t0-1} .. h_{t0+K-2} of the chunk
//   bc  [kBwdK][2N]          f32  the chunk's B | C rows
//   sc  [kBwdK][16]          f32x4 per (step, channel): dt, dt u, dv, u
//   sx  [kBwdK][16]          f32x2 per (step, channel): d(dt)/d(delta), dy silu'(z)
//   red [2][16][32]          f32  (N = 16) a step's dB | dC values per channel, for the channel
//                                 sums; two tiles, used by alternate steps
// (N = 16, bf16: 31 KB, so that seven CTAs fit in an SM's 228 KB with their 1 KB reserve)
//   stage                         raw inputs of one chunk (refilled as soon as they are read)
template <typename T, typename TG, int N>
constexpr int bwd_smem_bytes() {
  return (kBwdK * (N / 2) * 32 + kBwdK * 2 * N + kBwdK * kBwdCh * 6 + (N == 16 ? 2 * kBwdCh * 32 : 0)) * 4 +
         (int)sizeof(BwdStage<T, TG, N>);
}

template <typename T, typename TG, int N>
__global__ void __launch_bounds__(32) scan_bwd_kernel(const BwdParams p) {
  constexpr int NH = N / 2;   // states per lane
  constexpr int P2 = NH / 2;  // packed pairs per lane
  constexpr int kItems = kBwdK * kBwdCh / 32;  // (step, channel) items per lane in a chunk
  extern __shared__ __align__(16) float sm[];
  float2* hs2 = reinterpret_cast<float2*>(sm);  // [kBwdK][P2][32]
  float* bc = sm + kBwdK * NH * 32;
  float4* sc = reinterpret_cast<float4*>(bc + kBwdK * 2 * N);  // [kBwdK][16]
  float2* sx = reinterpret_cast<float2*>(sc + kBwdK * kBwdCh);  // [kBwdK][16]
  float* red = reinterpret_cast<float*>(sx + kBwdK * kBwdCh);  // [16][32] when N = 16
  BwdStage<T, TG, N>& sg = *reinterpret_cast<BwdStage<T, TG, N>*>(red + (N == 16 ? 2 * kBwdCh * 32 : 0));
  const int lane = threadIdx.x, ch = lane >> 1, half = lane & 1, nb = half * NH;
  const int w = blockIdx.x;
  const int64_t b = blockIdx.y;
  const int64_t L = p.L, D = p.D;
  const int64_t d0 = (int64_t)w * kBwdCh, d = d0 + ch;
  const bool vd = d < D;
  constexpr bool kAccurate = sizeof(T) == 4;
  // the prologue's items all belong to channel lane & 15
  const int pch = lane & 15;
  const float pbias = (d0 + pch < D && p.delta_bias) ? p.delta_bias[d0 + pch] : 0.f;
  const int pc0 = 2 * (lane & 7);  // the bf16 prologue's channel pair
  const float2 pbias2 = p.delta_bias ? make_float2(d0 + pc0 < D ? p.delta_bias[d0 + pc0] : 0.f,
                                                   d0 + pc0 + 1 < D ? p.delta_bias[d0 + pc0 + 1] : 0.f)
                                     : make_float2(0.f, 0.f);

  float2 Av[P2], A2[P2], h[P2];  // A, A log2(e) (Av: the fp32 path's exact decay and sums)
#pragma unroll
  for (int q = 0; q < P2; ++q) {
    Av[q] = vd ? make_float2(p.A[d * N + nb + 2 * q], p.A[d * N + nb + 2 * q + 1]) : make_float2(0.f, 0.f);
    A2[q] = __fmul2_rn(Av[q], make_float2(kLog2e, kLog2e));
    h[q] = (vd && p.h0) ? make_float2(p.h0[(b * D + d) * N + nb + 2 * q], p.h0[(b * D + d) * N + nb + 2 * q + 1])
                        : make_float2(0.f, 0.f);
  }
  // the bf16 path divides with the fast approximate reciprocal (~2 ulp), well inside its
  // tolerance; the fp32 path keeps the correctly rounded one
  auto sigmoid = [&](float x) {
    return kAccurate ? __frcp_rn(1.f + __expf(-x)) : __fdividef(1.f, 1.f + __expf(-x));
  };
  // Chunk prologue: B | C rows to f32, and the per-(step, channel) scalars computed once
  // (not once per lane of the channel and per sweep). full = false: the forward sweep's
  // dt and dt u only (dy and z are not staged there).
  auto prologue = [&](bool full) {
    constexpr int kV = 16 / (int)sizeof(T);  // elements per 16-byte piece
    if constexpr (N % kV == 0) {
      for (int pc = lane; pc < kBwdK * N / kV; pc += 32) {
        const int e0 = pc * kV, k = e0 / N, n0 = e0 % N;
        vec_to_f32<T>(bc + k * 2 * N + n0, &sg.B[e0]);
        if (full) vec_to_f32<T>(bc + k * 2 * N + N + n0, &sg.C[e0]);
      }
    } else {
      for (int i = lane; i < kBwdK * N; i += 32) {
        const int k = i / N, n = i % N;
        bc[k * 2 * N + n] = to_f32(sg.B[i]);
        if (full) bc[k * 2 * N + N + n] = to_f32(sg.C[i]);
      }
    }
    if constexpr (!kAccurate) {
      // bf16 path: two adjacent channels per lane (c0, c0 + 1; the same for every j),
      // steps 4 j + lane / 8, with packed ops
      const int c0 = 2 * (lane & 7);
#pragma unroll
      for (int j = 0; j < kItems / 2; ++j) {
        const int k = 4 * j + (lane >> 3);
        const float2 r = __fadd2_rn(ld_pair(&sg.dl[k][c0]), pbias2);
        float2 dt = r, sr = make_float2(1.f, 1.f);
        if (p.delta_softplus) {
          dt = softplus2_bwd(r);
          if (full) sr = sigmoid2_bwd(r);
        }
        const float2 x = ld_pair(&sg.u[k][c0]);
        float2 dv = make_float2(0.f, 0.f), dyz = make_float2(0.f, 0.f);
        if (full) {
          const float2 dyv = ld_pair(&sg.dy[k][c0]);
          dv = dyv;
          if (p.z) {
            const float2 zz = ld_pair(&sg.z[k][c0]);
            const float2 sz = sigmoid2_bwd(zz);
            dv = __fmul2_rn(__fmul2_rn(dyv, zz), sz);  // dy silu(z)
            const float2 oms = __fadd2_rn(make_float2(1.f, 1.f), make_float2(-sz.x, -sz.y));
            dyz = __fmul2_rn(dyv, __fmul2_rn(sz, __ffma2_rn(zz, oms, make_float2(1.f, 1.f))));  // dy silu'(z)
          }
        }
        const float2 dtx = __fmul2_rn(dt, x);
        sc[k * kBwdCh + c0] = make_float4(dt.x, dtx.x, dv.x, x.x);
        sc[k * kBwdCh + c0 + 1] = make_float4(dt.y, dtx.y, dv.y, x.y);
        *reinterpret_cast<float4*>(&sx[k * kBwdCh + c0]) = make_float4(sr.x, dyz.x, sr.y, dyz.y);
      }
      __syncwarp();
      return;
    }
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
      const int k = 2 * j + (lane >> 4);
      const float r = to_f32(sg.dl[k][pch]) + pbias;
      float dt = r, sr = 1.f;
      if (p.delta_softplus) {
        dt = kAccurate ? softplus_precise(r) : fmaxf(r, 0.f) + kLn2 * lg2(1.f + ex2(fabsf(r) * -kLog2e));
        if (full) sr = sigmoid(r);
      }
      const float x = to_f32(sg.u[k][pch]);
      float dv = 0.f, dyz = 0.f;
      if (full) {
        const float dyv = to_f32(sg.dy[k][pch]);
        dv = dyv;
        if (p.z) {
          const float zz = to_f32(sg.z[k][pch]);
          const float s = sigmoid(zz);
          dv = dyv * zz * s;                          // dy silu(z)
          dyz = dyv * (s * (1.f + zz * (1.f - s)));   // dy silu'(z)
        }
      }
      sc[k * kBwdCh + pch] = make_float4(dt, dt * x, dv, x);
      sx[k * kBwdCh + pch] = make_float2(sr, dyz);
    }
    __syncwarp();
  };
  // One step of the recurrence for this lane's pairs from the scalars of step k.
  auto fwd_step = [&](int k) {
    const float4 s = sc[k * kBwdCh + ch];
    const float2 dt2 = make_float2(s.x, s.x), du2 = make_float2(s.y, s.y);
    float2 b2[P2];
    load_pairs<P2>(bc + k * 2 * N + nb, b2);
#pragma unroll
    for (int q = 0; q < P2; ++q) h[q] = __ffma2_rn(decay2<kAccurate>(dt2, Av[q], A2[q]), h[q], __fmul2_rn(du2, b2[q]));
  };

  // ---- forward sweep, only when the checkpoints were not supplied ----
  if (!p.ck_ready) {
    if (p.nc > 1) {
      stage_chunk<T, TG, N>(sg, p, b, 0, d0, false, lane);
    }
    for (int c = 0; c < p.nc; ++c) {
      if (vd) {
        float2* ckp = reinterpret_cast<float2*>(p.ck + (((int64_t)b * p.nc + c) * D + d) * N + nb);
#pragma unroll
        for (int q = 0; q < P2; ++q) ckp[q] = h[q];
      }
      if (c == p.nc - 1) break;  // the state after the last chunk is not needed
      cp_async_wait_all();
      __syncwarp();
      prologue(false);
      if (c + 1 < p.nc - 1) stage_chunk<T, TG, N>(sg, p, b, c + 1, d0, false, lane);
      for (int k = 0; k < kBwdK; ++k) fwd_step(k);  // chunks before the last are full
      __syncwarp();
    }
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
  constexpr int NV = 2 * NH;
  constexpr int kLog = NV == 16 ? 4 : NV == 8 ? 3 : 2;
  const int vidx = (lane >> (5 - kLog)) & (NV - 1);
  // kind * N + state of the channel sum this lane ends with (the shared-memory sums of
  // N = 16 leave sum j in lane j)
  const int n_red = N == 16 ? lane : (vidx / NH) * N + nb + (vidx % NH);
  const bool writer = (lane & ((1 << (5 - kLog)) - 2)) == 0;
  TG* du = static_cast<TG*>(p.du) + b * L * D + d;
  TG* ddl = static_cast<TG*>(p.ddelta) + b * L * D + d;
  TG* dzp = p.dz ? static_cast<TG*>(p.dz) + b * L * D + d : nullptr;
  const int64_t pstride = (int64_t)p.W * 2 * N;
  float* part = p.part + ((b * L) * p.W + w) * 2 * N + n_red;  // + t * W * 2N
  // Channel sums through shared memory (N = 16): lane (ch, half) stores its 16 values (dB,
  // then dC, of its 8 states) into row ch of red[16][32]; lane j then adds column j over
  // the 16 rows, the sum for kind j >> 4 and state j & 15 (so n_red = j). Float4 group g of
  // row ch sits at g ^ f(ch), f(ch) = (ch & 1) | (ch & 2) << 1: the 16-byte stores (8 lanes
  // per phase) and the column reads each touch 32 distinct banks.
  const int fch = (ch & 1) | ((ch & 2) << 1);
  float4* red_w = reinterpret_cast<float4*>(red + ch * 32);
  int rbuf = 0;  // float offset of this step's tile: 0 or kBwdCh * 32, alternating
  int rd_off[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) rd_off[c] = ((((lane >> 2) ^ ((c & 1) | ((c & 2) << 1))) << 2) | (lane & 3));

  stage_chunk<T, TG, N>(sg, p, b, p.nc - 1, d0, true, lane);
  for (int c = p.nc - 1; c >= 0; --c) {
    const int64_t t0 = (int64_t)c * kBwdK;
    const int kc = (int)((L - t0) < kBwdK ? (L - t0) : kBwdK);
    cp_async_wait_all();
    __syncwarp();
    prologue(true);
    if (c > 0) stage_chunk<T, TG, N>(sg, p, b, c - 1, d0, true, lane);
    // recompute the chunk's states from its checkpoint
    {
      const float2* ckp = reinterpret_cast<const float2*>(p.ck + (((int64_t)b * p.nc + c) * D + d) * N + nb);
#pragma unroll
      for (int q = 0; q < P2; ++q) h[q] = vd ? ckp[q] : make_float2(0.f, 0.f);
      // (the state after the last step stays in h: the reverse walk starts from it)
      // walked by pointer, as the reverse sweep below
      const float4* rsc = sc + ch;
      const float* rbc = bc + nb;
      float2* rhs = hs2 + lane;
#pragma unroll 4
      for (int k = 0; k < kc; ++k) {
#pragma unroll
        for (int q = 0; q < P2; ++q) rhs[q * 32] = h[q];  // the state before step k
        const float4 s = *rsc;
        const float2 dt2 = make_float2(s.x, s.x), du2 = make_float2(s.y, s.y);
        float2 b2[P2];
        load_pairs<P2>(rbc, b2);
#pragma unroll
        for (int q = 0; q < P2; ++q) h[q] = __ffma2_rn(decay2<kAccurate>(dt2, Av[q], A2[q]), h[q], __fmul2_rn(du2, b2[q]));
        rsc += kBwdCh;
        rbc += 2 * N;
        rhs += P2 * 32;
      }
    }
    // walk it backwards; h[] holds h_t of the current step (the chunk's last state first)
    const int64_t tl = t0 + kc - 1;
    TG* pdu = du + tl * D;
    TG* pddl = ddl + tl * D;
    TG* pdz = (dzp ? dzp : du) + tl * D;  // advanced always, written only with dz
    float* ppart = part + tl * pstride;
    const float4* scp = sc + (kc - 1) * kBwdCh + ch;
    const float2* sxp = sx + (kc - 1) * kBwdCh + ch;
    const float* bcp = bc + (kc - 1) * 2 * N + nb;
    const float2* hsp = hs2 + (kc - 1) * P2 * 32 + lane;
#pragma unroll 4
    for (int k = kc - 1; k >= 0; --k) {
      const float4 s = *scp;  // dt, dt u, dv, u
      const float2 sxv = *sxp;
      const float2 dt2 = make_float2(s.x, s.x), du2 = make_float2(s.y, s.y), dv2 = make_float2(s.z, s.z);
      float2 b2[P2], c2[P2];
      load_pairs<P2>(bcp, b2);
      load_pairs<P2>(bcp + N, c2);
      float2 vacc = make_float2(0.f, 0.f), sgB = make_float2(0.f, 0.f), sAg = make_float2(0.f, 0.f);
      float vr[NV];
#pragma unroll
      for (int q = 0; q < P2; ++q) {
        const float2 hp = hsp[q * 32];                        // h_{t-1}
        const float2 a = decay2<kAccurate>(dt2, Av[q], A2[q]);
        g[q] = __ffma2_rn(dv2, c2[q], g[q]);                  // g = dL/dh_t
        const float2 cv = __fmul2_rn(dv2, h[q]);              // dC_t: dv h_t
        vacc = __ffma2_rn(c2[q], h[q], vacc);                 // C_t . h_t
        const float2 bv = __fmul2_rn(g[q], du2);              // dB_t: g dt u
        sgB = __ffma2_rn(g[q], b2[q], sgB);                   // sum g B_t
        const float2 gah = __fmul2_rn(g[q], __fmul2_rn(a, hp));
        dA_acc[q] = __ffma2_rn(gah, dt2, dA_acc[q]);          // dA: g a h_{t-1} dt
        sAg = __ffma2_rn(kAccurate ? Av[q] : A2[q], gah, sAg); // sum A g a h_{t-1} (A log2 e on bf16)
        g[q] = __fmul2_rn(g[q], a);                           // dL/dh_{t-1} through the recurrence
        h[q] = hp;
        vr[2 * q] = bv.x;
        vr[2 * q + 1] = bv.y;
        vr[NH + 2 * q] = cv.x;
        vr[NH + 2 * q + 1] = cv.y;
      }
      float v = vacc.x + vacc.y, gb = sgB.x + sgB.y, ag = sAg.x + sAg.y;
      v += __shfl_xor_sync(0xffffffffu, v, 1);  // the channel's other half
      gb += __shfl_xor_sync(0xffffffffu, gb, 1);
      ag += __shfl_xor_sync(0xffffffffu, ag, 1);
      v = fmaf(Dk, s.w, v);                                         // read-out before the gate
      const float dux = fmaf(s.z, Dk, s.x * gb);                    // du = dv D + dt sum g B
      const float ddt = fmaf(s.w, gb, (kAccurate ? 1.f : kLn2) * ag);  // d(dt)
      const float dr = ddt * sxv.x;
      dD_acc = fmaf(s.z, s.w, dD_acc);
      dbias_acc += dr;
      if (vd) {  // both lanes of the channel hold the same sums and write the same values
        *pdu = from_f32<TG>(dux);
        *pddl = from_f32<TG>(dr);
        if (dzp) *pdz = from_f32<TG>(sxv.y * v);  // dz = dy v silu'(z)
      }
      pdu -= D;
      pddl -= D;
      pdz -= D;
      scp -= kBwdCh;
      sxp -= kBwdCh;
      bcp -= 2 * N;
      hsp -= P2 * 32;
      float sr;
      if constexpr (N == 16) {
        float4* rw = red_w + rbuf / 4;
        const float* rr = red + rbuf;
        rw[(2 * half) ^ fch] = make_float4(vr[0], vr[1], vr[2], vr[3]);
        rw[(2 * half + 1) ^ fch] = make_float4(vr[4], vr[5], vr[6], vr[7]);
        rw[(4 + 2 * half) ^ fch] = make_float4(vr[8], vr[9], vr[10], vr[11]);
        rw[(5 + 2 * half) ^ fch] = make_float4(vr[12], vr[13], vr[14], vr[15]);
        __syncwarp();
        sr = rr[rd_off[0]];
#pragma unroll
        for (int c = 1; c < kBwdCh; ++c) sr += rr[c * 32 + rd_off[c & 3]];
        rbuf ^= kBwdCh * 32;  // the next step writes the other tile; this one is rewritten two
                              // steps on, after the next step's barrier
      } else {
        sr = bwd_transpose_reduce<NV>(vr, lane);
      }
      if (writer) *ppart = sr;
      ppart -= pstride;
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
