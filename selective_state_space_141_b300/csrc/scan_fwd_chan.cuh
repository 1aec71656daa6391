// scan_fwd_chan.cuh -- channel-parallel fused forward scan for bf16 I/O (sm_103a).
//
// Same computation as scan_fwd_generic (see scan_fwd.cuh for the definition and its
// sources), organised for B300:
//  * One lane owns one channel and ALL of its N states, so the read-out C.h is a
//    private sum (no cross-lane reduction) and B_t, C_t are warp-wide broadcasts.
//  * The per-state work runs on packed f32x2 FMA/FMUL (half the issue slots of
//    scalar FP32), the decay 2^(dt*A*log2 e) on the SFU: 4 FP32 ops + 1 ex2 per state
//    and step, which saturate the FP32 pipe (128/clk/SM) and the SFU (32 ex2/clk/SM)
//    at the same rate.
//  * A CTA covers 128 consecutive channels of one batch row and walks the sequence
//    in chunks of TC steps. Tiles of u, delta, z (TC x 128 bf16) and B, C (TC x N)
//    arrive by TMA into an S-stage shared-memory ring guarded by mbarriers:
//      warp 4 (one lane)  issues the TMA loads            full[s]  (tx bytes)
//      warp 5             converts B, C to fp32 in smem   ready[s] (32 arrivals)
//      warps 0..3         run the recurrence              empty[s] (4 arrivals)
//  * The state h never leaves registers; y goes straight to global memory, the final
//    state once at the end.
// Every mbarrier wait is bounded (tma.cuh); on timeout a warp records the error word
// and returns, and the TMA issuer waits (bounded) for its loads still in flight.
#pragma once

#include "common.cuh"
#include "scan_fwd.cuh"
#include "tma.cuh"

namespace ssm {

constexpr int kChanCTA = 128;  // channels per CTA (4 consumer warps x 32 lanes)
constexpr int kChanThreads = 192;

template <int N, int TC>
struct ChanLayout {
  static constexpr int kTileIO = TC * kChanCTA * 2;  // bf16 (TC x 128)
  static constexpr int kTileBC = TC * N * 2;         // bf16 (TC x N)
  static constexpr int kTileBC32 = TC * 2 * N * 4;   // fp32 (TC x [B | C])
  static constexpr int kStage = 3 * kTileIO + 2 * kTileBC + kTileBC32;
  static_assert(kTileIO % 128 == 0 && kTileBC % 128 == 0 && kTileBC32 % 128 == 0, "tile alignment");
};

template <int N, int TC, int S>
constexpr int chan_smem_bytes() {
  return S * ChanLayout<N, TC>::kStage + 3 * S * 8;
}

// Softplus for the bf16 path: 2^x and log2 on the SFU; e^r below 2^-10 uses
// log1p(e) ~ e (1 - e/2), where forming 1 + e would lose the low bits.
__device__ __forceinline__ float softplus_fast(float r) {
  const float e = ex2(r * kLog2e);
  const float lg = lg2(1.f + e) * kLn2;
  const float small = e * fmaf(-0.5f, e, 1.f);
  const float v = e < 0.0009765625f ? small : lg;
  return r > 20.f ? r : v;
}

// SiLU for the bf16 path: z sigmoid(z) = 0.5 z (1 + tanh(z / 2)), one SFU op.
__device__ __forceinline__ float silu_fast(float z) {
  const float hz = 0.5f * z;
  return fmaf(hz, tanh_fast(hz), hz);
}

template <typename TY, int N, int TC, int S>
__global__ void __launch_bounds__(kChanThreads, 1)
scan_fwd_chan(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
              const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
              const __grid_constant__ CUtensorMap tm_C, const FwdParams p) {
  using Lay = ChanLayout<N, TC>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Lay::kStage);
  uint64_t* ready = full + S;
  uint64_t* empty = ready + S;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b = blockIdx.y;
  const int64_t d0 = (int64_t)blockIdx.x * kChanCTA;
  const int64_t L = p.L, D = p.D;
  const int nchunks = (int)((L + TC - 1) / TC);
  const bool has_z = p.z != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&ready[s], 32);
      mbar_init(&empty[s], 4);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 4) {  // ---------------- TMA issuer ----------------
    if (lane == 0) {
      prefetch_tensormap(&tm_u);
      prefetch_tensormap(&tm_dl);
      if (has_z) prefetch_tensormap(&tm_z);
      prefetch_tensormap(&tm_B);
      prefetch_tensormap(&tm_C);
      const uint32_t tx = (has_z ? 3 : 2) * Lay::kTileIO + 2 * Lay::kTileBC;
      int issued = 0;
      for (int k = 0; k < nchunks; ++k) {
        const int s = k % S;
        if (k >= S && !mbar_wait(&empty[s], ((k / S) - 1) & 1, kErrWaitEmpty)) break;
        unsigned char* st = smem + s * Lay::kStage;
        mbar_arrive_expect_tx(&full[s], tx);
        const int32_t row = (int32_t)(b * L + (int64_t)k * TC);
        const int32_t col = (int32_t)d0;
        tma_load_2d(st, &tm_u, col, row, &full[s]);
        tma_load_2d(st + Lay::kTileIO, &tm_dl, col, row, &full[s]);
        if (has_z) tma_load_2d(st + 2 * Lay::kTileIO, &tm_z, col, row, &full[s]);
        tma_load_2d(st + 3 * Lay::kTileIO, &tm_B, 0, row, &full[s]);
        tma_load_2d(st + 3 * Lay::kTileIO + Lay::kTileBC, &tm_C, 0, row, &full[s]);
        issued = k + 1;
      }
      // Never leave with loads in flight into this CTA's shared memory.
      for (int k = (issued > S ? issued - S : 0); k < issued; ++k)
        if (!mbar_wait(&full[k % S], (k / S) & 1, kErrWaitFull)) break;
    }
    return;
  }

  if (warp == 5) {  // ---------------- B, C -> fp32 ----------------
    for (int k = 0; k < nchunks; ++k) {
      const int s = k % S;
      if (!mbar_wait(&full[s], (k / S) & 1, kErrWaitFull)) return;
      const unsigned char* st = smem + s * Lay::kStage;
      const __nv_bfloat16* Bt = reinterpret_cast<const __nv_bfloat16*>(st + 3 * Lay::kTileIO);
      const __nv_bfloat16* Ct = reinterpret_cast<const __nv_bfloat16*>(st + 3 * Lay::kTileIO + Lay::kTileBC);
      float* bc = reinterpret_cast<float*>(smem + s * Lay::kStage + 3 * Lay::kTileIO + 2 * Lay::kTileBC);
#pragma unroll 4
      for (int i = lane; i < TC * N; i += 32) {
        const int t = i / N, n = i % N;
        bc[t * 2 * N + n] = __bfloat162float(Bt[i]);
        bc[t * 2 * N + N + n] = __bfloat162float(Ct[i]);
      }
      mbar_arrive(&ready[s]);
    }
    return;
  }

  // ---------------- consumers: warps 0..3, one channel per lane ----------------
  const int j = warp * 32 + lane;
  const int64_t d = d0 + j;
  const bool vd = d < D;
  float2 A2[N / 2], h[N / 2];
#pragma unroll
  for (int q = 0; q < N / 2; ++q) {
    A2[q] = vd ? make_float2(p.A[d * N + 2 * q] * kLog2e, p.A[d * N + 2 * q + 1] * kLog2e)
               : make_float2(0.f, 0.f);
    h[q] = make_float2(0.f, 0.f);
  }
  const float bias = (vd && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const float Dk = (vd && p.Dskip) ? p.Dskip[d] : 0.f;
  const bool has_D = p.Dskip != nullptr;
  const bool sp = p.delta_softplus != 0;
  TY* __restrict__ yout = static_cast<TY*>(p.y) + b * L * D + d;

  for (int k = 0; k < nchunks; ++k) {
    const int s = k % S;
    const uint32_t par = (k / S) & 1;
    if (!mbar_wait(&ready[s], par, kErrWaitReady)) return;
    if (!mbar_wait(&full[s], par, kErrWaitFull)) return;
    const unsigned char* st = smem + s * Lay::kStage;
    const __nv_bfloat16* su = reinterpret_cast<const __nv_bfloat16*>(st) + j;
    const __nv_bfloat16* sd = reinterpret_cast<const __nv_bfloat16*>(st + Lay::kTileIO) + j;
    const __nv_bfloat16* sz = reinterpret_cast<const __nv_bfloat16*>(st + 2 * Lay::kTileIO) + j;
    const float* bc = reinterpret_cast<const float*>(st + 3 * Lay::kTileIO + 2 * Lay::kTileBC);
    const int tc = (int)((L - (int64_t)k * TC) < TC ? (L - (int64_t)k * TC) : TC);
    TY* yk = yout + (int64_t)k * TC * D;

#pragma unroll 2
    for (int t = 0; t < tc; ++t) {
      const float uu = __bfloat162float(su[t * kChanCTA]);
      const float r = __bfloat162float(sd[t * kChanCTA]) + bias;
      const float dt = sp ? softplus_fast(r) : r;
      const float du = dt * uu;
      const float2 dt2 = make_float2(dt, dt), du2 = make_float2(du, du);
      const float4* bc4 = reinterpret_cast<const float4*>(bc + t * 2 * N);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < N / 4; ++q) {
        const float4 bq = bc4[q];
        const float4 cq = bc4[N / 4 + q];
        const float2 x0 = __fmul2_rn(dt2, A2[2 * q]);
        const float2 x1 = __fmul2_rn(dt2, A2[2 * q + 1]);
        const float2 a0 = make_float2(ex2(x0.x), ex2(x0.y));           // A-bar = exp(dt A)
        const float2 a1 = make_float2(ex2(x1.x), ex2(x1.y));
        const float2 b0 = __fmul2_rn(du2, make_float2(bq.x, bq.y));     // (dt u) B
        const float2 b1 = __fmul2_rn(du2, make_float2(bq.z, bq.w));
        h[2 * q] = __ffma2_rn(a0, h[2 * q], b0);                        // h = A-bar h + B-bar u
        h[2 * q + 1] = __ffma2_rn(a1, h[2 * q + 1], b1);
        acc0 = __ffma2_rn(make_float2(cq.x, cq.y), h[2 * q], acc0);    // C . h
        acc1 = __ffma2_rn(make_float2(cq.z, cq.w), h[2 * q + 1], acc1);
      }
      float v = (acc0.x + acc0.y) + (acc1.x + acc1.y);
      if (has_D) v = fmaf(Dk, uu, v);
      if (has_z) v *= silu_fast(__bfloat162float(sz[t * kChanCTA]));
      if (vd) yk[(int64_t)t * D] = from_f32<TY>(v);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  if (vd && p.last_state) {
    float4* ls = reinterpret_cast<float4*>(p.last_state + (b * D + d) * N);
#pragma unroll
    for (int q = 0; q < N / 4; ++q) ls[q] = make_float4(h[2 * q].x, h[2 * q].y, h[2 * q + 1].x, h[2 * q + 1].y);
  }
}

}  // namespace ssm
