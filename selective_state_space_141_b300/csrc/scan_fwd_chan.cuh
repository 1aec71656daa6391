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
//    arrive by TMA (3-D maps over (D, L, batch), zero fill past L) into an S-stage
//    shared-memory ring guarded by mbarriers:
//      warp 4 (one lane)  issues the TMA loads            full[s]  (tx bytes)
//      warp 5             converts B, C to fp32 in smem   ready[s] (32 arrivals)
//      warps 0..3         run the recurrence              empty[s] (4 arrivals)
//  * y of each chunk goes to a per-warp shared tile (double-buffered) and leaves by
//    one TMA store per warp per chunk; the store clips at L and D. The state h never
//    leaves registers; the final state is written once at the end.
//  * The softplus and gate switches are template parameters, so the unrolled step
//    loops carry no branches; an absent D skip or bias is a zero value.
// Every mbarrier wait is bounded (tma.cuh); on timeout a warp records the error word
// and returns, and the TMA issuer waits (bounded) for its loads still in flight.
#pragma once

#include "common.cuh"
#include "scan_fwd.cuh"
#include "tma.cuh"

namespace ssm {

constexpr int kChanCTA = 128;  // channels per CTA (4 consumer warps x 32 lanes)
constexpr int kChanThreads = 192;

template <typename TY, int N, int TC>
struct ChanLayout {
  static constexpr int kTileIO = TC * kChanCTA * 2;     // bf16 (TC x 128)
  static constexpr int kTileBC = TC * N * 2;            // bf16 (TC x N)
  static constexpr int kTileBC32 = TC * 2 * N * 4;      // fp32 (TC x [B | C])
  static constexpr int kStage = 3 * kTileIO + 2 * kTileBC + kTileBC32;
  static constexpr int kTileY = TC * 32 * (int)sizeof(TY);  // one warp's y tile (TC x 32)
  static_assert(kTileIO % 128 == 0 && kTileBC % 128 == 0 && kTileBC32 % 128 == 0 && kTileY % 128 == 0,
                "tile alignment");
};

template <typename TY, int N, int TC, int S>
constexpr int chan_smem_bytes() {
  using Lay = ChanLayout<TY, N, TC>;
  return S * Lay::kStage + 4 * 2 * Lay::kTileY + 3 * S * 8;
}

// Softplus of two steps for the bf16 path: max(r, 0) + log1p(e^-|r|), with 2^x and
// log2 on the SFU and the rest as packed f32x2 ops. Overflow-free for any r; for very
// negative r the rounding of 1 + e leaves an absolute error near 1e-7 in dt.
__device__ __forceinline__ float2 softplus2_fast(float2 r) {
  const float2 e = make_float2(ex2(fabsf(r.x) * -kLog2e), ex2(fabsf(r.y) * -kLog2e));
  const float2 op = __fadd2_rn(e, make_float2(1.f, 1.f));
  const float2 lg = make_float2(lg2(op.x), lg2(op.y));
  return __ffma2_rn(lg, make_float2(kLn2, kLn2), make_float2(fmaxf(r.x, 0.f), fmaxf(r.y, 0.f)));
}

// SiLU of two steps for the bf16 path: z sigmoid(z) = 0.5 z (1 + tanh(z / 2)), one SFU
// op per value.
__device__ __forceinline__ float2 silu2_fast(float2 z) {
  const float2 hz = __fmul2_rn(z, make_float2(0.5f, 0.5f));
  return __ffma2_rn(hz, make_float2(tanh_fast(hz.x), tanh_fast(hz.y)), hz);
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int32_t c0, int32_t c1,
                                             int32_t c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most n committed bulk stores still read shared memory.
template <int n>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(n) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

constexpr int kChanSub = 8;  // steps per sub-chunk

// The block's causal depthwise width-4 conv + SiLU computed on the fly ("Mamba and State
// Space Models", "The Mamba Block"): the u tile then holds the conv input x, and each
// lane (one channel) keeps its weights and the window of its last three inputs.
//   u_t = silu(b + w0 x_{t-3} + w1 x_{t-2} + w2 x_{t-1} + w3 x_t)
struct ConvLane {
  float2 w0, w1, w2, w3, b;  // each weight twice, for two steps per packed op
  float x0, x1, x2;          // x_{t-3}, x_{t-2}, x_{t-1}
};

// u of steps t and t+1 from their inputs xa = x_t, xb = x_{t+1}; advances the window.
template <bool kConv>
__device__ __forceinline__ float2 chan_u2(ConvLane& c, float xa, float xb) {
  if (!kConv) return make_float2(xa, xb);
  float2 acc = __ffma2_rn(c.w0, make_float2(c.x0, c.x1), c.b);
  acc = __ffma2_rn(c.w1, make_float2(c.x1, c.x2), acc);
  acc = __ffma2_rn(c.w2, make_float2(c.x2, xa), acc);
  acc = __ffma2_rn(c.w3, make_float2(xa, xb), acc);
  c.x0 = c.x2;
  c.x1 = xa;
  c.x2 = xb;
  return silu2_fast(acc);
}

// Zero-order hold: B-bar u = phi(z) (dt u) B with z = dt A and phi(z) = (e^z - 1) / z, from
// x = z log2(e) and a = 2^x already computed for the decay: (a - 1) / z where |z| >= 1/64
// (the cancellation in a - 1 then costs at most ~2e-5 of phi), the series 1 + z/2 + z^2/6
// below (remainder under 2e-7; exact at z = 0). phi times the pair of dt u values.
__device__ __forceinline__ float2 zoh_scale2(float2 x, float2 a, float2 dup) {
  const float2 z = __fmul2_rn(x, make_float2(kLn2, kLn2));
  const float2 ser = __ffma2_rn(z, __ffma2_rn(z, make_float2(1.f / 6.f, 1.f / 6.f), make_float2(0.5f, 0.5f)),
                                make_float2(1.f, 1.f));
  const float2 em1 = __fadd2_rn(a, make_float2(-1.f, -1.f));
  const float phx = fabsf(z.x) < 0.015625f ? ser.x : __fdividef(em1.x, z.x);
  const float phy = fabsf(z.y) < 0.015625f ? ser.y : __fdividef(em1.y, z.y);
  return __fmul2_rn(dup, make_float2(phx, phy));
}

// kChanSub steps of one lane (one channel, all N states), in three phases so that one
// warp per SM sub-partition finds independent work: (1) step sizes (independent
// softplus chains, two steps per packed op), (2) the recurrence (only h carries from
// step to step), (3) D skip, gate and y staging (two steps per packed op).
// kTail: steps at or past tc get dt = 0 and no input, so exp(0) = 1 exactly leaves h
// bit-for-bit unchanged (selects, not multiplies; those rows hold zero fill).
template <typename TY, int N, bool kSoftplus, bool kGate, bool kTail, bool kConv, bool kZoh = false>
__device__ __forceinline__ void chan_subchunk(const __nv_bfloat16* su, const __nv_bfloat16* sd,
                                              const __nv_bfloat16* sz, const float* bc, TY* yt, int t0, int tc,
                                              float bias, float Dk, const float2 (&A2)[N / 2], float2 (&h)[N / 2],
                                              ConvLane& cv) {
  float2 u2[kChanSub / 2], dt2[kChanSub / 2], du2[kChanSub / 2], y2[kChanSub / 2];
#pragma unroll
  for (int i = 0; i < kChanSub / 2; ++i) {
    const int t = t0 + 2 * i;
    u2[i] = chan_u2<kConv>(cv, __bfloat162float(su[t * kChanCTA]), __bfloat162float(su[(t + 1) * kChanCTA]));
    const float2 r = __fadd2_rn(make_float2(__bfloat162float(sd[t * kChanCTA]), __bfloat162float(sd[(t + 1) * kChanCTA])),
                                make_float2(bias, bias));
    float2 d = kSoftplus ? softplus2_fast(r) : r;
    if (kTail) d = make_float2(t < tc ? d.x : 0.f, t + 1 < tc ? d.y : 0.f);
    dt2[i] = d;
    du2[i] = __fmul2_rn(d, u2[i]);
    if (kTail) du2[i] = make_float2(t < tc ? du2[i].x : 0.f, t + 1 < tc ? du2[i].y : 0.f);
  }
  float yv[kChanSub];
#pragma unroll
  for (int i = 0; i < kChanSub; ++i) {
    const float dts = (i & 1) ? dt2[i / 2].y : dt2[i / 2].x;
    const float dus = (i & 1) ? du2[i / 2].y : du2[i / 2].x;
    const float2 dtp = make_float2(dts, dts), dup = make_float2(dus, dus);
    const float4* bc4 = reinterpret_cast<const float4*>(bc + (t0 + i) * 2 * N);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
      const float4 bq = bc4[q];
      const float4 cq = bc4[N / 4 + q];
      const float2 x0 = __fmul2_rn(dtp, A2[2 * q]);
      const float2 x1 = __fmul2_rn(dtp, A2[2 * q + 1]);
      const float2 a0 = make_float2(ex2(x0.x), ex2(x0.y));           // A-bar = exp(dt A)
      const float2 a1 = make_float2(ex2(x1.x), ex2(x1.y));
      const float2 b0 = __fmul2_rn(kZoh ? zoh_scale2(x0, a0, dup) : dup, make_float2(bq.x, bq.y));  // (dt u) B
      const float2 b1 = __fmul2_rn(kZoh ? zoh_scale2(x1, a1, dup) : dup, make_float2(bq.z, bq.w));
      h[2 * q] = __ffma2_rn(a0, h[2 * q], b0);                        // h = A-bar h + B-bar u
      h[2 * q + 1] = __ffma2_rn(a1, h[2 * q + 1], b1);
      acc0 = __ffma2_rn(make_float2(cq.x, cq.y), h[2 * q], acc0);    // C . h
      acc1 = __ffma2_rn(make_float2(cq.z, cq.w), h[2 * q + 1], acc1);
    }
    const float2 acc = __fadd2_rn(acc0, acc1);
    yv[i] = acc.x + acc.y;
  }
#pragma unroll
  for (int i = 0; i < kChanSub / 2; ++i) {
    const int t = t0 + 2 * i;
    y2[i] = __ffma2_rn(make_float2(Dk, Dk), u2[i], make_float2(yv[2 * i], yv[2 * i + 1]));
    if (kGate)
      y2[i] = __fmul2_rn(y2[i], silu2_fast(make_float2(__bfloat162float(sz[t * kChanCTA]),
                                                      __bfloat162float(sz[(t + 1) * kChanCTA]))));
    yt[t * 32] = from_f32<TY>(y2[i].x);
    yt[(t + 1) * 32] = from_f32<TY>(y2[i].y);
  }
}

// Aggregate pass over kChanSub steps: the recurrence from the given state without the
// read-out (no C, no y), plus the running sum of dt, from which the decay product of a
// whole segment is exp(A * sum dt). Same tail rule as chan_subchunk.
template <int N, bool kSoftplus, bool kTail, bool kConv, bool kZoh = false>
__device__ __forceinline__ void chan_subchunk_agg(const __nv_bfloat16* su, const __nv_bfloat16* sd, const float* bc,
                                                  int t0, int tc, float bias, const float2 (&A2)[N / 2],
                                                  float2 (&h)[N / 2], float& sdt, ConvLane& cv) {
  float2 dt2[kChanSub / 2], du2[kChanSub / 2];
#pragma unroll
  for (int i = 0; i < kChanSub / 2; ++i) {
    const int t = t0 + 2 * i;
    const float2 u2 = chan_u2<kConv>(cv, __bfloat162float(su[t * kChanCTA]), __bfloat162float(su[(t + 1) * kChanCTA]));
    const float2 r = __fadd2_rn(make_float2(__bfloat162float(sd[t * kChanCTA]), __bfloat162float(sd[(t + 1) * kChanCTA])),
                                make_float2(bias, bias));
    float2 d = kSoftplus ? softplus2_fast(r) : r;
    if (kTail) d = make_float2(t < tc ? d.x : 0.f, t + 1 < tc ? d.y : 0.f);
    dt2[i] = d;
    du2[i] = __fmul2_rn(d, u2);
    if (kTail) du2[i] = make_float2(t < tc ? du2[i].x : 0.f, t + 1 < tc ? du2[i].y : 0.f);
    sdt += d.x + d.y;
  }
#pragma unroll
  for (int i = 0; i < kChanSub; ++i) {
    const float dts = (i & 1) ? dt2[i / 2].y : dt2[i / 2].x;
    const float dus = (i & 1) ? du2[i / 2].y : du2[i / 2].x;
    const float2 dtp = make_float2(dts, dts), dup = make_float2(dus, dus);
    const float4* b4 = reinterpret_cast<const float4*>(bc + (t0 + i) * 2 * N);
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
      const float4 bq = b4[q];
      const float2 x0 = __fmul2_rn(dtp, A2[2 * q]);
      const float2 x1 = __fmul2_rn(dtp, A2[2 * q + 1]);
      const float2 a0 = make_float2(ex2(x0.x), ex2(x0.y));
      const float2 a1 = make_float2(ex2(x1.x), ex2(x1.y));
      h[2 * q] = __ffma2_rn(a0, h[2 * q], __fmul2_rn(kZoh ? zoh_scale2(x0, a0, dup) : dup, make_float2(bq.x, bq.y)));
      h[2 * q + 1] =
          __ffma2_rn(a1, h[2 * q + 1], __fmul2_rn(kZoh ? zoh_scale2(x1, a1, dup) : dup, make_float2(bq.z, bq.w)));
    }
  }
}

// kAgg = false: the full pass (y, and last_state from the last segment); with kCk it also
//               writes the state checkpoints (p.ck) for the backward pass.
// kAgg = true:  the aggregate pass of a segmented scan (seg_E, seg_P; no y), or of one
//               segment writing the checkpoints only.
// blockIdx = (channel block of 128, batch row, sequence segment).
// kConv: the u tensor holds the conv input x; u is its causal conv + SiLU (ConvLane).
template <typename TY, int N, int TC, int S, bool kSoftplus, bool kGate, bool kAgg, bool kConv, bool kCk = false,
          bool kZoh = false>
__global__ void __launch_bounds__(kChanThreads, 1)
scan_fwd_chan(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
              const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
              const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_y,
              const FwdParams p) {
  using Lay = ChanLayout<TY, N, TC>;
  constexpr bool kZ = kGate && !kAgg;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ytiles = smem + S * Lay::kStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(ytiles + 4 * 2 * Lay::kTileY);
  uint64_t* ready = full + S;
  uint64_t* empty = ready + S;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t b = (int32_t)blockIdx.y;
  const int seg = (int)blockIdx.z;
  const int64_t d0 = (int64_t)blockIdx.x * kChanCTA;
  const int64_t L = p.L, D = p.D;
  const int64_t t_begin = (int64_t)seg * p.seg_len;
  const int64_t t_end = (t_begin + p.seg_len) < L ? (t_begin + p.seg_len) : L;
  const int nchunks = (int)((t_end - t_begin + TC - 1) / TC);
  const long long lim = p.wait_cycles > 0 ? p.wait_cycles : kWaitCycles;

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
    if (lane == 0 && !p.fault_skip_loads) {
      prefetch_tensormap(&tm_u);
      prefetch_tensormap(&tm_dl);
      if (kZ) prefetch_tensormap(&tm_z);
      prefetch_tensormap(&tm_B);
      if (!kAgg) prefetch_tensormap(&tm_C);
      constexpr uint32_t tx = (kZ ? 3 : 2) * Lay::kTileIO + (kAgg ? 1 : 2) * Lay::kTileBC;
      int issued = 0;
      for (int k = 0; k < nchunks; ++k) {
        const int s = k % S;
        if (k >= S && !mbar_wait(&empty[s], ((k / S) - 1) & 1, kErrWaitEmpty, lim)) break;
        unsigned char* st = smem + s * Lay::kStage;
        mbar_arrive_expect_tx(&full[s], tx);
        const int32_t t0 = (int32_t)(t_begin + (int64_t)k * TC), col = (int32_t)d0;
        tma_load_3d(st, &tm_u, col, t0, b, &full[s]);
        tma_load_3d(st + Lay::kTileIO, &tm_dl, col, t0, b, &full[s]);
        if (kZ) tma_load_3d(st + 2 * Lay::kTileIO, &tm_z, col, t0, b, &full[s]);
        tma_load_3d(st + 3 * Lay::kTileIO, &tm_B, 0, t0, b, &full[s]);
        if (!kAgg) tma_load_3d(st + 3 * Lay::kTileIO + Lay::kTileBC, &tm_C, 0, t0, b, &full[s]);
        issued = k + 1;
      }
      // Wait (bounded) for the loads still in flight before leaving. The wait limit is far
      // longer than any copy takes (about a second against microseconds), so a load can
      // outlive the CTA only if the copy engine stopped completing copies altogether.
      for (int k = (issued > S ? issued - S : 0); k < issued; ++k)
        if (!mbar_wait(&full[k % S], (k / S) & 1, kErrWaitFull, lim)) break;
    }
    return;
  }

  if (warp == 5) {  // ---------------- B, C -> fp32 ----------------
    for (int k = 0; k < nchunks; ++k) {
      const int s = k % S;
      if (!mbar_wait(&full[s], (k / S) & 1, kErrWaitFull, lim)) return;
      const unsigned char* st = smem + s * Lay::kStage;
      const __nv_bfloat16* Bt = reinterpret_cast<const __nv_bfloat16*>(st + 3 * Lay::kTileIO);
      const __nv_bfloat16* Ct = reinterpret_cast<const __nv_bfloat16*>(st + 3 * Lay::kTileIO + Lay::kTileBC);
      float* bc = reinterpret_cast<float*>(smem + s * Lay::kStage + 3 * Lay::kTileIO + 2 * Lay::kTileBC);
      // Rows past this segment's end become exact zeros (they may hold the next
      // segment's data), so padded steps add nothing even for non-finite inputs there.
      const int64_t tk = t_begin + (int64_t)k * TC;
      const int tc = (int)((t_end - tk) < TC ? (t_end - tk) : TC);
#pragma unroll 4
      for (int i = lane; i < TC * N; i += 32) {
        const int t = i / N, n = i % N;
        bc[t * 2 * N + n] = t < tc ? __bfloat162float(Bt[i]) : 0.f;
        if (!kAgg) bc[t * 2 * N + N + n] = t < tc ? __bfloat162float(Ct[i]) : 0.f;
      }
      mbar_arrive(&ready[s]);
    }
    return;
  }

  // ---------------- consumers: warps 0..3, one channel per lane ----------------
  const int j = warp * 32 + lane;
  const int64_t d = d0 + j;
  const bool vd = d < D;
  const int64_t sidx = (((int64_t)seg * p.batch + b) * D + d) * N;  // [segment][batch][D][N]
  const SegY sy{p.seg_y, p.seg_y_bf16, L, D, p.seg_len, N};
  float2 A2[N / 2], h[N / 2];
#pragma unroll
  for (int q = 0; q < N / 2; ++q) {
    A2[q] = vd ? make_float2(p.A[d * N + 2 * q] * kLog2e, p.A[d * N + 2 * q + 1] * kLog2e)
               : make_float2(0.f, 0.f);
    if (vd && p.seg_y && !kAgg)  // start state from this segment's rows of y (read before any y store)
      h[q] = make_float2(seg_slot_load(sy, 0, seg, b, d, 2 * q), seg_slot_load(sy, 0, seg, b, d, 2 * q + 1));
    else
      h[q] = (vd && p.seg_h0) ? make_float2(p.seg_h0[sidx + 2 * q], p.seg_h0[sidx + 2 * q + 1])
                              : make_float2(0.f, 0.f);
  }
  const float bias = (vd && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const float Dk = (vd && p.Dskip) ? p.Dskip[d] : 0.f;
  unsigned char* ywarp = ytiles + warp * 2 * Lay::kTileY;  // this warp's two y tiles
  float sdt = 0.f;
  ConvLane cv{};
  if (kConv && vd) {
    const float* w = p.conv_w + d * 4;
    cv.w0 = make_float2(w[0], w[0]);
    cv.w1 = make_float2(w[1], w[1]);
    cv.w2 = make_float2(w[2], w[2]);
    cv.w3 = make_float2(w[3], w[3]);
    const float cb = p.conv_b ? p.conv_b[d] : 0.f;
    cv.b = make_float2(cb, cb);
    float xw[3] = {0.f, 0.f, 0.f};
    if (seg == 0) {  // the three inputs before the sequence: the carried conv state, or zeros
      if (p.conv_state) {
        const __nv_bfloat16* cs = static_cast<const __nv_bfloat16*>(p.conv_state) + ((int64_t)b * D + d) * 3;
        for (int k = 0; k < 3; ++k) xw[k] = __bfloat162float(cs[k]);
      }
    } else {  // a later segment: the three inputs before its first step
      const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.u);
      for (int k = 0; k < 3; ++k) xw[k] = __bfloat162float(x[((int64_t)b * L + t_begin - 3 + k) * D + d]);
    }
    cv.x0 = xw[0];
    cv.x1 = xw[1];
    cv.x2 = xw[2];
  }

  for (int k = 0; k < nchunks; ++k) {
    const int s = k % S;
    const uint32_t par = (k / S) & 1;
    if (!mbar_wait(&ready[s], par, kErrWaitReady, lim)) break;
    if (!mbar_wait(&full[s], par, kErrWaitFull, lim)) break;
    const unsigned char* st = smem + s * Lay::kStage;
    const __nv_bfloat16* su = reinterpret_cast<const __nv_bfloat16*>(st) + j;
    const __nv_bfloat16* sd = reinterpret_cast<const __nv_bfloat16*>(st + Lay::kTileIO) + j;
    const __nv_bfloat16* sz = reinterpret_cast<const __nv_bfloat16*>(st + 2 * Lay::kTileIO) + j;
    const float* bc = reinterpret_cast<const float*>(st + 3 * Lay::kTileIO + 2 * Lay::kTileBC);
    const int64_t tk = t_begin + (int64_t)k * TC;
    const int tc = (int)((t_end - tk) < TC ? (t_end - tk) : TC);
    // Checkpoints (the aggregate pass, or the full pass with kCk): the state before step
    // tk + t0, when that step starts a checkpoint chunk.
    auto checkpoint = [&](int t0) {
      if ((kAgg || kCk) && p.ck && vd && t0 % kCkSteps == 0) {
        float4* c4 = reinterpret_cast<float4*>(p.ck + (((int64_t)b * p.ck_nc + (tk + t0) / kCkSteps) * D + d) * N);
#pragma unroll
        for (int q = 0; q < N / 4; ++q) c4[q] = make_float4(h[2 * q].x, h[2 * q].y, h[2 * q + 1].x, h[2 * q + 1].y);
      }
    };
    if (kAgg) {
      if (tc == TC) {
        for (int t0 = 0; t0 < TC; t0 += kChanSub) {
          checkpoint(t0);
          chan_subchunk_agg<N, kSoftplus, false, kConv, kZoh>(su, sd, bc, t0, tc, bias, A2, h, sdt, cv);
        }
      } else {
        for (int t0 = 0; t0 < tc; t0 += kChanSub) {
          checkpoint(t0);
          chan_subchunk_agg<N, kSoftplus, true, kConv, kZoh>(su, sd, bc, t0, tc, bias, A2, h, sdt, cv);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      continue;
    }
    TY* ytile = reinterpret_cast<TY*>(ywarp + (k & 1) * Lay::kTileY);
    TY* yt = ytile + lane;
    // The tile written two chunks ago must have been read out by its TMA store.
    if (k >= 2) {
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
    }
    if (tc == TC) {
      for (int t0 = 0; t0 < TC; t0 += kChanSub) {
        checkpoint(t0);
        chan_subchunk<TY, N, kSoftplus, kGate, false, kConv, kZoh>(su, sd, sz, bc, yt, t0, tc, bias, Dk, A2, h, cv);
      }
    } else {
      for (int t0 = 0; t0 < tc; t0 += kChanSub) {
        checkpoint(t0);
        chan_subchunk<TY, N, kSoftplus, kGate, true, kConv, kZoh>(su, sd, sz, bc, yt, t0, tc, bias, Dk, A2, h, cv);
      }
    }
    // Release the input stage, then send this chunk's y tile (rows past L and columns
    // past D are clipped by the TMA store; segments start on chunk boundaries).
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    fence_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(&tm_y, ytile, (int32_t)(d0 + warp * 32), (int32_t)tk, b);
      bulk_commit();
    }
  }

  if (kAgg) {
    if (vd && p.seg_y) {
#pragma unroll
      for (int q = 0; q < N / 2; ++q) {
        seg_slot_store(sy, 1, seg, b, d, 2 * q, h[q].x);
        seg_slot_store(sy, 1, seg, b, d, 2 * q + 1, h[q].y);
        seg_slot_store(sy, 2, seg, b, d, 2 * q, ex2(A2[q].x * sdt));
        seg_slot_store(sy, 2, seg, b, d, 2 * q + 1, ex2(A2[q].y * sdt));
      }
    } else if (vd && p.seg_E) {
      float4* e4 = reinterpret_cast<float4*>(p.seg_E + sidx);
      float4* p4 = reinterpret_cast<float4*>(p.seg_P + sidx);
#pragma unroll
      for (int q = 0; q < N / 4; ++q) {
        e4[q] = make_float4(h[2 * q].x, h[2 * q].y, h[2 * q + 1].x, h[2 * q + 1].y);
        p4[q] = make_float4(ex2(A2[2 * q].x * sdt), ex2(A2[2 * q].y * sdt), ex2(A2[2 * q + 1].x * sdt),
                            ex2(A2[2 * q + 1].y * sdt));
      }
    }
    return;
  }
  if (lane == 0) bulk_wait_all();

  if (vd && p.last_state && seg == (int)gridDim.z - 1) {
    float4* ls = reinterpret_cast<float4*>(p.last_state + ((int64_t)b * D + d) * N);
#pragma unroll
    for (int q = 0; q < N / 4; ++q) ls[q] = make_float4(h[2 * q].x, h[2 * q].y, h[2 * q + 1].x, h[2 * q + 1].y);
  }
}

// Carry between sequence segments: for every (batch, channel, state) the segment
// aggregates (P_s, E_s) are pairs of the recurrence h -> P h + E, combined in time order
// by (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2) ("8.7 State Space Models (Mamba)", section
// 4.1 and "Mamba and State Space Models", "Hardware-Aware Parallel Scan": the recurrence
// is an associative scan). Element e of an item's scan is (1, h0) for e = 0 (h0 = 0 when
// absent) and segment e-1's aggregate otherwise; after an inclusive scan element e holds
// the state at the start of segment e.
//   * within a warp: a Hillis-Steele scan over 32 elements with __shfl_up_sync;
//   * across warps (nseg > 32: up to 128 segments over 4 warps): each warp's total goes
//     to shared memory and every warp composes the totals of the warps before it (the
//     block carry), then applies that carry to its elements.
// CTA of 128 threads; `wpi` warps per item (1, 2 or 4: ceil(nseg / 32)), 4 / wpi items
// per CTA. kInY: the values live in y (SegY), else flat [segment][batch * D * N] arrays.
template <bool kInY>
__global__ void __launch_bounds__(128) seg_carry_kernel(const SegY sy, const float* __restrict__ E,
                                                       const float* __restrict__ P, const float* __restrict__ h0,
                                                       float* __restrict__ H, int nseg, int wpi, int64_t nbdn) {
  __shared__ float2 tot[4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wi = warp % wpi;  // warp within the item
  const int64_t idx = (int64_t)blockIdx.x * (4 / wpi) + warp / wpi;
  const bool valid = idx < nbdn;
  const int e = wi * 32 + lane;  // scan element
  int n = 0;
  int64_t d = 0, b = 0;
  if (kInY && valid) {
    n = (int)(idx % sy.N);
    d = (idx / sy.N) % sy.D;
    b = idx / ((int64_t)sy.N * sy.D);
  }
  float a = 1.f, c = 0.f;
  if (valid) {
    if (e == 0) {
      c = h0 ? h0[idx] : 0.f;
    } else if (e < nseg) {
      a = kInY ? seg_slot_load(sy, 2, e - 1, b, d, n) : P[(int64_t)(e - 1) * nbdn + idx];
      c = kInY ? seg_slot_load(sy, 1, e - 1, b, d, n) : E[(int64_t)(e - 1) * nbdn + idx];
    }
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float a_up = __shfl_up_sync(0xffffffffu, a, off);
    const float c_up = __shfl_up_sync(0xffffffffu, c, off);
    if (lane >= off) {  // (a_up, c_up) o (a, c)
      c = fmaf(a, c_up, c);
      a = a * a_up;
    }
  }
  if (wpi > 1) {  // block carry: compose the totals of this item's earlier warps
    if (lane == 31) tot[warp] = make_float2(a, c);
    __syncthreads();
    float ca = 1.f, cc = 0.f;
    for (int w = warp - wi; w < warp; ++w) {
      const float2 t = tot[w];
      cc = fmaf(t.x, cc, t.y);
      ca *= t.x;
    }
    c = fmaf(a, cc, c);
  }
  if (valid && e < nseg) {
    if (kInY) seg_slot_store(sy, 0, e, b, d, n, c);
    else H[(int64_t)e * nbdn + idx] = c;
  }
}

}  // namespace ssm
