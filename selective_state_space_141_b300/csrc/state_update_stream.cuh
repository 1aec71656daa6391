// state_update_stream.cuh -- the decode step (bf16 inputs, N = 16; plain, or with the
// forward pass's step-size map) as a streamed, persistent kernel.
//
// Same step and the same arithmetic as state_update_kernel<bf16, TY, 16, kExt> ("8.7
// State Space Models (Mamba)", section 5: O(1) work per generated token on a fixed d*n
// state; "Mamba and State Space Models", "Selective scan pseudo-code", one iteration of
// the loop body): for each channel (b, d), with dt = delta (kMap: softplus(delta + bias[d])
// or delta + bias[d] as the forward pass maps it) and x the token input (kConv: the
// block's causal conv + SiLU of it, silu(conv_b + w0 cs0 + w1 cs1 + w2 cs2 + w3 x) over the
// carried conv state, which is then shifted to (cs1, cs2, x))
//   state[n] = exp(dt A[d,n]) state[n] + dt B[b,n] x,   y = (C[b] . state + D x) silu(z)
//
// The step reads and writes the whole fp32 state once, so its time is the time to move
// those bytes. Here the bytes in flight per SM do not depend on the thread count: one
// producer thread per CTA streams tiles of kDecTile consecutive channels (their state and
// A rows, x, delta, z and the batch row's B and C) into a ring of kDecStages shared-memory
// stages with 1-D bulk copies, completion counted on an mbarrier per stage; the consumer
// threads update a tile from shared memory, write the state back with 16-byte stores and
// release the stage. CTAs are persistent (a fixed grid walks all tiles), so there is no
// tail of short-lived blocks. Every wait is bounded (tma.cuh).
#pragma once

#include "common.cuh"
#include "state_update.cuh"
#include "tma.cuh"

namespace ssm {

// Tile and ring depth measured on the 2.8B-shaped decode step (256 x 5120): 128 channels
// x 2 stages (17 KB each; several CTAs per SM) 29.9 us per step; 64 x 4: 31.6; 64 x 8:
// 37.2; 256 x 3: 30.6; 128 x 1 (no overlap): 34.8.
constexpr int kDecTile = 128;                 // channels per tile (D % kDecTile == 0)
constexpr int kDecStages = 2;                 // tiles in flight per CTA
constexpr int kDecConsumers = 2 * kDecTile;   // two threads per channel, 8 states each

struct alignas(16) DecStage {
  float state[kDecTile * 16];
  float A[kDecTile * 16];
  __nv_bfloat16 x[kDecTile];
  __nv_bfloat16 dl[kDecTile];
  __nv_bfloat16 z[kDecTile];
  __nv_bfloat16 B[16];
  __nv_bfloat16 C[16];
  float bias[kDecTile];  // kMap with delta_bias only
  float cw[kDecTile * 4];                // kConv: conv weights, 4 per channel
  float cb[kDecTile];                    // kConv with conv_b
  __nv_bfloat16 cs[kDecTile * 3 + 8];    // kConv: conv state, 3 per channel (+ pad to 16 B)
  int64_t d0;                            // the tile's first channel index d (written by the producer)
  int64_t pad;
};
static_assert(sizeof(DecStage) % 16 == 0, "stage members start 16-byte aligned");

constexpr int dec_stream_smem_bytes() { return kDecStages * (int)sizeof(DecStage) + 2 * kDecStages * 8; }

// Eight bf16 values (one 16-byte vector) to fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// grid: persistent (a multiple of the SM count, at most one CTA per tile); block:
// kDecConsumers consumer threads + one producer warp.
// wait_cycles: the limit of every wait (0: the default); skip_loads (failure-detection
// tests only): the producer issues no copies, so every consumer wait runs out.
// kMap: the step-size map (delta_bias, delta_softplus) is compiled in; kConv: the conv
// prologue (conv_w, conv_b, conv_state).
template <typename TY, bool kMap, bool kConv>
__global__ void __launch_bounds__(kDecConsumers + 32) state_update_stream(const DecodeParams p, int64_t ntiles,
                                                                          long long wait_cycles, int skip_loads) {
  extern __shared__ __align__(128) unsigned char smem[];
  DecStage* stg = reinterpret_cast<DecStage*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kDecStages * sizeof(DecStage));
  uint64_t* empty = full + kDecStages;
  const int tid = threadIdx.x;
  const long long lim = wait_cycles > 0 ? wait_cycles : kWaitCycles;
  constexpr int N = 16;
  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecConsumers / 32);
    }
    mbar_fence_init();
  }
  __syncthreads();

  const int64_t D = p.D;
  if (tid >= kDecConsumers) {  // ---------------- producer ----------------
    if (tid == kDecConsumers && !skip_loads) {
      const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.x);
      const __nv_bfloat16* dl = static_cast<const __nv_bfloat16*>(p.delta);
      const __nv_bfloat16* z = static_cast<const __nv_bfloat16*>(p.z);
      const __nv_bfloat16* B = static_cast<const __nv_bfloat16*>(p.B);
      const __nv_bfloat16* C = static_cast<const __nv_bfloat16*>(p.C);
      const bool bias = kMap && p.delta_bias, cbias = kConv && p.conv_b;
      const uint32_t tx = 2 * kDecTile * N * 4 + (z ? 3 : 2) * kDecTile * 2 + 2 * N * 2 + (bias ? kDecTile * 4 : 0) +
                          (kConv ? kDecTile * 4 * 4 + kDecTile * 3 * 2 : 0) + (cbias ? kDecTile * 4 : 0);
      int i = 0;
      for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
        const int s = i % kDecStages;
        if (i >= kDecStages && !mbar_wait(&empty[s], ((i / kDecStages) - 1) & 1, kErrWaitEmpty, lim)) break;
        DecStage& sg = stg[s];
        const int64_t c0 = tile * kDecTile, b = c0 / D, d0 = c0 - b * D;
        mbar_expect_tx(&full[s], tx);  // the copies first; the arrive after the tile's d0 below
        bulk_load(sg.state, p.state + c0 * N, kDecTile * N * 4, &full[s]);
        bulk_load(sg.A, p.A + d0 * N, kDecTile * N * 4, &full[s]);
        bulk_load(sg.x, x + c0, kDecTile * 2, &full[s]);
        bulk_load(sg.dl, dl + c0, kDecTile * 2, &full[s]);
        if (z) bulk_load(sg.z, z + c0, kDecTile * 2, &full[s]);
        bulk_load(sg.B, B + b * N, N * 2, &full[s]);
        bulk_load(sg.C, C + b * N, N * 2, &full[s]);
        if (bias) bulk_load(sg.bias, p.delta_bias + d0, kDecTile * 4, &full[s]);
        if (kConv) {
          bulk_load(sg.cw, p.conv_w + d0 * 4, kDecTile * 4 * 4, &full[s]);
          bulk_load(sg.cs, static_cast<const __nv_bfloat16*>(p.conv_state) + c0 * 3, kDecTile * 3 * 2, &full[s]);
          if (cbias) bulk_load(sg.cb, p.conv_b + d0, kDecTile * 4, &full[s]);
        }
        sg.d0 = d0;             // the tile's first channel index, for the consumers
        mbar_arrive(&full[s]);  // releases d0; the phase completes when the copies have landed
      }
      // Wait (bounded) for the copies still in flight before leaving.
      const int issued = i;
      for (int k = (issued > kDecStages ? issued - kDecStages : 0); k < issued; ++k)
        if (!mbar_wait(&full[k % kDecStages], (k / kDecStages) & 1, kErrWaitFull, lim)) break;
    }
    return;
  }

  // ---------------- consumers: thread = (channel j of the tile, state half g) ----------------
  const int j = tid >> 1, g = tid & 1, lane = tid & 31;
  // the step-size-map variant advances the tile's first channel, (tile * kDecTile) mod D, by a
  // fixed step per tile (measured faster there; the plain variant keeps the division)
  int64_t dt0 = ((int64_t)blockIdx.x * kDecTile) % D;
  const int64_t dstep = ((int64_t)gridDim.x * kDecTile) % D;
  int i = 0;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
    const int s = i % kDecStages;
    if (!mbar_wait(&full[s], (i / kDecStages) & 1, kErrWaitFull, lim)) break;
    const DecStage& sg = stg[s];
    const int64_t bd = tile * kDecTile + j;
    const __nv_bfloat16 xraw = sg.x[j];
    float x = __bfloat162float(xraw);
    __nv_bfloat16 cs1, cs2;
    if (kConv) {  // the block's causal conv + SiLU over (cs0, cs1, cs2, x), as state_update_kernel
      const float* w = sg.cw + j * 4;
      const __nv_bfloat16 cs0 = sg.cs[j * 3];
      cs1 = sg.cs[j * 3 + 1];
      cs2 = sg.cs[j * 3 + 2];
      float c = p.conv_b ? sg.cb[j] : 0.f;
      c = fmaf(w[0], __bfloat162float(cs0), c);
      c = fmaf(w[1], __bfloat162float(cs1), c);
      c = fmaf(w[2], __bfloat162float(cs2), c);
      c = fmaf(w[3], x, c);
      x = silu_precise(c);
    }
    float dt = __bfloat162float(sg.dl[j]);
    if (kMap && p.delta_bias) dt += sg.bias[j];
    if (kMap && p.delta_softplus) dt = softplus_precise(dt);
    const float zz = p.z ? __bfloat162float(sg.z[j]) : 0.f;
    // d: from the producer's tile offset with the conv prologue, by the running offset with
    // the step-size map, by division in the plain step (each measured fastest for its variant)
    const int64_t d = kConv ? sg.d0 + j : (kMap ? dt0 : (tile * kDecTile) % D) + j;
    if (kMap && !kConv) {
      dt0 += dstep;
      if (dt0 >= D) dt0 -= D;
    }
    const float dx = dt * x;
    const float4* sp = reinterpret_cast<const float4*>(sg.state + j * N + g * 8);
    const float4* ap = reinterpret_cast<const float4*>(sg.A + j * N + g * 8);
    float sv[8], av[8], Bv[8], Cv[8];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float4 s4 = sp[q], a4 = ap[q];
      sv[4 * q] = s4.x; sv[4 * q + 1] = s4.y; sv[4 * q + 2] = s4.z; sv[4 * q + 3] = s4.w;
      av[4 * q] = a4.x; av[4 * q + 1] = a4.y; av[4 * q + 2] = a4.z; av[4 * q + 3] = a4.w;
    }
    bf16x8_to_f32(reinterpret_cast<const uint4*>(sg.B)[g], Bv);
    bf16x8_to_f32(reinterpret_cast<const uint4*>(sg.C)[g], Cv);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // the stage is read: release it to the producer
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float a = decay<false>(dt, av[k], av[k] * kLog2e);  // as state_update_kernel (bf16)
      sv[k] = fmaf(a, sv[k], dx * Bv[k]);
      acc = fmaf(Cv[k], sv[k], acc);
    }
    float4* out = reinterpret_cast<float4*>(p.state + bd * N + g * 8);
    out[0] = make_float4(sv[0], sv[1], sv[2], sv[3]);
    out[1] = make_float4(sv[4], sv[5], sv[6], sv[7]);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (kConv && g == 0) {  // shift the conv state: (cs1, cs2, the raw input)
      __nv_bfloat16* cso = static_cast<__nv_bfloat16*>(p.conv_state) + bd * 3;
      cso[0] = cs1;
      cso[1] = cs2;
      cso[2] = xraw;
    }
    if (g == 0) {
      float o = acc;
      if (p.Dskip) o = fmaf(p.Dskip[d], x, o);
      if (p.z) o *= silu_precise(zz);
      static_cast<TY*>(p.y)[bd] = from_f32<TY>(o);
    }
  }
}

}  // namespace ssm
