// ssd_fwd.cuh -- Mamba-2 SSD forward (scalar decay per head), chunked, sm_103a.
//
// Per batch row b and head h (group g of B, C), with a P x N state S:
//   dt = delta[b,t,h] + dt_bias[h] (softplus when asked)      a_t = exp(dt A[h])
//   S_t = a_t S_{t-1} + dt x_t B_t^T                           y_t = S_t C_t + D[h] x_t
// ("Mamba and State Space Models", "Mamba-2 and State Space Duality"; "8.7 State Space
// Models (Mamba)", Mamba-2: A-bar_t = a_t I per head). The sequence is cut into chunks of
// Q = 64 steps; inside a chunk the recurrence is the masked quadratic (dual) form, outside
// it the state is carried: with cs_j = sum_{k<=j} dt_k A (within the chunk),
//   Y   = W X + diag(exp(cs)) C S_prev^T + D X,   W_ji = (C_j . B_i) exp(cs_j - cs_i) dt_i (j >= i)
//   S   = exp(cs_end) S_prev + X^T diag(w) B,      w_i  = exp(cs_end - cs_i) dt_i
// (W and w B reach the tensor cores as bf16 high + low pairs, ~16 significant bits: a
// single bf16 rounding of these products of inputs would cost 2^-9 of |y| per term, and
// w B feeds the carried state every chunk, where that rounding accumulates)
// The four contractions (C B^T, W X, C S^T, X^T (w B)) run on the tensor cores
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation); the state stays on chip in fp32
// (with a bf16 copy as the operand of C S^T) for the whole sequence: one CTA of 8 warps
// per (batch, head) walks the chunks in order, prefetching the next chunk's inputs into
// registers while the current one is computed.
#pragma once

#include "common.cuh"

namespace ssm {

struct SsdParams {
  const __nv_bfloat16* x;      // (batch, L, H, P)
  const __nv_bfloat16* delta;  // (batch, L, H)
  const float* A;              // (H)
  const __nv_bfloat16* B;      // (batch, L, G, N)
  const __nv_bfloat16* C;      // (batch, L, G, N)
  const float* Dskip;          // (H), nullable
  const float* dt_bias;        // (H), nullable
  int dt_softplus;
  const float* h0;             // (batch, H, P, N), nullable
  void* y;                     // (batch, L, H, P), bf16 or f32
  float* last_state;           // (batch, H, P, N), nullable
  int64_t batch, L, H, G;
  // chunk-parallel schedule (workspace): per (b, c, h) the chunk's own state
  // contribution S_c (fp32, P x N), the state entering the chunk (bf16, P x N), and the
  // chunk's decay exp(sum dt A)
  float* ws_S;
  __nv_bfloat16* ws_H;
  float* ws_dec;
  int nc;
};

constexpr int kSsdQ = 64;
constexpr int kSsdThreads = 256;
constexpr int kSsdPad = 8;  // bf16 elements of row padding: conflict-free fragment loads

template <int P, int N>
constexpr int ssd_smem_bytes() {
  constexpr int LQ = kSsdQ + kSsdPad, LN = N + kSsdPad;
  return 2 * (P * LQ + 2 * kSsdQ * LN + 2 * N * LQ + 2 * kSsdQ * LQ + P * LN) + 4 * (P * N + 2 * kSsdQ);
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// A fragment (16 x 16 at (m0, k0)) of a row-major [m][k] bf16 matrix with row stride ld.
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], const __nv_bfloat16* M, int ld, int m0, int k0, int lane) {
  const int g = lane >> 2, t = lane & 3;
  a[0] = *reinterpret_cast<const uint32_t*>(M + (m0 + g) * ld + k0 + 2 * t);
  a[1] = *reinterpret_cast<const uint32_t*>(M + (m0 + g + 8) * ld + k0 + 2 * t);
  a[2] = *reinterpret_cast<const uint32_t*>(M + (m0 + g) * ld + k0 + 8 + 2 * t);
  a[3] = *reinterpret_cast<const uint32_t*>(M + (m0 + g + 8) * ld + k0 + 8 + 2 * t);
}
// B fragment (16 x 8, k x n, at (k0, n0)) of a matrix stored as [n][k] (row stride ld).
__device__ __forceinline__ void frag_b(uint32_t (&b)[2], const __nv_bfloat16* M, int ld, int n0, int k0, int lane) {
  const int g = lane >> 2, t = lane & 3;
  b[0] = *reinterpret_cast<const uint32_t*>(M + (n0 + g) * ld + k0 + 2 * t);
  b[1] = *reinterpret_cast<const uint32_t*>(M + (n0 + g) * ld + k0 + 8 + 2 * t);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Registers holding one chunk's inputs (prefetched while the previous chunk computes).
template <int P, int N>
struct SsdChunkRegs {
  static constexpr int kX = kSsdQ * P / 8 / kSsdThreads;   // uint4 (8 bf16) per thread
  static constexpr int kBC = kSsdQ * N / 8 / kSsdThreads;
  uint4 x[kX], b[kBC], c[kBC];
  float dt;
};

template <int P, int N, bool kC = true>
__device__ __forceinline__ void ssd_fetch(SsdChunkRegs<P, N>& r, const SsdParams& p, int64_t b, int64_t h, int64_t g,
                                          int64_t t0, int tid) {
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int k = 0; k < SsdChunkRegs<P, N>::kX; ++k) {
    const int i = tid + k * kSsdThreads, t = i % kSsdQ, p0 = (i / kSsdQ) * 8;
    r.x[k] = t0 + t < p.L ? *reinterpret_cast<const uint4*>(p.x + ((b * p.L + t0 + t) * p.H + h) * P + p0) : z4;
  }
#pragma unroll
  for (int k = 0; k < SsdChunkRegs<P, N>::kBC; ++k) {
    const int i = tid + k * kSsdThreads, t = i / (N / 8), n0 = (i % (N / 8)) * 8;
    const bool v = t0 + t < p.L;
    const int64_t o = ((b * p.L + t0 + t) * p.G + g) * N + n0;
    r.b[k] = v ? *reinterpret_cast<const uint4*>(p.B + o) : z4;
    if (kC) r.c[k] = v ? *reinterpret_cast<const uint4*>(p.C + o) : z4;
  }
  r.dt = 0.f;
  if (tid < kSsdQ && t0 + tid < p.L) {
    float rr = __bfloat162float(p.delta[(b * p.L + t0 + tid) * p.H + h]) + (p.dt_bias ? p.dt_bias[h] : 0.f);
    r.dt = p.dt_softplus ? softplus_precise(rr) : rr;
  }
}

template <int P, int N, bool kC = true>
__device__ __forceinline__ void ssd_store(const SsdChunkRegs<P, N>& r, __nv_bfloat16* XT, __nv_bfloat16* Bs,
                                          __nv_bfloat16* Cs, float* dts, int tid) {
  constexpr int LQ = kSsdQ + kSsdPad, LN = N + kSsdPad;
#pragma unroll
  for (int k = 0; k < SsdChunkRegs<P, N>::kX; ++k) {
    const int i = tid + k * kSsdThreads, t = i % kSsdQ, p0 = (i / kSsdQ) * 8;
    const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(&r.x[k]);
#pragma unroll
    for (int e = 0; e < 8; ++e) XT[(p0 + e) * LQ + t] = v[e];  // transposed: [p][t]
  }
#pragma unroll
  for (int k = 0; k < SsdChunkRegs<P, N>::kBC; ++k) {
    const int i = tid + k * kSsdThreads, t = i / (N / 8), n0 = (i % (N / 8)) * 8;
    *reinterpret_cast<uint4*>(Bs + t * LN + n0) = r.b[k];
    if (kC) *reinterpret_cast<uint4*>(Cs + t * LN + n0) = r.c[k];
  }
  if (tid < kSsdQ) dts[tid] = r.dt;
}

// grid (H, batch), block 256 (8 warps), dynamic smem ssd_smem_bytes<P, N>().
template <int P, int N, typename TY>
__global__ void __launch_bounds__(kSsdThreads, 1) ssd_fwd_kernel(const SsdParams p) {
  constexpr int Q = kSsdQ, LQ = Q + kSsdPad, LN = N + kSsdPad;
  static_assert(P == 64 || P == 128, "head dim");
  static_assert(N == 64 || N == 128, "state dim");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* XT = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [P][LQ]   X^T of the chunk
  __nv_bfloat16* Bs = XT + P * LQ;                                  // [Q][LN]   B rows
  __nv_bfloat16* Cs = Bs + Q * LN;                                  // [Q][LN]   C rows
  __nv_bfloat16* wBT = Cs + Q * LN;                                 // [N][LQ]   (w B)^T, bf16 high part
  __nv_bfloat16* wBL = wBT + N * LQ;                                // [N][LQ]   (w B)^T - high part, bf16
  __nv_bfloat16* Ws = wBL + N * LQ;                                 // [Q][LQ]   masked decayed C B^T, high
  __nv_bfloat16* WsL = Ws + Q * LQ;                                 // [Q][LQ]   its low part
  __nv_bfloat16* Hb = WsL + Q * LQ;                                 // [P][LN]   state, bf16 copy
  float* Hf = reinterpret_cast<float*>(Hb + P * LN);                // [P][N]    state, fp32
  float* dts = Hf + P * N;                                          // [Q]
  float* cs = dts + Q;                                              // [Q]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int64_t h = blockIdx.x, b = blockIdx.y, g = h / (p.H / p.G);
  const float Ah = p.A[h], Dh = p.Dskip ? p.Dskip[h] : 0.f;

  for (int i = tid; i < P * N; i += kSsdThreads) {
    const float v = p.h0 ? p.h0[(b * p.H + h) * P * N + i] : 0.f;
    Hf[i] = v;
    Hb[(i / N) * LN + i % N] = __float2bfloat16_rn(v);
  }
  const int nc = (int)((p.L + Q - 1) / Q);
  SsdChunkRegs<P, N> nxt;
  if (nc > 0) {
    ssd_fetch<P, N>(nxt, p, b, h, g, 0, tid);
    ssd_store<P, N>(nxt, XT, Bs, Cs, dts, tid);
  }
  __syncthreads();

  for (int c = 0; c < nc; ++c) {
    const int64_t t0 = (int64_t)c * Q;
    const int tc = (int)((p.L - t0) < Q ? (p.L - t0) : Q);
    if (c + 1 < nc) ssd_fetch<P, N>(nxt, p, b, h, g, t0 + Q, tid);  // in flight during this chunk

    // cumulative decay exponent within the chunk (padded steps have dt = 0)
    if (warp == 0) {
      const float v0 = dts[2 * lane] * Ah, v1 = dts[2 * lane + 1] * Ah;
      float s = v0 + v1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float up = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += up;
      }
      const float ex = s - (v0 + v1);
      cs[2 * lane] = ex + v0;
      cs[2 * lane + 1] = ex + v0 + v1;
    }
    __syncthreads();
    const float cs_end = cs[Q - 1];

    // (w B)^T with w_t = exp(cs_end - cs_t) dt_t, as a bf16 pair high + low: this operand
    // feeds the carried state every chunk, where a single bf16 rounding would accumulate
    for (int i = tid; i < Q * N; i += kSsdThreads) {
      const int t = i % Q, n = i / Q;
      const float v = __bfloat162float(Bs[t * LN + n]) * __expf(cs_end - cs[t]) * dts[t];
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      wBT[n * LQ + t] = hi;
      wBL[n * LQ + t] = __float2bfloat16_rn(v - __bfloat162float(hi));
    }
    // W = C B^T masked to j >= i and decayed: warp -> 16 rows (m-tile), 32 columns
    {
      const int mt = warp & 3, nh = warp >> 2;
      float acc[4][4] = {};
#pragma unroll
      for (int k0 = 0; k0 < N; k0 += 16) {
        uint32_t a[4];
        frag_a(a, Cs, LN, mt * 16, k0, lane);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          uint32_t bb[2];
          frag_b(bb, Bs, LN, nh * 32 + nt * 8, k0, lane);
          mma_16816(acc[nt], a, bb);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int j = mt * 16 + gq + 8 * hf, i0 = nh * 32 + nt * 8 + 2 * tq;
          const float w0 = j >= i0 ? acc[nt][2 * hf] * __expf(cs[j] - cs[i0]) * dts[i0] : 0.f;
          const float w1 = j >= i0 + 1 ? acc[nt][2 * hf + 1] * __expf(cs[j] - cs[i0 + 1]) * dts[i0 + 1] : 0.f;
          const __nv_bfloat162 hi = __floats2bfloat162_rn(w0, w1);
          *reinterpret_cast<__nv_bfloat162*>(Ws + j * LQ + i0) = hi;
          *reinterpret_cast<uint32_t*>(WsL + j * LQ + i0) =
              pack_bf16(w0 - __low2float(hi), w1 - __high2float(hi));
        }
      }
    }
    __syncthreads();

    // Y = W X + diag(exp(cs)) C S_prev^T + D X: warp -> 16 rows, P/2 columns
    {
      constexpr int NT = P / 16;
      const int mt = warp & 3, nh = warp >> 2;
      float ad[NT][4] = {}, ao[NT][4] = {};
#pragma unroll
      for (int k0 = 0; k0 < Q; k0 += 16) {
        uint32_t a[4], al[4];
        frag_a(a, Ws, LQ, mt * 16, k0, lane);
        frag_a(al, WsL, LQ, mt * 16, k0, lane);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          uint32_t bb[2];
          frag_b(bb, XT, LQ, nh * (P / 2) + nt * 8, k0, lane);
          mma_16816(ad[nt], a, bb);
          mma_16816(ad[nt], al, bb);
        }
      }
#pragma unroll
      for (int k0 = 0; k0 < N; k0 += 16) {
        uint32_t a[4];
        frag_a(a, Cs, LN, mt * 16, k0, lane);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          uint32_t bb[2];
          frag_b(bb, Hb, LN, nh * (P / 2) + nt * 8, k0, lane);
          mma_16816(ao[nt], a, bb);
        }
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int j = mt * 16 + gq + 8 * hf;
        if (j < tc) {
          const float e = __expf(cs[j]);
          TY* yrow = static_cast<TY*>(p.y) + ((b * p.L + t0 + j) * p.H + h) * P;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int pc = nh * (P / 2) + nt * 8 + 2 * tq;
            const float v0 = ad[nt][2 * hf] + e * ao[nt][2 * hf] + Dh * __bfloat162float(XT[pc * LQ + j]);
            const float v1 = ad[nt][2 * hf + 1] + e * ao[nt][2 * hf + 1] + Dh * __bfloat162float(XT[(pc + 1) * LQ + j]);
            if (sizeof(TY) == 2)
              *reinterpret_cast<uint32_t*>(yrow + pc) = pack_bf16(v0, v1);
            else
              *reinterpret_cast<float2*>(yrow + pc) = make_float2(v0, v1);
          }
        }
      }
    }
    __syncthreads();  // every read of the old state is done

    // S = exp(cs_end) S_prev + X^T (w B)
    {
      constexpr int MT = P / 16, WPM = 8 / MT, NTW = (N / 8) / WPM;
      const int mt = warp % MT, nq = warp / MT;
      float acc[NTW][4] = {};
#pragma unroll
      for (int k0 = 0; k0 < Q; k0 += 16) {
        uint32_t a[4];
        frag_a(a, XT, LQ, mt * 16, k0, lane);
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          uint32_t bb[2];
          frag_b(bb, wBT, LQ, (nq * NTW + nt) * 8, k0, lane);
          mma_16816(acc[nt], a, bb);
          frag_b(bb, wBL, LQ, (nq * NTW + nt) * 8, k0, lane);
          mma_16816(acc[nt], a, bb);
        }
      }
      const float dec = __expf(cs_end);
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int pr = mt * 16 + gq + 8 * hf, nc0 = (nq * NTW + nt) * 8 + 2 * tq;
          float2* hp = reinterpret_cast<float2*>(Hf + pr * N + nc0);
          const float2 old = *hp;
          const float2 nw = make_float2(fmaf(dec, old.x, acc[nt][2 * hf]), fmaf(dec, old.y, acc[nt][2 * hf + 1]));
          *hp = nw;
          *reinterpret_cast<uint32_t*>(Hb + pr * LN + nc0) = pack_bf16(nw.x, nw.y);
        }
      }
    }
    __syncthreads();
    if (c + 1 < nc) {
      ssd_store<P, N>(nxt, XT, Bs, Cs, dts, tid);
      __syncthreads();
    }
  }

  if (p.last_state)
    for (int i = tid; i < P * N; i += kSsdThreads) p.last_state[(b * p.H + h) * P * N + i] = Hf[i];
}

// ---- chunk-parallel schedule ----------------------------------------------------------
// Pass 1 (grid (nc, H, batch)): the state each chunk adds from zero, S_c = X^T diag(w) B,
// and its decay exp(cs_end). Pass 2 (element-wise): H_0 = h0, H_{c+1} = dec_c H_c + S_c,
// storing every entering state H_c (bf16: the operand of the read-out) and the final
// state. Pass 3 (grid (nc, H, batch)): Y = W X + diag(exp(cs)) C H_c^T + D X. The same
// per-chunk arithmetic as ssd_fwd_kernel, spread over every chunk at once.

template <int P, int N>
constexpr int ssd_state_smem_bytes() {
  constexpr int LQ = kSsdQ + kSsdPad;
  return 2 * (P * LQ + 2 * N * LQ + kSsdQ * (N + kSsdPad)) + 4 * 2 * kSsdQ;
}
template <int P, int N>
constexpr int ssd_scan_smem_bytes() {
  constexpr int LQ = kSsdQ + kSsdPad, LN = N + kSsdPad;
  return 2 * (P * LQ + 2 * kSsdQ * LN + 2 * kSsdQ * LQ + P * LN) + 4 * 2 * kSsdQ;
}

// cs_j = sum_{k <= j} dt_k A over the chunk (warp 0; dt = 0 on padded steps).
__device__ __forceinline__ void ssd_cumsum(const float* dts, float* cs, float Ah, int warp, int lane) {
  if (warp == 0) {
    const float v0 = dts[2 * lane] * Ah, v1 = dts[2 * lane + 1] * Ah;
    float s = v0 + v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float up = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += up;
    }
    const float ex = s - (v0 + v1);
    cs[2 * lane] = ex + v0;
    cs[2 * lane + 1] = ex + v0 + v1;
  }
}

template <int P, int N>
__global__ void __launch_bounds__(kSsdThreads) ssd_chunk_state_kernel(const SsdParams p) {
  constexpr int Q = kSsdQ, LQ = Q + kSsdPad, LN = N + kSsdPad;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* XT = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [P][LQ]
  __nv_bfloat16* wBT = XT + P * LQ;                                 // [N][LQ] high
  __nv_bfloat16* wBL = wBT + N * LQ;                                // [N][LQ] low
  __nv_bfloat16* Bs = wBL + N * LQ;                                 // [Q][LN]
  float* dts = reinterpret_cast<float*>(Bs + Q * LN);
  float* cs = dts + Q;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int c = blockIdx.x;
  const int64_t h = blockIdx.y, b = blockIdx.z, g = h / (p.H / p.G), t0 = (int64_t)c * Q;
  {
    SsdChunkRegs<P, N> r;
    ssd_fetch<P, N, false>(r, p, b, h, g, t0, tid);  // C is not needed here
    ssd_store<P, N, false>(r, XT, Bs, nullptr, dts, tid);
  }
  __syncthreads();
  ssd_cumsum(dts, cs, p.A[h], warp, lane);
  __syncthreads();
  const float cs_end = cs[Q - 1];
  for (int i = tid; i < Q * N; i += kSsdThreads) {
    const int t = i % Q, n = i / Q;
    const float v = __bfloat162float(Bs[t * LN + n]) * __expf(cs_end - cs[t]) * dts[t];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    wBT[n * LQ + t] = hi;
    wBL[n * LQ + t] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
  __syncthreads();
  constexpr int MT = P / 16, WPM = 8 / MT, NTW = (N / 8) / WPM;
  const int mt = warp % MT, nq = warp / MT;
  float acc[NTW][4] = {};
#pragma unroll
  for (int k0 = 0; k0 < Q; k0 += 16) {
    uint32_t a[4];
    frag_a(a, XT, LQ, mt * 16, k0, lane);
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
      uint32_t bb[2];
      frag_b(bb, wBT, LQ, (nq * NTW + nt) * 8, k0, lane);
      mma_16816(acc[nt], a, bb);
      frag_b(bb, wBL, LQ, (nq * NTW + nt) * 8, k0, lane);
      mma_16816(acc[nt], a, bb);
    }
  }
  float* S = p.ws_S + (((b * p.nc + c) * p.H + h) * P) * N;
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int pr = mt * 16 + gq + 8 * hf, nc0 = (nq * NTW + nt) * 8 + 2 * tq;
      *reinterpret_cast<float2*>(S + pr * N + nc0) = make_float2(acc[nt][2 * hf], acc[nt][2 * hf + 1]);
    }
  }
  if (tid == 0) p.ws_dec[(b * p.H + h) * p.nc + c] = __expf(cs_end);
}

// One thread per (b, h, state element): the carry over chunks.
template <int P, int N>
__global__ void __launch_bounds__(256) ssd_state_pass_kernel(const SsdParams p) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // over batch * H * P * N
  constexpr int64_t PN = (int64_t)P * N;
  if (i >= p.batch * p.H * PN) return;
  const int64_t e = i % PN, bh = i / PN, h = bh % p.H, b = bh / p.H;
  float st = p.h0 ? p.h0[bh * PN + e] : 0.f;
  const float* dec = p.ws_dec + bh * p.nc;
  const int64_t cstride = p.H * PN;  // from one chunk's entry to the next
  const float* S = p.ws_S + ((b * p.nc) * p.H + h) * PN + e;
  __nv_bfloat16* Ho = p.ws_H + ((b * p.nc) * p.H + h) * PN + e;
  // Eight chunks' contributions are loaded before any of them is used (the stores of the
  // entering states would otherwise keep each load behind the previous store).
  for (int c0 = 0; c0 < p.nc; c0 += 8) {
    float sv[8], dv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      sv[k] = c0 + k < p.nc ? __ldg(S + (c0 + k) * cstride) : 0.f;
      dv[k] = c0 + k < p.nc ? __ldg(dec + c0 + k) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (c0 + k < p.nc) {
        Ho[(c0 + k) * cstride] = __float2bfloat16_rn(st);
        st = fmaf(dv[k], st, sv[k]);
      }
    }
  }
  if (p.last_state) p.last_state[bh * PN + e] = st;
}

template <int P, int N, typename TY>
__global__ void __launch_bounds__(kSsdThreads) ssd_chunk_scan_kernel(const SsdParams p) {
  constexpr int Q = kSsdQ, LQ = Q + kSsdPad, LN = N + kSsdPad;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* XT = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [P][LQ]
  __nv_bfloat16* Bs = XT + P * LQ;                                  // [Q][LN]
  __nv_bfloat16* Cs = Bs + Q * LN;                                  // [Q][LN]
  __nv_bfloat16* Ws = Cs + Q * LN;                                  // [Q][LQ] high
  __nv_bfloat16* WsL = Ws + Q * LQ;                                 // [Q][LQ] low
  __nv_bfloat16* Hb = WsL + Q * LQ;                                 // [P][LN] entering state
  float* dts = reinterpret_cast<float*>(Hb + P * LN);
  float* cs = dts + Q;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int c = blockIdx.x;
  const int64_t h = blockIdx.y, b = blockIdx.z, g = h / (p.H / p.G), t0 = (int64_t)c * Q;
  const int tc = (int)((p.L - t0) < Q ? (p.L - t0) : Q);
  const float Dh = p.Dskip ? p.Dskip[h] : 0.f;
  {
    SsdChunkRegs<P, N> r;
    ssd_fetch<P, N>(r, p, b, h, g, t0, tid);
    ssd_store<P, N>(r, XT, Bs, Cs, dts, tid);
    const __nv_bfloat16* Hg = p.ws_H + (((b * p.nc + c) * p.H + h) * P) * N;
    for (int i = tid; i < P * N / 8; i += kSsdThreads) {
      const int pr = (i * 8) / N, n0 = (i * 8) % N;
      *reinterpret_cast<uint4*>(Hb + pr * LN + n0) = *reinterpret_cast<const uint4*>(Hg + pr * N + n0);
    }
  }
  __syncthreads();
  ssd_cumsum(dts, cs, p.A[h], warp, lane);
  __syncthreads();
  {
    const int mt = warp & 3, nh = warp >> 2;
    float acc[4][4] = {};
#pragma unroll
    for (int k0 = 0; k0 < N; k0 += 16) {
      uint32_t a[4];
      frag_a(a, Cs, LN, mt * 16, k0, lane);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        uint32_t bb[2];
        frag_b(bb, Bs, LN, nh * 32 + nt * 8, k0, lane);
        mma_16816(acc[nt], a, bb);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int j = mt * 16 + gq + 8 * hf, i0 = nh * 32 + nt * 8 + 2 * tq;
        const float w0 = j >= i0 ? acc[nt][2 * hf] * __expf(cs[j] - cs[i0]) * dts[i0] : 0.f;
        const float w1 = j >= i0 + 1 ? acc[nt][2 * hf + 1] * __expf(cs[j] - cs[i0 + 1]) * dts[i0 + 1] : 0.f;
        const __nv_bfloat162 hi = __floats2bfloat162_rn(w0, w1);
        *reinterpret_cast<__nv_bfloat162*>(Ws + j * LQ + i0) = hi;
        *reinterpret_cast<uint32_t*>(WsL + j * LQ + i0) = pack_bf16(w0 - __low2float(hi), w1 - __high2float(hi));
      }
    }
  }
  __syncthreads();
  {
    constexpr int NT = P / 16;
    const int mt = warp & 3, nh = warp >> 2;
    float ad[NT][4] = {}, ao[NT][4] = {};
#pragma unroll
    for (int k0 = 0; k0 < Q; k0 += 16) {
      uint32_t a[4], al[4];
      frag_a(a, Ws, LQ, mt * 16, k0, lane);
      frag_a(al, WsL, LQ, mt * 16, k0, lane);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint32_t bb[2];
        frag_b(bb, XT, LQ, nh * (P / 2) + nt * 8, k0, lane);
        mma_16816(ad[nt], a, bb);
        mma_16816(ad[nt], al, bb);
      }
    }
#pragma unroll
    for (int k0 = 0; k0 < N; k0 += 16) {
      uint32_t a[4];
      frag_a(a, Cs, LN, mt * 16, k0, lane);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint32_t bb[2];
        frag_b(bb, Hb, LN, nh * (P / 2) + nt * 8, k0, lane);
        mma_16816(ao[nt], a, bb);
      }
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int j = mt * 16 + gq + 8 * hf;
      if (j < tc) {
        const float e = __expf(cs[j]);
        TY* yrow = static_cast<TY*>(p.y) + ((b * p.L + t0 + j) * p.H + h) * P;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int pc = nh * (P / 2) + nt * 8 + 2 * tq;
          const float v0 = ad[nt][2 * hf] + e * ao[nt][2 * hf] + Dh * __bfloat162float(XT[pc * LQ + j]);
          const float v1 = ad[nt][2 * hf + 1] + e * ao[nt][2 * hf + 1] + Dh * __bfloat162float(XT[(pc + 1) * LQ + j]);
          if (sizeof(TY) == 2)
            *reinterpret_cast<uint32_t*>(yrow + pc) = pack_bf16(v0, v1);
          else
            *reinterpret_cast<float2*>(yrow + pc) = make_float2(v0, v1);
        }
      }
    }
  }
}

}  // namespace ssm
