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
// Two schedules. Without a workspace, ssd_fwd_kernel: one CTA of 8 warps per (batch, head)
// walks the chunks in order with the fp32 state on chip (the four contractions C B^T, W X,
// C S^T, X^T (w B) on mma.sync m16n8k16), prefetching the next chunk's inputs into
// registers while the current one is computed. With a workspace, the chunk-parallel
// schedule further down: step sizes and C B^T per chunk, the state walk, and the read-out
// of every chunk at once, on tcgen05 for P = 128.
#pragma once

#include "common.cuh"
#include "tma.cuh"
#include "umma.cuh"

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
  // chunk-parallel schedule (workspace): per (b, c, h) the state entering the chunk
  // (bf16 P x N; for P = 128 a K-major tensor-core operand image: 8 x 8 core matrices
  // (p / 8, n / 8) of 8 rows p x 16 bytes, (p8, n8) at p8 (N / 8) 128 + n8 128 bytes; for
  // P = 64 mma.sync fragment order: [P/8][N/16][32 lanes][2] pairs, the pair (row 8 j +
  // lane / 4, columns 16 k + 2 (lane % 4) (+ 1)) and the same 8 columns on), its step sizes
  // dt and cumulative decay exponents cs (fp32, Q each); per (b, c, g) C B^T of the chunk
  // (fp32, Q rows of kSsdCBPitch)
  __nv_bfloat16* ws_H;
  float* ws_dt;
  float* ws_cs;
  float* ws_CB;
  int nc;
  // Failure detection (tcgen05 kernels): the limit of every bounded wait in cycles (0: the
  // default of about one second), and a test-only switch that stops the copier issuing
  // copies, so that every wait for data runs out.
  long long wait_cycles;
  int fault_skip_loads;
};

constexpr int kSsdQ = 64;
constexpr int kSsdCBPitch = kSsdQ + 8;  // floats per row of C B^T in the workspace (bank-spread reads)
constexpr int kSsdThreads = 256;
constexpr int kSsdPad = 8;  // bf16 elements of row padding: conflict-free fragment loads

template <int P, int N>
constexpr int ssd_smem_bytes() {
  constexpr int LQ = kSsdQ + kSsdPad, LN = N + kSsdPad;
  return 2 * (P * LQ + 2 * kSsdQ * LN + 2 * N * LQ + 2 * kSsdQ * LQ + P * LN) + 4 * (P * N + 2 * kSsdQ);
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm(
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
// Pass 0 (block per (b, c)): dt_t = softplus(delta + dt_bias) and cs_t = sum_{k<=t} dt_k A
//   for every head of the chunk (dt = 0 past L), and C B^T of the chunk for every group
//   (shared by the group's heads).
// Pass 1 (CTA per (b, h, block of 32 state columns)): the state walk. The block's columns
//   of S stay in tensor-core accumulators (fp32) from chunk to chunk:
//     H_c -> workspace (bf16, the operand of the read-out),  S <- exp(cs_end) S + X^T (w B),
//   w_t = exp(cs_end - cs_t) dt_t; the final S is last_state. Only the states the read-out
//   needs leave the chip; each chunk's inputs arrive by cp.async while the previous chunk
//   is computed.
// Pass 2 (persistent, item = (b, c, h)): Y = W X + diag(exp(cs)) C H_c^T + D X, with W the
//   group's C B^T masked to j >= i and decayed by exp(cs_j - cs_i) dt_i for this head.
//   Two CTAs of 8 warps per SM walk the items (h fastest, so CTAs working at the same time
//   share C B^T and C in L2); each CTA copies an item's inputs by cp.async, then computes
//   it, so one CTA's copies overlap the other's arithmetic.
// Fragments come from shared memory by ldmatrix (transposed where the contraction runs
// over time); w B and W reach the tensor cores as bf16 high + low pairs.

__device__ __forceinline__ uint32_t ssd_saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const __nv_bfloat16* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(ssd_saddr(p))
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const __nv_bfloat16* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(ssd_saddr(p))
               : "memory");
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t (&r)[2], const __nv_bfloat16* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(ssd_saddr(p))
               : "memory");
}
// 16-byte global -> shared copy; zero fill when !valid (src must still be a mapped address)
__device__ __forceinline__ void ssd_cp16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ssd_saddr(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void ssd_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int n>
__device__ __forceinline__ void ssd_cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}
// (lo, hi) bf16 halves of a fragment register as floats (lo = the lower index)
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t r) {
  return make_float2(__uint_as_float(r << 16), __uint_as_float(r & 0xffff0000u));
}
// v -> (high, low) bf16 pairs with high + low = v to ~16 significant bits
__device__ __forceinline__ void split_bf16x2(float2 v, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(v.x, v.y);
  const float2 h = bf16x2_to_f2(hi);
  lo = pack_bf16(v.x - h.x, v.y - h.y);
}

// Q rows of W 16-byte chunks each, row t of a (batch, L, ...) tensor at src + t * pitch,
// zero past rows_valid, into dst with row stride ld (elements).
template <int W>
__device__ __forceinline__ void ssd_stage_rows(__nv_bfloat16* dst, int ld, const __nv_bfloat16* src, int64_t pitch,
                                               int64_t rows_valid, const __nv_bfloat16* any, int tid) {
  for (int i = tid; i < kSsdQ * W; i += kSsdThreads) {
    const int t = i / W, k = i % W;
    const bool v = t < rows_valid;
    ssd_cp16(dst + t * ld + 8 * k, v ? src + t * pitch + 8 * k : any, v);
  }
}
// dt and cs of item it (Q floats each) into a stage.
__device__ __forceinline__ void ssd_stage_floats(unsigned char* st, const SsdParams& p, int64_t it, int off_dt,
                                                 int off_cs, int tid) {
  if (tid < 2 * (kSsdQ / 4)) {
    const int k = tid % (kSsdQ / 4);
    const float* src = (tid < kSsdQ / 4 ? p.ws_dt : p.ws_cs) + it * kSsdQ + 4 * k;
    ssd_cp16(st + (tid < kSsdQ / 4 ? off_dt : off_cs) + 16 * k, src, true);
  }
}

constexpr int kSsdNB = 32;  // state columns per CTA of the state walk

template <int P>
struct SsdWalkStage {
  static constexpr int LP = P + kSsdPad, LB = kSsdNB + kSsdPad;
  static constexpr int kX = 0, kB = kX + kSsdQ * LP * 2, kDt = kB + kSsdQ * LB * 2, kCs = kDt + kSsdQ * 4;
  static constexpr int kBytes = kCs + kSsdQ * 4, kStages = 2;
  static constexpr int kWB = kStages * kBytes;  // (w B) high and low, two buffers: [2][2][Q][LB] bf16
  static_assert(kBytes % 16 == 0, "stage layout");
};
template <int P>
constexpr int ssd_walk_smem_bytes() {
  return SsdWalkStage<P>::kWB + 4 * kSsdQ * SsdWalkStage<P>::LB * 2;
}

// Pass 0. grid (nc, batch), block 256. (a) warp w takes heads w, w + 8, ...; lane l steps
// 2l, 2l + 1. (b) per group g: CB = C B^T of the chunk (fp32, Q x Q, zero rows and columns
// past L); warp w computes rows 16 (w & 3) .. + 15, columns 32 (w >> 2) .. + 31.
template <int N>
__global__ void __launch_bounds__(256) ssd_prep_kernel(const SsdParams p) {
  constexpr int Q = kSsdQ, LN = N + kSsdPad;
  __shared__ __align__(16) __nv_bfloat16 Cs[Q * LN], Bs[Q * LN];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3, c = blockIdx.x;
  const int64_t b = blockIdx.y, t0 = (int64_t)c * Q, t = t0 + 2 * lane;
  for (int64_t h = warp; h < p.H; h += 8) {
    const float bias = p.dt_bias ? p.dt_bias[h] : 0.f, Ah = p.A[h];
    float d[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      d[k] = 0.f;
      if (t + k < p.L) {
        const float r = __bfloat162float(p.delta[(b * p.L + t + k) * p.H + h]) + bias;
        d[k] = p.dt_softplus ? softplus_precise(r) : r;
      }
    }
    const float v0 = d[0] * Ah, v1 = d[1] * Ah;
    float s = v0 + v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float up = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += up;
    }
    const float ex = s - (v0 + v1);
    const int64_t o = ((b * p.nc + c) * p.H + h) * Q + 2 * lane;
    *reinterpret_cast<float2*>(p.ws_dt + o) = make_float2(d[0], d[1]);
    *reinterpret_cast<float2*>(p.ws_cs + o) = make_float2(ex + v0, ex + v0 + v1);
  }
  const int64_t rv = p.L - t0;
  const int mt = warp & 3, n0 = (warp >> 2) * 32;
  for (int64_t g = 0; g < p.G; ++g) {
    __syncthreads();  // the previous group's tiles are no longer read
    for (int i = tid; i < Q * (N / 8); i += 256) {
      const int r = i / (N / 8), k = i % (N / 8);
      const int64_t o = ((b * p.L + t0 + r) * p.G + g) * N + 8 * k;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(Cs + r * LN + 8 * k) = r < rv ? *reinterpret_cast<const uint4*>(p.C + o) : z;
      *reinterpret_cast<uint4*>(Bs + r * LN + 8 * k) = r < rv ? *reinterpret_cast<const uint4*>(p.B + o) : z;
    }
    __syncthreads();
    float acc[4][4] = {};
#pragma unroll
    for (int ks = 0; ks < N / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, Cs + (mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LN + ks * 16 + (lane >> 4) * 8);
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t bb[4];
        ldsm_x4(bb, Bs + (n0 + np * 16 + (lane & 7) + (lane >> 4) * 8) * LN + ks * 16 + ((lane >> 3) & 1) * 8);
        const uint32_t b0[2] = {bb[0], bb[1]}, b1[2] = {bb[2], bb[3]};
        mma_16816(acc[2 * np], a, b0);
        mma_16816(acc[2 * np + 1], a, b1);
      }
    }
    float* CB = p.ws_CB + ((b * p.nc + c) * p.G + g) * Q * kSsdCBPitch;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        *reinterpret_cast<float2*>(CB + (mt * 16 + gq + 8 * hf) * kSsdCBPitch + n0 + nt * 8 + 2 * tq) =
            make_float2(acc[nt][2 * hf], acc[nt][2 * hf + 1]);
  }
}

// Pass 1. grid (N / 32, H, batch), block 256: the CTA holds state columns 32 bx .. + 31 and
// all P rows; warp w holds rows 16 (w % MT) .. + 15 (MT = P / 16 row tiles) and NTW column
// tiles of 8 starting at 8 NTW (w / MT). Per chunk, w B of the CTA's columns is formed once
// in shared memory (bf16 high + low); X^T comes straight from the staged X by ldmatrix.
template <int P, int N>
__global__ void __launch_bounds__(kSsdThreads, 3) ssd_state_walk_kernel(const SsdParams p) {
  using St = SsdWalkStage<P>;
  constexpr int Q = kSsdQ, S = St::kStages, LP = St::LP, LB = St::LB, NB = kSsdNB;
  constexpr int MT = P / 16, WPM = 8 / MT, NTW = (NB / 8) / WPM;
  static_assert(MT * WPM == 8 && NTW % 2 == 0, "warp tiling");
  static_assert(S >= 2, "the ring waits for all but the newest S - 2 groups");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* wBbuf = reinterpret_cast<__nv_bfloat16*>(smem_raw + St::kWB);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int nb0 = blockIdx.x * NB;
  const int64_t h = blockIdx.y, b = blockIdx.z, g = h / (p.H / p.G);
  const int row0 = (warp % MT) * 16, col0 = (warp / MT) * NTW * 8;  // within the CTA's block
  const int nc = p.nc;
  auto load = [&](int s, int c) {
    unsigned char* st = smem_raw + s * St::kBytes;
    const int64_t t0 = (int64_t)c * Q, rv = p.L - t0;
    ssd_stage_rows<P / 8>(reinterpret_cast<__nv_bfloat16*>(st + St::kX), LP, p.x + ((b * p.L + t0) * p.H + h) * P,
                          p.H * P, rv, p.x, tid);
    ssd_stage_rows<NB / 8>(reinterpret_cast<__nv_bfloat16*>(st + St::kB), LB,
                           p.B + ((b * p.L + t0) * p.G + g) * N + nb0, p.G * N, rv, p.B, tid);
    ssd_stage_floats(st, p, (b * nc + c) * p.H + h, St::kDt, St::kCs, tid);
  };
  // acc[nt]: rows row0 + gq (+ 8), columns nb0 + col0 + 8 nt + 2 tq (+ 1)
  const int64_t sbase = ((b * p.H + h) * P + row0 + gq) * N + nb0 + col0 + 2 * tq;
  float acc[NTW][4];
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const float2 v = p.h0 ? *reinterpret_cast<const float2*>(p.h0 + sbase + 8 * hf * N + 8 * nt)
                            : make_float2(0.f, 0.f);
      acc[nt][2 * hf] = v.x;
      acc[nt][2 * hf + 1] = v.y;
    }
#pragma unroll
  for (int k = 0; k < S - 1; ++k) {
    if (k < nc) load(k, k);
    ssd_cp_commit();
  }
  for (int c = 0; c < nc; ++c) {
    ssd_cp_wait<S - 2>();  // chunk c has landed (this thread's copies)
    __syncthreads();       // ... everyone's; and every warp is done with chunk c - 1
    if (c + S - 1 < nc) load((c + S - 1) % S, c + S - 1);
    ssd_cp_commit();
    const unsigned char* st = smem_raw + (c % S) * St::kBytes;
    const __nv_bfloat16* Xs = reinterpret_cast<const __nv_bfloat16*>(st + St::kX);  // [t][p]
    const __nv_bfloat16* Bs = reinterpret_cast<const __nv_bfloat16*>(st + St::kB);  // [t][n of the block]
    const float* dts = reinterpret_cast<const float*>(st + St::kDt);
    const float* css = reinterpret_cast<const float*>(st + St::kCs);
    __nv_bfloat16* wbh = wBbuf + (c & 1) * 2 * Q * LB;  // [t][n] high
    __nv_bfloat16* wbl = wbh + Q * LB;                   // [t][n] low
    const float cs_end = css[Q - 1];
    static_assert(NB == 32, "w B rows: half a warp per row");
    for (int e = tid; e < Q * NB / 2; e += kSsdThreads) {
      // a warp covers rows t and t + 4 (80-byte pitch: disjoint banks)
      const int q = e >> 5, l = e & 31, t = (q >> 2) * 8 + (q & 3) + (l >> 4) * 4, n = 2 * (l & 15);
      const float w = __expf(cs_end - css[t]) * dts[t];
      const float2 v = bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(Bs + t * LB + n));
      uint32_t hi, lo;
      split_bf16x2(make_float2(v.x * w, v.y * w), hi, lo);
      *reinterpret_cast<uint32_t*>(wbh + t * LB + n) = hi;
      *reinterpret_cast<uint32_t*>(wbl + t * LB + n) = lo;
    }
    // the state entering chunk c, for the read-out, in fragment order (256 contiguous bytes
    // per warp store)
    uint2* Ho = reinterpret_cast<uint2*>(p.ws_H + ((b * nc + c) * p.H + h) * (int64_t)P * N) + lane;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int kp = 0; kp < NTW / 2; ++kp)
        Ho[((row0 / 8 + hf) * (N / 16) + (nb0 + col0) / 16 + kp) * 32] =
            make_uint2(pack_bf16(acc[2 * kp][2 * hf], acc[2 * kp][2 * hf + 1]),
                       pack_bf16(acc[2 * kp + 1][2 * hf], acc[2 * kp + 1][2 * hf + 1]));
    const float dec = __expf(cs_end);
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] *= dec;
    __syncthreads();  // w B is complete
#pragma unroll
    for (int ks = 0; ks < Q / 16; ++ks) {
      const int k0 = ks * 16;
      uint32_t a[4];  // (X^T)[p][t] fragment, from X stored [t][p]
      ldsm_x4_t(a, Xs + (k0 + (lane & 7) + (lane >> 4) * 8) * LP + row0 + ((lane >> 3) & 1) * 8);
      uint32_t bh[NTW / 2][4], bl[NTW / 2][4];
#pragma unroll
      for (int np = 0; np < NTW / 2; ++np) {
        const int o = (k0 + (lane & 7) + ((lane >> 3) & 1) * 8) * LB + col0 + np * 16 + (lane >> 4) * 8;
        ldsm_x4_t(bh[np], wbh + o);
        ldsm_x4_t(bl[np], wbl + o);
      }
#pragma unroll
      for (int np = 0; np < NTW / 2; ++np) {
        const uint32_t b0[2] = {bh[np][0], bh[np][1]}, b1[2] = {bh[np][2], bh[np][3]};
        mma_16816(acc[2 * np], a, b0);
        mma_16816(acc[2 * np + 1], a, b1);
      }
#pragma unroll
      for (int np = 0; np < NTW / 2; ++np) {
        const uint32_t b0[2] = {bl[np][0], bl[np][1]}, b1[2] = {bl[np][2], bl[np][3]};
        mma_16816(acc[2 * np], a, b0);
        mma_16816(acc[2 * np + 1], a, b1);
      }
    }
  }
  if (p.last_state) {
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        *reinterpret_cast<float2*>(p.last_state + sbase + 8 * hf * N + 8 * nt) =
            make_float2(acc[nt][2 * hf], acc[nt][2 * hf + 1]);
  }
  ssd_cp_wait<0>();
}

// Pass 1 on the 5th-generation tensor cores (P = 128). grid (N / 32, H,
// batch), block 192: warps 0-3 are workers, warp 4's lane 0 issues the MMAs, warp 5's
// lane 0 issues the copies. Per chunk c:
//   copier: chunk c by TMA into stage c % 2 once the MMA of chunk c - 2 has released it
//     (X as two 64 x 64 boxes with the 128-byte swizzle, B as one 32 x 64 box, dt and cs
//     as bulk copies, all on one mbarrier);
//   workers: form w B of chunk c (bf16 high + low) in stage c % 2 and signal full; then,
//     for chunk c - 1, load its MMA result from TMEM (one
//     state row per thread: warp w has TMEM lanes 32 w .. 32 w + 31), write the entering
//     state (bf16, the read-out's K-major image), update the fp32 state registers
//     S <- exp(cs_end) S + S_c and release the TMEM buffer;
//   MMA thread: X^T [w B high | w B low] as 4 tcgen05.mma (M = 128 state rows, N = 64:
//     the 32 state columns of the high part beside those of the low part, K = 16 steps)
//     into TMEM buffer c % 2 (the workers add the two halves: S_c = X^T w B), then commit
//     to the buffer's full barrier and to the stage's empty barrier. Side by side, one MMA
//     reads each X tile once, halving the tensor core's time per chunk (three CTAs per SM
//     share it).
// So the MMA of chunk c runs while the workers finish chunk c - 1 and start chunk c + 1.
// X is an MN-major operand with the 128-byte swizzle (a 128-byte row = 64 state rows of
// one step; 8 steps per 1 KB atom; the descriptor's LBO is the distance between atoms along
// M and its SBO the distance between atoms along K; measured on B300 against a host
// product), so TMA moves 128-byte rows. w B is an MN-major operand without swizzle (16-byte
// rows of 8 bf16 along the state columns, 8 steps per core matrix; core matrices (n8, t8)
// at n8 * 128 + t8 * 1024, n8 0-3 the high part and 4-7 the low part). Steps past L in a
// batch row's last chunk are zeroed (X) or masked (w B) after the copy, so the next row's
// data never enters. Every wait is bounded; one that runs out raises a CTA-wide abort flag
// that ends every role's loop.
constexpr int kTcP = 128;
constexpr int kTcWorkers = 128;
constexpr int kTcThreads = kTcWorkers + 64;
template <int N>
struct SsdTcWalk {
  static constexpr int kX = 0;                            // X: [p half][t][64 p] swizzled, 16 KB
  static constexpr int kB = kX + kSsdQ * kTcP * 2;        // raw B, [t][32 columns], 4 KB
  static constexpr int kW = kB + kSsdQ * kSsdNB * 2;      // [w B high | w B low]: 8 x 8 core matrices (n8, t8), 8 KB
  static constexpr int kDt = kW + 2 * kSsdQ * kSsdNB * 2; // dt [Q]
  static constexpr int kCs = kDt + kSsdQ * 4;             // cs [Q]
  static constexpr int kStage = (kCs + kSsdQ * 4 + 1023) / 1024 * 1024;  // swizzle atoms 1 KB aligned
  static constexpr int kBar = 2 * kStage;                 // full, empty, tfull, tempty, loaded [2] each
  static constexpr int kSlot = kBar + 10 * 8;             // TMEM address
  static constexpr int kAbort = kSlot + 4;
  static constexpr int kBytes = kAbort + 12 + 1024;       // + room to align the base to 1 KB
  // operand strides (bytes): X atoms (64 p x 8 t, 1 KB) at p-half * 8192 + t8 * 1024; w B core
  // matrix (n8, t8) at n8 * 128 + t8 * 1024
  static constexpr uint32_t kXlbo = 8192, kXsbo = 1024, kWlbo = 1024, kWsbo = 128;
};

// Bounded wait on a barrier phase that also gives up once another role has aborted.
// Suspended between checks (up to 2 us a try), so that waiting warps leave the issue
// slots to the warps with work. The limit is read from the parameters only once the first
// try has failed, so no role keeps it in registers (the state walk needs three CTAs per SM).
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort, const SsdParams& p,
                                        int err = kErrWaitMma) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long limit = p.wait_cycles > 0 ? p.wait_cycles : kWaitCycles;
  const long long start = clock64();
  while (!mbar_try_wait_suspend(bar, parity, 2000u)) {
    if (*abort) return false;
    if (clock64() - start > limit) {
      atomicCAS(&g_ssm_error, 0, err);
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Barrier over n threads (id bar_id) that also returns the AND of every thread's v.
__device__ __forceinline__ bool bar_and(bool v, int bar_id, int n) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\nbar.red.and.pred p, %2, %3, q;\nselp.u32 %0, 1, 0, p;\n}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(bar_id), "r"(n)
      : "memory");
  return r != 0;
}

template <int N>
__global__ void __launch_bounds__(kTcThreads, 3)
    ssd_state_walk_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                             const SsdParams p) {
  using L = SsdTcWalk<N>;
  constexpr int Q = kSsdQ, P = kTcP, NB = kSsdNB;
  constexpr uint32_t kIdesc = umma_idesc_bf16(P, 2 * NB, true, true);  // N: high and low columns
  extern __shared__ __align__(16) unsigned char smem_dyn[];
  unsigned char* smem_raw = smem_dyn + ((1024u - (umma_saddr(smem_dyn) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + L::kBar);
  uint64_t* empty = full + 2;
  uint64_t* tfull = full + 4;
  uint64_t* tempty = full + 6;
  uint64_t* loaded = full + 8;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem_raw + L::kSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem_raw + L::kAbort);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb0 = blockIdx.x * NB;
  const int64_t h = blockIdx.y, b = blockIdx.z, g = h / (p.H / p.G);
  const int nc = p.nc;
  const int64_t item0 = (b * nc) * p.H + h;  // item of chunk c: item0 + c * H

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], kTcWorkers);
      mbar_init(&empty[i], 1);
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kTcWorkers);
      mbar_init(&loaded[i], 1);
    }
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_b);
    *abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(slot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  // chunk c into stage s by TMA (X 16 KB, B 4 KB, dt and cs 256 B each)
  auto load = [&](int s, int c) {
    unsigned char* st = smem_raw + s * L::kStage;
    const int32_t row = (int32_t)(b * p.L + (int64_t)c * Q);
    mbar_arrive_expect_tx(&loaded[s], (uint32_t)(Q * P * 2 + Q * NB * 2 + 2 * Q * 4));
    tma_load_3d_bar(st + L::kX, &tm_x, 0, (int32_t)h, row, &loaded[s]);
    tma_load_3d_bar(st + L::kX + L::kXlbo, &tm_x, 64, (int32_t)h, row, &loaded[s]);
    tma_load_2d(st + L::kB, &tm_b, (int32_t)(g * N + nb0), row, &loaded[s]);
    const int64_t it = item0 + (int64_t)c * p.H;
    bulk_load(st + L::kDt, p.ws_dt + it * Q, Q * 4, &loaded[s]);
    bulk_load(st + L::kCs, p.ws_cs + it * Q, Q * 4, &loaded[s]);
  };

  if (warp == 5) {  // ---------------- copier ----------------
    if (lane == 0 && !p.fault_skip_loads) {
      for (int c = 0; c < nc; ++c) {
        // stage c % 2 last held chunk c - 2: wait until its MMA has read it
        if (c >= 2 && !tc_wait(&empty[c & 1], (uint32_t)(((c - 2) >> 1) & 1), abort, p)) break;
        load(c & 1, c);
      }
    }
  } else if (warp == 4) {  // ---------------- MMA issuer ----------------
    if (lane == 0) {
      for (int c = 0; c < nc; ++c) {
        const int s = c & 1;
        if (!tc_wait(&full[s], (uint32_t)((c >> 1) & 1), abort, p)) break;
        if (c >= 2 && !tc_wait(&tempty[s], (uint32_t)(((c - 2) >> 1) & 1), abort, p)) break;
        tc_fence_after();
        const unsigned char* st = smem_raw + s * L::kStage;
        const uint32_t xa = umma_saddr(st + L::kX), wa = umma_saddr(st + L::kW);
        const uint32_t d = tmem + 64u * (uint32_t)s;
#pragma unroll
        for (int ks = 0; ks < Q / 16; ++ks) {
          const uint64_t ad = umma_sdesc(xa + ks * 2 * L::kXsbo, L::kXlbo, L::kXsbo, 2);
          umma_bf16(d, ad, umma_sdesc(wa + ks * 2 * L::kWlbo, L::kWlbo, L::kWsbo), kIdesc, ks > 0);
        }
        umma_commit(&tfull[s]);
        umma_commit(&empty[s]);
      }
    }
  } else {  // ---------------- workers ----------------
    const int prow = tid;  // this thread's state row (TMEM lane)
    float S[NB];
    {
      const int64_t o = ((b * p.H + h) * P + prow) * N + nb0;
#pragma unroll
      for (int j = 0; j < NB; j += 4) {
        const float4 v = p.h0 ? *reinterpret_cast<const float4*>(p.h0 + o + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        S[j] = v.x;
        S[j + 1] = v.y;
        S[j + 2] = v.z;
        S[j + 3] = v.w;
      }
    }
    // chunk c's result -> entering state out, state update (dec = exp(cs_end) of chunk c);
    // releases its TMEM buffer
    auto epilogue = [&](int c, float dec) {
      const int s = c & 1;
      if (!tc_wait(&tfull[s], (uint32_t)((c >> 1) & 1), abort, p)) return false;
      tc_fence_after();
      float Sc[NB];
      {  // the high part's 32 columns, then the low part's
        const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16) + 64u * (uint32_t)s;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t hv[16], lv[16];
          tmem_ld16_nowait(ta + 16u * hf, hv);
          tmem_ld16_nowait(ta + 32u + 16u * hf, lv);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) Sc[16 * hf + j] = __uint_as_float(hv[j]) + __uint_as_float(lv[j]);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[s]);
      // K-major operand image for the read-out: this row's 32 columns are 4 core-matrix
      // rows of 16 bytes, (p8, n8) at p8 (N / 8) 128 + n8 128 + (p % 8) 16 bytes
      unsigned char* Ho = reinterpret_cast<unsigned char*>(p.ws_H + (item0 + (int64_t)c * p.H) * P * N) +
                          (prow >> 3) * (N / 8) * 128 + (nb0 >> 3) * 128 + (prow & 7) * 16;
#pragma unroll
      for (int q = 0; q < NB / 8; ++q) {
        const float* v = S + 8 * q;
        *reinterpret_cast<uint4*>(Ho + q * 128) =
            make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) S[j] = fmaf(dec, S[j], Sc[j]);
      return true;
    };

    bool ok = true;        // this thread's waits so far
    float dec_prev = 0.f;  // exp(cs_end) of chunk c - 1
    for (int c = 0; c < nc; ++c) {
      const int s = c & 1;
      if (ok && !tc_wait(&loaded[s], (uint32_t)((c >> 1) & 1), abort, p, kErrWaitFull)) ok = false;
      const int rv = (int)((p.L - (int64_t)c * Q) < Q ? (p.L - (int64_t)c * Q) : Q);
      if (ok && rv < Q) {  // steps past L: zero rows of X (another batch row's data or fill)
        unsigned char* st = smem_raw + s * L::kStage;
        for (int i = tid; i < (Q - rv) * (P / 8); i += kTcWorkers) {  // a step's row: 8 chunks per half
          const int t = rv + i / (P / 8), k = i % (P / 8);
          *reinterpret_cast<uint4*>(st + L::kX + (k >> 3) * L::kXlbo + t * 128 + (k & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // every worker's view of the stage; the workers leave the loop together if any wait
      // ran out
      if (!bar_and(ok, 1, kTcWorkers)) {
        ok = false;
        break;
      }
      float dec_cur;
      {  // w B of chunk c (bf16 high + low), thread -> (t, 8 columns) x 2
        unsigned char* st = smem_raw + s * L::kStage;
        const float* dts = reinterpret_cast<const float*>(st + L::kDt);
        const float* css = reinterpret_cast<const float*>(st + L::kCs);
        const float cs_end = css[Q - 1];
        dec_cur = __expf(cs_end);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int i = tid + r * kTcWorkers;
          const int t = (i >> 5) * 8 + (i & 7), n8 = (i >> 3) & 3;
          const float w = __expf(cs_end - css[t]) * dts[t];
          const uint4 raw = *reinterpret_cast<const uint4*>(st + L::kB + t * (NB * 2) + n8 * 16);
          const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 v = bf16x2_to_f2(rw[k]);
            split_bf16x2(t < rv ? make_float2(v.x * w, v.y * w) : make_float2(0.f, 0.f), hi[k], lo[k]);
          }
          const int off = n8 * L::kWsbo + (t >> 3) * L::kWlbo + (t & 7) * 16;
          *reinterpret_cast<uint4*>(st + L::kW + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(st + L::kW + off + 4 * L::kWsbo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      fence_smem_to_async();
      mbar_arrive(&full[s]);
      if (c >= 1 && !epilogue(c - 1, dec_prev)) ok = false;
      dec_prev = dec_cur;
    }
    if (ok && nc >= 1) ok = epilogue(nc - 1, dec_prev);
    if (p.last_state && ok) {
      const int64_t o = ((b * p.H + h) * P + prow) * N + nb0;
#pragma unroll
      for (int j = 0; j < NB; j += 4)
        *reinterpret_cast<float4*>(p.last_state + o + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Item (b, c, h) of the persistent read-out pass.
struct SsdItem {
  int64_t b, c, h, g, t0;
};

// The items first, first + step, first + 2 step, ... of a persistent CTA, decoded as
// (b, c, h) counters that advance with carries: a few integer operations per item where
// dividing each item index costs several 64-bit divisions per thread (items < 2^31, checked
// on the host).
struct SsdItemWalk {
  uint32_t H, nc, hpg, h, c, b, sh, sq;
  __device__ __forceinline__ void init(const SsdParams& p, uint32_t first, uint32_t step) {
    H = (uint32_t)p.H;
    nc = (uint32_t)p.nc;
    hpg = (uint32_t)(p.H / p.G);
    const uint32_t q = first / H;
    h = first - q * H;
    c = q % nc;
    b = q / nc;
    sq = step / H;
    sh = step - sq * H;
  }
  __device__ __forceinline__ void advance() {
    h += sh;
    uint32_t cq = sq;
    if (h >= H) {
      h -= H;
      ++cq;
    }
    c += cq;
    if (c >= nc) {
      const uint32_t w = c / nc;
      b += w;
      c -= w * nc;
    }
  }
  __device__ __forceinline__ SsdItem item() const {
    SsdItem r;
    r.h = h;
    r.c = c;
    r.b = b;
    r.g = hpg == H ? 0 : h / hpg;
    r.t0 = (int64_t)c * kSsdQ;
    return r;
  }
};

// Pass 2. Per item the inputs arrive by TMA and bulk copies on one mbarrier (one thread
// issues them): X and C as 64 x 64 boxes with the 128-byte swizzle (rows of 128 bytes; the
// 16-byte chunk c of row r at chunk c ^ (r % 8), so that ldmatrix reads them without bank
// conflicts), the entering state, C B^T, dt and cs as contiguous copies. W is built once
// per item in shared memory; the causal work of a row block grows with its index, so warp
// (mp, pq) takes row blocks mp and 3 - mp (rows 16 m .. 16 m + 15) and columns pq P/4 ..
// + P/4 - 1: every warp does the same number of tensor-core operations. Two CTAs per SM:
// one CTA's copies overlap the other's arithmetic.
template <int P, int N>
struct SsdScanSmem {
  static constexpr int LQ = kSsdQ + kSsdPad;
  static constexpr int kX = 0;                         // X: P / 64 halves of [Q][128 B], swizzled
  static constexpr int kC = kX + kSsdQ * P * 2;         // C: N / 64 halves, swizzled
  static constexpr int kH = kC + kSsdQ * N * 2;         // entering state, fragment order
  static constexpr int kCB = kH + P * N * 2;            // C B^T, [Q][Q] fp32
  static constexpr int kDt = kCB + kSsdQ * kSsdCBPitch * 4;
  static constexpr int kCs = kDt + kSsdQ * 4;
  static constexpr int kW = kCs + kSsdQ * 4;            // W high, W low: [Q][LQ] bf16 each
  static constexpr int kBar = kW + 2 * kSsdQ * LQ * 2;
  static constexpr int kBytes = kBar + 16 + 1024;       // + room to align the base to 1 KB
  static constexpr uint32_t kTx = kSsdQ * P * 2 + kSsdQ * N * 2 + P * N * 2 + kSsdQ * kSsdCBPitch * 4 + 2 * kSsdQ * 4;
  static_assert(kC % 1024 == 0 && kH % 1024 == 0, "swizzled boxes start 1 KB aligned");
};
template <int P, int N>
constexpr int ssd_scan_smem_bytes() {
  return SsdScanSmem<P, N>::kBytes;
}
// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled [rows][128 B] tile
__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

template <int P, int N, typename TY>
__global__ void __launch_bounds__(kSsdThreads, 2)
    ssd_chunk_scan_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_c,
                          const SsdParams p) {
  using Sm = SsdScanSmem<P, N>;
  constexpr int LQ = Sm::LQ, NQ = P / 32, Q = kSsdQ;
  static_assert(NQ % 2 == 0, "two column tiles per ldmatrix");
  extern __shared__ __align__(16) unsigned char smem_dyn[];
  unsigned char* sm = smem_dyn + ((1024u - (umma_saddr(smem_dyn) & 1023u)) & 1023u);
  __nv_bfloat16* Wh = reinterpret_cast<__nv_bfloat16*>(sm + Sm::kW);  // [j][i] high
  __nv_bfloat16* Wl = Wh + Q * LQ;                                    // [j][i] low
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Sm::kBar);
  const unsigned char* Xs = sm + Sm::kX;
  const unsigned char* Cs = sm + Sm::kC;
  const uint2* Hs = reinterpret_cast<const uint2*>(sm + Sm::kH);  // fragment order
  const float* CBs = reinterpret_cast<const float*>(sm + Sm::kCB);
  const float* dts = reinterpret_cast<const float*>(sm + Sm::kDt);
  const float* css = reinterpret_cast<const float*>(sm + Sm::kCs);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int64_t items = p.batch * p.nc * p.H;
  if (tid == 0) {
    mbar_init(bar, 1);
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_c);
    mbar_fence_init();
  }
  __syncthreads();
  const int mp = warp & 1, pc0 = (warp >> 1) * (P / 4);
  const int mrow[2] = {mp, 3 - mp};
  bool ok = true;
  SsdItemWalk wk;
  wk.init(p, blockIdx.x, gridDim.x);
  for (int k = 0;; ++k, wk.advance()) {
    const int64_t it = blockIdx.x + (int64_t)k * gridDim.x;
    if (it >= items) break;
    const SsdItem m = wk.item();
    if (tid == 0) {
      const int32_t row = (int32_t)(m.b * p.L + m.t0);
      mbar_arrive_expect_tx(bar, Sm::kTx);
#pragma unroll
      for (int hx = 0; hx < P / 64; ++hx) tma_load_3d_bar(sm + Sm::kX + hx * 8192, &tm_x, 64 * hx, (int32_t)m.h, row, bar);
#pragma unroll
      for (int hc = 0; hc < N / 64; ++hc)
        tma_load_2d(sm + Sm::kC + hc * 8192, &tm_c, (int32_t)(m.g * N + 64 * hc), row, bar);
      bulk_load(sm + Sm::kH, p.ws_H + it * (int64_t)P * N, P * N * 2, bar);
      bulk_load(sm + Sm::kCB, p.ws_CB + ((m.b * p.nc + m.c) * p.G + m.g) * Q * kSsdCBPitch, Q * kSsdCBPitch * 4, bar);
      bulk_load(sm + Sm::kDt, p.ws_dt + it * Q, Q * 4, bar);
      bulk_load(sm + Sm::kCs, p.ws_cs + it * Q, Q * 4, bar);
    }
    const float Dh = p.Dskip ? p.Dskip[m.h] : 0.f;
    if (ok && !mbar_wait(bar, (uint32_t)(k & 1), kErrWaitFull)) ok = false;
    const int rv = (int)((p.L - m.t0) < Q ? (p.L - m.t0) : Q);
    if (ok && rv < Q) {  // steps past L: zero rows of X (another batch row's data or fill)
      for (int i = tid; i < (Q - rv) * (P / 8); i += kSsdThreads) {
        const int t = rv + i / (P / 8), c = i % (P / 8);
        *reinterpret_cast<uint4*>(sm + Sm::kX + (c >> 3) * 8192 + t * 128 + (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (!__syncthreads_and(ok)) break;  // a copy that never landed stops every thread

    // W_ji = (C B^T)_ji exp(cs_j - cs_i) dt_i for j >= i (else 0), as bf16 high + low
    for (int e = tid; e < Q * Q / 2; e += kSsdThreads) {
      const int j = e / (Q / 2), i = 2 * (e % (Q / 2));
      const float2 cb = *reinterpret_cast<const float2*>(CBs + j * kSsdCBPitch + i);
      const float cj = css[j];
      const float2 v = make_float2(j >= i ? cb.x * __expf(cj - css[i]) * dts[i] : 0.f,
                                   j >= i + 1 ? cb.y * __expf(cj - css[i + 1]) * dts[i + 1] : 0.f);
      uint32_t hi, lo;
      split_bf16x2(v, hi, lo);
      *reinterpret_cast<uint32_t*>(Wh + j * LQ + i) = hi;
      *reinterpret_cast<uint32_t*>(Wl + j * LQ + i) = lo;
    }

    float acc[2][NQ][4] = {};
    // C H^T
#pragma unroll
    for (int ks = 0; ks < N / 16; ++ks) {
      uint32_t a[2][4];
      const int kc = 2 * ks + (lane >> 4);  // 16-byte chunk along n
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = mrow[r] * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm_x4(a[r], reinterpret_cast<const __nv_bfloat16*>(Cs + (kc >> 3) * 8192 + sw128(row, kc & 7)));
      }
#pragma unroll
      for (int nt = 0; nt < NQ; ++nt) {
        const uint2 hv = Hs[((pc0 / 8 + nt) * (N / 16) + ks) * 32 + lane];  // H^T fragment of column tile
        const uint32_t bb[2] = {hv.x, hv.y};
#pragma unroll
        for (int r = 0; r < 2; ++r) mma_16816(acc[r][nt], a[r], bb);
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float e0 = __expf(css[mrow[r] * 16 + gq]), e1 = __expf(css[mrow[r] * 16 + gq + 8]);
#pragma unroll
      for (int nt = 0; nt < NQ; ++nt) {
        acc[r][nt][0] *= e0;
        acc[r][nt][1] *= e0;
        acc[r][nt][2] *= e1;
        acc[r][nt][3] *= e1;
      }
    }
    __syncthreads();  // W is complete
    // W X over the row blocks' causal column blocks
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      if (ks > mrow[1] && ks > mrow[0]) continue;
      uint32_t xb[NQ / 2][4];  // X[t][p] fragments of column tiles (pc0 + 16 np) and (+ 8)
      const int t = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int np = 0; np < NQ / 2; ++np) {
        const int pc = (pc0 + np * 16) / 8 + (lane >> 4);  // 16-byte chunk along p
        ldsm_x4_t(xb[np], reinterpret_cast<const __nv_bfloat16*>(Xs + (pc >> 3) * 8192 + sw128(t, pc & 7)));
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (ks > mrow[r]) continue;
        uint32_t wh[4], wl[4];
        const int wo = (mrow[r] * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LQ + ks * 16 + (lane >> 4) * 8;
        ldsm_x4(wh, Wh + wo);
        ldsm_x4(wl, Wl + wo);
#pragma unroll
        for (int np = 0; np < NQ / 2; ++np) {
          const uint32_t b0[2] = {xb[np][0], xb[np][1]}, b1[2] = {xb[np][2], xb[np][3]};
          mma_16816(acc[r][2 * np], wh, b0);
          mma_16816(acc[r][2 * np + 1], wh, b1);
        }
#pragma unroll
        for (int np = 0; np < NQ / 2; ++np) {
          const uint32_t b0[2] = {xb[np][0], xb[np][1]}, b1[2] = {xb[np][2], xb[np][3]};
          mma_16816(acc[r][2 * np], wl, b0);
          mma_16816(acc[r][2 * np + 1], wl, b1);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int j = mrow[r] * 16 + gq + 8 * hf;
        if (j < rv) {
          TY* yrow = static_cast<TY*>(p.y) + ((m.b * p.L + m.t0 + j) * p.H + m.h) * P;
#pragma unroll
          for (int nt = 0; nt < NQ; ++nt) {
            const int pc = pc0 + nt * 8 + 2 * tq;
            const float2 xv = bf16x2_to_f2(
                *reinterpret_cast<const uint32_t*>(Xs + (pc >> 6) * 8192 + sw128(j, (pc >> 3) & 7) + (pc & 7) * 2));
            const float v0 = fmaf(Dh, xv.x, acc[r][nt][2 * hf]), v1 = fmaf(Dh, xv.y, acc[r][nt][2 * hf + 1]);
            if (sizeof(TY) == 2)
              *reinterpret_cast<uint32_t*>(yrow + pc) = pack_bf16(v0, v1);
            else
              *reinterpret_cast<float2*>(yrow + pc) = make_float2(v0, v1);
          }
        }
      }
    fence_smem_to_async();  // this thread's stores into the stage come before the next copies
    __syncthreads();        // the copies of the next item may overwrite every buffer
  }
}

// Pass 2 on the 5th-generation tensor cores (P = 128): per item (b, c, h) the outputs as
// their transpose, M = 128 head rows p by N = 64 steps t,
//   Y^T = X^T W^T + (H C^T) diag(exp(cs)),   W_ti = (C B^T)_ti exp(cs_t - cs_i) dt_i (t >= i),
// with D folded into W's diagonal (D x_t = sum_i x_i D [i == t]). Two TMEM accumulators per
// item (double-buffered across items): D1 = X^T W^T (X an MN-major operand with the
// 128-byte swizzle; W^T a K-major operand without swizzle, bf16 high + low, built by the
// workers from C B^T) and D2 = H C^T (H the walk's K-major image; C a K-major operand with
// the 128-byte swizzle, K-steps 32 bytes apart inside the swizzle atom). Warp-specialised
// like the walk, with two stages: warp 17's lane 0 copies item k by TMA and bulk copies into
// stage k % 2 once the MMAs of item k - 2 have read it; warps 0-15 zero the rows past L,
// build W^T and exp(cs), and write the previous item's outputs (warp w: head rows 32 (w % 4)
// .. + 31, one per thread, and steps 16 (w / 4) .. + 15; a warp stores 32 consecutive head
// channels of a step); warp 16's lane 0 issues 8 + N / 16 MMAs per item.
constexpr int kTcScanWorkers = 512;
constexpr int kTcScanThreads = kTcScanWorkers + 64;
template <int N>
struct SsdTcScan {
  static constexpr int Q = kSsdQ, P = kTcP;
  // one stage (two per CTA: item k in stage k % 2)
  static constexpr int kX = 0;                          // X: 2 halves [Q][128 B], swizzled
  static constexpr int kC = kX + Q * P * 2;             // C: N / 64 halves [Q][128 B], swizzled
  static constexpr int kH = kC + Q * N * 2;             // entering state, K-major image
  static constexpr int kCB = kH + P * N * 2;            // C B^T, Q rows of kSsdCBPitch floats
  static constexpr int kDt = kCB + Q * kSsdCBPitch * 4;
  static constexpr int kCs = kDt + Q * 4;
  static constexpr int kW = kCs + Q * 4;                // W^T high, then low: 8 x 8 core matrices each
  static constexpr int kStage = (kW + 2 * Q * Q * 2 + 1023) / 1024 * 1024;
  static constexpr int kEcs = 2 * kStage;               // exp(cs) of the last two items, [2][Q]
  static constexpr int kBar = kEcs + 2 * Q * 4;         // loaded[2], empty[2], full[2], tfull[2], tempty[2]
  static constexpr int kSlot = kBar + 10 * 8;
  static constexpr int kAbort = kSlot + 4;
  static constexpr int kBytes = kAbort + 12 + 1024;     // + room to align the base to 1 KB
  static constexpr uint32_t kTx = Q * P * 2 + Q * N * 2 + P * N * 2 + Q * kSsdCBPitch * 4 + 2 * Q * 4;
  static constexpr uint32_t kHsbo = (N / 8) * 128;      // H image: core matrices (p8, n8) at p8 kHsbo + n8 128
  static_assert(kC % 1024 == 0 && kH % 1024 == 0 && kW % 16 == 0, "operand alignment");
};

template <int N, typename TY>
__global__ void __launch_bounds__(kTcScanThreads, 1)
    ssd_chunk_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_c,
                             const SsdParams p) {
  using L = SsdTcScan<N>;
  constexpr int Q = kSsdQ, P = kTcP;
  constexpr uint32_t kIdesc1 = umma_idesc_bf16(P, Q, true, false);   // X^T (MN-major) x W^T (K-major)
  constexpr uint32_t kIdesc2 = umma_idesc_bf16(P, Q, false, false);  // H (K-major) x C^T (K-major)
  extern __shared__ __align__(16) unsigned char smem_dyn[];
  unsigned char* sm = smem_dyn + ((1024u - (umma_saddr(smem_dyn) & 1023u)) & 1023u);
  uint64_t* loaded = reinterpret_cast<uint64_t*>(sm + L::kBar);  // [2]
  uint64_t* empty = loaded + 2;                                   // [2]
  uint64_t* full = loaded + 4;                                    // [2]
  uint64_t* tfull = loaded + 6;                                   // [2]
  uint64_t* tempty = loaded + 8;                                  // [2]
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + L::kSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);
  float* ecs = reinterpret_cast<float*>(sm + L::kEcs);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t items = p.batch * p.nc * p.H;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&loaded[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&full[i], kTcScanWorkers);
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kTcScanWorkers);
    }
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_c);
    *abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (warp == 17) {  // ---------------- copier ----------------
    if (lane == 0 && !p.fault_skip_loads) {
      SsdItemWalk wk;
      wk.init(p, blockIdx.x, gridDim.x);
      for (int k = 0;; ++k, wk.advance()) {
        const int64_t it = blockIdx.x + (int64_t)k * gridDim.x;
        if (it >= items) break;
        const int s = k & 1;
        // stage s last held item k - 2: wait until its MMAs have read it
        if (k >= 2 && !tc_wait(&empty[s], (uint32_t)(((k - 2) >> 1) & 1), abort, p)) break;
        unsigned char* st = sm + s * L::kStage;
        const SsdItem m = wk.item();
        const int32_t row = (int32_t)(m.b * p.L + m.t0);
        mbar_arrive_expect_tx(&loaded[s], L::kTx);
        tma_load_3d_bar(st + L::kX, &tm_x, 0, (int32_t)m.h, row, &loaded[s]);
        tma_load_3d_bar(st + L::kX + 8192, &tm_x, 64, (int32_t)m.h, row, &loaded[s]);
#pragma unroll
        for (int hc = 0; hc < N / 64; ++hc)
          tma_load_2d(st + L::kC + hc * 8192, &tm_c, (int32_t)(m.g * N + 64 * hc), row, &loaded[s]);
        bulk_load(st + L::kH, p.ws_H + it * (int64_t)P * N, P * N * 2, &loaded[s]);
        bulk_load(st + L::kCB, p.ws_CB + ((m.b * p.nc + m.c) * p.G + m.g) * Q * kSsdCBPitch, Q * kSsdCBPitch * 4,
                  &loaded[s]);
        bulk_load(st + L::kDt, p.ws_dt + it * Q, Q * 4, &loaded[s]);
        bulk_load(st + L::kCs, p.ws_cs + it * Q, Q * 4, &loaded[s]);
      }
    }
  } else if (warp == 16) {  // ---------------- MMA issuer ----------------
    if (lane == 0) {
      for (int k = 0;; ++k) {
        const int64_t it = blockIdx.x + (int64_t)k * gridDim.x;
        if (it >= items) break;
        const int s = k & 1;
        if (!tc_wait(&full[s], (uint32_t)((k >> 1) & 1), abort, p)) break;
        if (k >= 2 && !tc_wait(&tempty[s], (uint32_t)(((k - 2) >> 1) & 1), abort, p)) break;
        tc_fence_after();
        const unsigned char* st = sm + s * L::kStage;
        const uint32_t xa = umma_saddr(st + L::kX), ca = umma_saddr(st + L::kC), ha = umma_saddr(st + L::kH);
        const uint32_t wh = umma_saddr(st + L::kW), wl = wh + Q * Q * 2;
        const uint32_t d1 = tmem + 128u * (uint32_t)s, d2 = d1 + 64u;
#pragma unroll
        for (int ks = 0; ks < Q / 16; ++ks) {  // X^T W^T over the chunk's steps i
          const uint64_t ad = umma_sdesc(xa + ks * 2048, 8192, 1024, 2);
          umma_bf16(d1, ad, umma_sdesc(wh + ks * 256, 128, 1024), kIdesc1, ks > 0);
          umma_bf16(d1, ad, umma_sdesc(wl + ks * 256, 128, 1024), kIdesc1, true);
        }
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks)  // H C^T over the state columns n
          umma_bf16(d2, umma_sdesc(ha + ks * 256, 128, L::kHsbo),
                    umma_sdesc(ca + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, 2), kIdesc2, ks > 0);
        umma_commit(&tfull[s]);
        umma_commit(&empty[s]);
      }
    }
  } else {  // ---------------- workers ----------------
    const int q = warp & 3, th = warp >> 2;  // TMEM lane quarter, quarter of the steps
    const int prow = 32 * q + lane;          // head row of this thread in the epilogue (TMEM lane)
    // item k's outputs (y rows of its chunk; the MMA results in TMEM buffer k % 2)
    auto epilogue = [&](int k, const SsdItem& m) {
      const int rv = (int)((p.L - m.t0) < Q ? (p.L - m.t0) : Q);
      const int bsel = k & 1;
      if (!tc_wait(&tfull[bsel], (uint32_t)((k >> 1) & 1), abort, p)) return false;
      tc_fence_after();
      uint32_t v1[16], v2[16];
      const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + 128u * (uint32_t)bsel + 16u * (uint32_t)th;
      tmem_ld16_nowait(ta, v1);
      tmem_ld16_nowait(ta + 64u, v2);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&tempty[bsel]);
      const float* e = ecs + bsel * Q + 16 * th;
      const int64_t ystride = p.H * P;
      TY* yb = static_cast<TY*>(p.y) + ((m.b * p.L + m.t0 + 16 * th) * p.H + m.h) * P + prow;
      const int tn = rv - 16 * th;  // steps of this quarter inside the sequence
      if (tn >= 16) {  // a whole quarter: no per-step bounds
#pragma unroll
        for (int c = 0; c < 16; ++c)
          yb[c * ystride] = from_f32<TY>(fmaf(e[c], __uint_as_float(v2[c]), __uint_as_float(v1[c])));
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (c < tn) *yb = from_f32<TY>(fmaf(e[c], __uint_as_float(v2[c]), __uint_as_float(v1[c])));
          yb += ystride;
        }
      }
      return true;
    };
    bool ok = true;
    int k = 0;
    SsdItemWalk wk;
    wk.init(p, blockIdx.x, gridDim.x);
    SsdItem mprev{};  // the previous item, whose outputs this iteration writes
    for (;; ++k, wk.advance()) {
      const int64_t it = blockIdx.x + (int64_t)k * gridDim.x;
      if (it >= items) break;
      const int s = k & 1;
      unsigned char* st = sm + s * L::kStage;
      const SsdItem m = wk.item();
      const int rv = (int)((p.L - m.t0) < Q ? (p.L - m.t0) : Q);
      if (ok && !tc_wait(&loaded[s], (uint32_t)((k >> 1) & 1), abort, p, kErrWaitFull)) ok = false;
      if (ok && rv < Q) {  // steps past L: zero rows of X (another batch row's data or fill)
        for (int i = tid; i < (Q - rv) * (P / 8); i += kTcScanWorkers) {
          const int t = rv + i / (P / 8), c = i % (P / 8);
          *reinterpret_cast<uint4*>(st + L::kX + (c >> 3) * 8192 + t * 128 + (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // the item's cs in log2 units, so that W's decays are one ex2 each
      if (ok && tid < Q) reinterpret_cast<float*>(st + L::kCs)[tid] *= kLog2e;
      if (!bar_and(ok, 1, kTcScanWorkers)) {
        ok = false;
        break;
      }
      {  // W^T (bf16 high + low, K-major core matrices (t / 8, i / 8)) and exp(cs) of item k
        const float* CBs = reinterpret_cast<const float*>(st + L::kCB);
        const float* dts = reinterpret_cast<const float*>(st + L::kDt);
        const float* css = reinterpret_cast<const float*>(st + L::kCs);
        const float Dh = p.Dskip ? p.Dskip[m.h] : 0.f;
#pragma unroll
        for (int r = 0; r < (Q * Q / 8) / kTcScanWorkers; ++r) {
          // eight consecutive threads write one core matrix (rows t % 8 of columns i8)
          const int u = tid + r * kTcScanWorkers;
          const int t8 = u >> 6, t = t8 * 8 + (u & 7), i8 = (u >> 3) & 7;
          const float ct = css[t];
          const int off = (t >> 3) * 1024 + i8 * 128 + (t & 7) * 16;
          uint4 hv = make_uint4(0u, 0u, 0u, 0u), lv = hv;
          if (i8 <= t8) {  // blocks above the diagonal stay zero
            const float4 cb0 = *reinterpret_cast<const float4*>(CBs + t * kSsdCBPitch + 8 * i8);
            const float4 cb1 = *reinterpret_cast<const float4*>(CBs + t * kSsdCBPitch + 8 * i8 + 4);
            const float4 ci0 = *reinterpret_cast<const float4*>(css + 8 * i8);
            const float4 ci1 = *reinterpret_cast<const float4*>(css + 8 * i8 + 4);
            const float4 di0 = *reinterpret_cast<const float4*>(dts + 8 * i8);
            const float4 di1 = *reinterpret_cast<const float4*>(dts + 8 * i8 + 4);
            const float cbv[8] = {cb0.x, cb0.y, cb0.z, cb0.w, cb1.x, cb1.y, cb1.z, cb1.w};
            const float civ[8] = {ci0.x, ci0.y, ci0.z, ci0.w, ci1.x, ci1.y, ci1.z, ci1.w};
            const float div[8] = {di0.x, di0.y, di0.z, di0.w, di1.x, di1.y, di1.z, di1.w};
            float w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int i = 8 * i8 + e;
              w[e] = t >= i ? cbv[e] * ex2(ct - civ[e]) * div[e] : 0.f;
              if (t == i) w[e] += Dh;
            }
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split_bf16x2(make_float2(w[2 * e], w[2 * e + 1]), hi[e], lo[e]);
            hv = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            lv = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
          *reinterpret_cast<uint4*>(st + L::kW + off) = hv;
          *reinterpret_cast<uint4*>(st + L::kW + Q * Q * 2 + off) = lv;
          if (i8 == 0) ecs[s * Q + t] = ex2(ct);
        }
      }
      fence_smem_to_async();
      mbar_arrive(&full[s]);
      if (k >= 1 && !epilogue(k - 1, mprev)) ok = false;
      mprev = m;
    }
    if (ok && k >= 1) epilogue(k - 1, mprev);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace ssm
