"""Seeded synthetic inputs for the selective scan and the decode step.

This module only draws random numbers and lays them out. It holds none of the scan's
arithmetic, so both the CUDA path and the CPU oracle can consume what it produces.

Recipe (one torch.Generator per workload, seeded with the workload's seed, on the
device the tensors are created on; draws in the fixed order u, delta, z, B, C, D_skip,
delta_bias, all in fp32, then rounded to the I/O type with round-to-nearest-even):

    u, z, B, C, D_skip   ~ N(0, 1)
    delta (raw)          ~ N(-2, 0.5)               (goes through +bias and softplus)
    delta_bias           ~ U(log(e^0.001 - 1), log(e^0.1 - 1))   (when the workload has one)
    A[d, n]              = -(n + 1)                  (S4D-real initialisation)

Decode: x, z, B, C, D_skip ~ N(0, 1); the step size is the softplus of an N(0, 1)
draw (a positive distribution: a raw N(0,1) step would make exp(delta*A) grow without
bound); the state starts at zero.

Workload sizes follow the 130M-, 1.4B- and 2.8B-parameter Mamba layer shapes
(d_inner = 2 * d_model, N = 16) plus a tiny fp32 case and a 131072-token sequence.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class FwdWorkload:
    name: str
    batch: int
    L: int
    D: int
    N: int
    dtype: torch.dtype
    has_bias: bool
    seed: int
    delta_softplus: bool = True
    notes: str = ""

    @property
    def elems(self) -> int:
        """B*L*D, the unit of the elem/s metric."""
        return self.batch * self.L * self.D

    @property
    def element_steps(self) -> int:
        """B*L*D*N: one discretise + update + read-out each."""
        return self.batch * self.L * self.D * self.N

    def compulsory_bytes(self, y_dtype: torch.dtype | None = None, last_state: bool = True) -> int:
        """Inputs read once plus outputs written once (B/C re-reads excluded)."""
        io = torch.finfo(self.dtype).bits // 8
        yb = torch.finfo(y_dtype or self.dtype).bits // 8
        bld = self.batch * self.L * self.D
        n = 3 * bld * io + bld * yb                    # u, delta, z in; y out
        n += 2 * self.batch * self.L * self.N * io     # B, C
        n += self.D * self.N * 4 + self.D * 4          # A, D_skip
        n += self.D * 4 if self.has_bias else 0        # delta_bias
        n += self.batch * self.D * self.N * 4 if last_state else 0
        return n


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    D: int
    N: int
    steps: int
    dtype: torch.dtype
    seed: int

    def bytes_per_step(self, y_dtype: torch.dtype | None = None) -> int:
        io = torch.finfo(self.dtype).bits // 8
        yb = torch.finfo(y_dtype or self.dtype).bits // 8
        bd = self.batch * self.D
        n = 2 * bd * self.N * 4                        # state read + written
        n += 3 * bd * io + bd * yb                     # x, delta, z in; y out
        n += 2 * self.batch * self.N * io              # B, C
        n += self.D * self.N * 4 + self.D * 4          # A, D_skip
        return n


TINY = FwdWorkload("tiny fp32 scan (1x256x64, N=16)", 1, 256, 64, 16, torch.float32, False, 0)
M130 = FwdWorkload("Mamba-130M layer scan (8x2048x1536, N=16)", 8, 2048, 1536, 16, torch.bfloat16, True, 1)
M1P4 = FwdWorkload("Mamba-1.4B layer scan (4x4096x4096, N=16)", 4, 4096, 4096, 16, torch.bfloat16, True, 2)
LONG = FwdWorkload("long-sequence scan (1x131072x2048, N=16)", 1, 131072, 2048, 16, torch.bfloat16, True, 3)
DECODE = DecodeWorkload("decode step, Mamba-2.8B layer (256x5120, N=16) x1024", 256, 5120, 16, 1024,
                        torch.bfloat16, 4)

# A quarter-length cut of the 1.4B layer (135 MB of inputs, still larger than L2) that
# profilers can replay quickly.
M1P4_L1024 = FwdWorkload("Mamba-1.4B layer scan, L cut to 1024 (4x1024x4096, N=16)", 4, 1024, 4096, 16,
                         torch.bfloat16, True, 2)

FWD_WORKLOADS = {"tiny": TINY, "m130m": M130, "m1p4b": M1P4, "long": LONG, "m1p4b_L1024": M1P4_L1024}

BIAS_LO = math.log(math.expm1(0.001))
BIAS_HI = math.log(math.expm1(0.1))


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def s4d_real_A(D: int, N: int, device="cpu") -> torch.Tensor:
    """A[d, n] = -(n + 1), fp32."""
    return (-torch.arange(1, N + 1, dtype=torch.float32, device=device)).repeat(D, 1).contiguous()


def fwd_inputs(w: FwdWorkload, device="cpu", seed: int | None = None, lti: bool = False) -> dict:
    """All forward-pass tensors of workload ``w`` on ``device``.

    ``lti=True`` gives the time-invariant sub-case: delta, B and C of step 0 repeated
    over every t (u and z still vary).
    """
    g = _gen(device, w.seed if seed is None else seed)
    b, L, D, N = w.batch, w.L, w.D, w.N
    f32 = torch.float32
    u = torch.randn(b, L, D, generator=g, device=device, dtype=f32)
    delta = torch.randn(b, L, D, generator=g, device=device, dtype=f32) * 0.5 - 2.0
    z = torch.randn(b, L, D, generator=g, device=device, dtype=f32)
    B = torch.randn(b, L, N, generator=g, device=device, dtype=f32)
    C = torch.randn(b, L, N, generator=g, device=device, dtype=f32)
    Dskip = torch.randn(D, generator=g, device=device, dtype=f32)
    bias = None
    if w.has_bias:
        bias = torch.rand(D, generator=g, device=device, dtype=f32) * (BIAS_HI - BIAS_LO) + BIAS_LO
    if lti:
        delta = delta[:, :1, :].expand(b, L, D)
        B = B[:, :1, :].expand(b, L, N)
        C = C[:, :1, :].expand(b, L, N)
    io = w.dtype
    return dict(
        u=u.to(io).contiguous(), delta=delta.to(io).contiguous(), z=z.to(io).contiguous(),
        B=B.to(io).contiguous(), C=C.to(io).contiguous(), D=Dskip.contiguous(),
        delta_bias=None if bias is None else bias.contiguous(), A=s4d_real_A(D, N, device),
        delta_softplus=w.delta_softplus,
    )


def decode_inputs(w: DecodeWorkload, device="cpu", steps: int | None = None, seed: int | None = None) -> dict:
    """Per-step decode tensors stacked over steps: x, delta, z (steps, batch, D); B, C
    (steps, batch, N); plus A (D, N), D (D) and a zero state (batch, D, N)."""
    g = _gen(device, w.seed if seed is None else seed)
    T = w.steps if steps is None else steps
    b, D, N = w.batch, w.D, w.N
    io, f32 = w.dtype, torch.float32
    x = torch.empty(T, b, D, dtype=io, device=device)
    delta = torch.empty(T, b, D, dtype=io, device=device)
    z = torch.empty(T, b, D, dtype=io, device=device)
    chunk = max(1, (1 << 26) // max(1, b * D))  # bound the fp32 staging to ~256 MB per tensor
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        x[t0:t1] = torch.randn(t1 - t0, b, D, generator=g, device=device, dtype=f32).to(io)
        raw = torch.randn(t1 - t0, b, D, generator=g, device=device, dtype=torch.float64)
        delta[t0:t1] = torch.nn.functional.softplus(raw).to(io)
        z[t0:t1] = torch.randn(t1 - t0, b, D, generator=g, device=device, dtype=f32).to(io)
    B = torch.randn(T, b, N, generator=g, device=device, dtype=f32).to(io)
    C = torch.randn(T, b, N, generator=g, device=device, dtype=f32).to(io)
    Dskip = torch.randn(D, generator=g, device=device, dtype=f32)
    return dict(x=x, delta=delta, z=z, B=B, C=C, D=Dskip, A=s4d_real_A(D, N, device),
                state=torch.zeros(b, D, N, dtype=f32, device=device))


def random_fwd(batch, L, D, N, dtype=torch.float32, device="cpu", seed=0, has_bias=True,
               has_D=True, has_z=True, delta_softplus=True) -> dict:
    """Arbitrary-shape forward inputs with the same distributions (for parity sweeps)."""
    w = FwdWorkload("random", batch, L, D, N, dtype, has_bias, seed, delta_softplus)
    d = fwd_inputs(w, device)
    if not has_D:
        d["D"] = None
    if not has_z:
        d["z"] = None
    return d


# ---- Mamba-2 SSD ------------------------------------------------------------------------
@dataclass(frozen=True)
class SsdWorkload:
    name: str
    batch: int
    L: int
    H: int
    P: int
    N: int
    G: int
    seed: int

    @property
    def tokens(self) -> int:
        return self.batch * self.L

    def flops(self, Q: int = 64) -> int:
        """Tensor-core work of the chunked algorithm per call: per chunk and head the
        contractions C B^T (2 Q^2 N), W X (2 Q^2 P), C S^T (2 Q N P) and X^T (w B) (2 Q N P),
        i.e. 2 Q N + 2 Q P + 4 N P per token and head (a ragged last chunk counted whole)."""
        chunks = (self.L + Q - 1) // Q
        return self.batch * self.H * chunks * (2 * Q * Q * self.N + 2 * Q * Q * self.P + 4 * Q * self.N * self.P)

    def compulsory_bytes(self) -> int:
        """x and y (bf16), delta (bf16), B and C (bf16), A, D, dt_bias (fp32), last_state (fp32)."""
        b, L, H, P, N, G = self.batch, self.L, self.H, self.P, self.N, self.G
        return 2 * (2 * b * L * H * P + b * L * H + 2 * b * L * G * N) + 4 * 3 * H + 4 * b * H * P * N


# A Mamba-2 layer in the pages' shape: "24 heads x 128 dims" per head; d_state 128 (the pages
# give none for Mamba-2; the common choice), one B/C group.
SSD_M2 = SsdWorkload("Mamba-2 layer SSD (4x4096, 24 heads x P=128, N=128, G=1)", 4, 4096, 24, 128, 128, 1, 7)


def ssd_inputs(w: SsdWorkload, device="cpu", seed: int | None = None) -> dict:
    """SSD tensors: x, B, C ~ N(0,1) and D ~ N(0,1) as for the Mamba-1 workloads; raw step
    size ~ N(-2, 0.5) plus a bias ~ U(log(e^0.001 - 1), log(e^0.1 - 1)) through softplus;
    A per head ~ -U(1, 16). bf16 x, delta, B, C; fp32 A, D, bias."""
    g = _gen(device, w.seed if seed is None else seed)
    b, L, H, P, N, G = w.batch, w.L, w.H, w.P, w.N, w.G
    f32, bf = torch.float32, torch.bfloat16
    x = torch.randn(b, L, H, P, generator=g, device=device, dtype=f32)
    delta = torch.randn(b, L, H, generator=g, device=device, dtype=f32) * 0.5 - 2.0
    B = torch.randn(b, L, G, N, generator=g, device=device, dtype=f32)
    C = torch.randn(b, L, G, N, generator=g, device=device, dtype=f32)
    D = torch.randn(H, generator=g, device=device, dtype=f32)
    bias = torch.rand(H, generator=g, device=device, dtype=f32) * (BIAS_HI - BIAS_LO) + BIAS_LO
    A = -(torch.rand(H, generator=g, device=device, dtype=f32) * 15.0 + 1.0)
    return dict(x=x.to(bf).contiguous(), delta=delta.to(bf).contiguous(), A=A, B=B.to(bf).contiguous(),
                C=C.to(bf).contiguous(), D=D, dt_bias=bias, dt_softplus=True)
