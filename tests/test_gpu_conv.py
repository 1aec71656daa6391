"""GPU parity of the conv prologue (the block's causal width-4 depthwise conv + SiLU in
front of the SSM, "Mamba and State Space Models", "The Mamba Block") fused into the
forward pass and the decode step, against the fp64 oracle (conv, then the scan) and
against structural identities: a sequence cut anywhere continues exactly from the
carried conv state and SSM state.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL_BF16, TOL_F32, check, to64
from selective_state_space_141_b300 import inputs, ssm

pytestmark = pytest.mark.gpu
DEV = "cuda"


def conv_inputs(b, L, D, N, dtype, seed):
    d = inputs.random_fwd(b, L, D, N, dtype, DEV, seed=seed)
    g = torch.Generator(device="cpu").manual_seed(seed + 1000)
    d["x"] = d.pop("u")
    d["conv_weight"] = (torch.randn(D, 4, generator=g) * 0.5).to(DEV)
    d["conv_bias"] = (torch.randn(D, generator=g) * 0.1).to(DEV)
    d["conv_state"] = torch.randn(b, D, 3, generator=g).to(dtype).to(DEV)
    return d


def gpu(d, conv_state, h0=None, y_dtype=None, use_workspace=True, sl=slice(None)):
    cut = lambda t: None if t is None else t[:, sl].contiguous()
    y, last = ssm.conv_selective_scan_fwd(cut(d["x"]), d["conv_weight"], cut(d["delta"]), d["A"], cut(d["B"]),
                                          cut(d["C"]), conv_bias=d["conv_bias"], conv_state=conv_state, D=d["D"],
                                          z=cut(d["z"]), delta_bias=d["delta_bias"],
                                          delta_softplus=d["delta_softplus"], h0=h0, y_dtype=y_dtype,
                                          use_workspace=use_workspace)
    torch.cuda.synchronize()
    assert ssm.device_error() == 0
    return y, last


def ref(d, conv_state, h0=None):
    return oracle.conv_selective_scan_fwd(d["x"], d["conv_weight"], d["A"], d["B"], d["C"], d["delta"],
                                          conv_bias=d["conv_bias"], conv_state=conv_state, D=d["D"], z=d["z"],
                                          delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"], h0=h0)


@pytest.mark.parametrize("shape", [(2, 77, 256, 16), (1, 130, 384, 8), (3, 45, 100, 16), (2, 33, 70, 4)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("with_state", [True, False], ids=["state", "zeros"])
def test_conv_fwd_vs_oracle(shape, dtype, with_state):
    b, L, D, N = shape
    d = conv_inputs(b, L, D, N, dtype, seed=71 + L)
    cs = d["conv_state"].clone() if with_state else None
    yr, lr, csr = ref(d, cs)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    y, last = gpu(d, cs)
    check(y, yr, tol, dtype == torch.bfloat16, "y")
    check(last, lr, tol, False, "last_state")
    if with_state:
        assert np.array_equal(to64(cs), csr), "next conv state"
    if dtype == torch.bfloat16:
        y32, _ = gpu(d, None if cs is None else d["conv_state"].clone(), y_dtype=torch.float32)
        check(y32, yr, tol, False, "y (fp32 output)")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("split", [1, 2, 3, 37, 64])
def test_conv_chunked_prefill_is_bit_exact(dtype, split, monkeypatch):
    """prefix, then the rest from the carried conv state and SSM state == one pass, bit
    for bit with the sequence segments off (segments reassociate the recurrence)."""
    monkeypatch.setenv("SSM_B300_SEGMENTS", "0")
    b, L, D, N = 2, 160, 256, 16
    d = conv_inputs(b, L, D, N, dtype, seed=72)
    cs_all = d["conv_state"].clone()
    y_all, last_all = gpu(d, cs_all)
    cs = d["conv_state"].clone()
    y1, mid = gpu(d, cs, sl=slice(0, split))
    y2, last2 = gpu(d, cs, h0=mid, sl=slice(split, L))
    assert torch.equal(torch.cat([y1, y2], dim=1), y_all)
    assert torch.equal(last2, last_all)
    assert torch.equal(cs, cs_all)


def test_conv_segmented_schedule(monkeypatch):
    """Later segments take their first three conv inputs from x before their start."""
    b, L, D, N = 1, 16384, 256, 16
    assert ssm.workspace_size(b, L, D, N) > 0
    d = conv_inputs(b, L, D, N, torch.bfloat16, seed=73)
    y, last = gpu(d, d["conv_state"].clone(), y_dtype=torch.float32)
    y_y, last_y = gpu(d, d["conv_state"].clone(), y_dtype=torch.float32, use_workspace=False)  # carries in y
    assert torch.equal(y, y_y) and torch.equal(last, last_y)
    monkeypatch.setenv("SSM_B300_SEGMENTS", "0")
    y_u, last_u = gpu(d, d["conv_state"].clone(), y_dtype=torch.float32, use_workspace=False)
    monkeypatch.delenv("SSM_B300_SEGMENTS")
    check(y, y_u, TOL_BF16, False, "segmented vs unsegmented y")
    check(last, last_u, TOL_BF16, False, "segmented vs unsegmented last_state")
    ds = np.sort(np.random.default_rng(74).choice(D, size=10, replace=False))
    idx = torch.as_tensor(ds, device=DEV)
    sub = dict(d)
    for k in ("x", "delta", "z"):
        sub[k] = d[k].index_select(2, idx)
    for k in ("A", "D", "delta_bias", "conv_weight", "conv_bias"):
        sub[k] = d[k].index_select(0, idx)
    yr, lr, _ = ref(sub, d["conv_state"].index_select(1, idx))
    check(y.index_select(2, idx), yr, TOL_BF16, False, "y sampled vs oracle")
    check(last.index_select(1, idx), lr, TOL_BF16, False, "last_state sampled vs oracle")


@pytest.mark.parametrize("N", [4, 8, 16])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_conv_decode_vs_oracle(N, dtype):
    b, D = 3, 150
    g = torch.Generator(device="cpu").manual_seed(75 + N)
    cs = torch.randn(b, D, 3, generator=g).to(dtype).to(DEV)
    state = torch.randn(b, D, N, generator=g).to(DEV)
    x = torch.randn(b, D, generator=g).to(dtype).to(DEV)
    w = (torch.randn(D, 4, generator=g) * 0.5).to(DEV)
    cb = (torch.randn(D, generator=g) * 0.1).to(DEV)
    raw = (torch.randn(b, D, generator=g) * 0.5 - 2.0).to(dtype).to(DEV)
    bias = (torch.rand(D, generator=g) * 0.05).to(DEV)
    A = -(torch.rand(D, N, generator=g) * 4 + 0.1).to(DEV)
    B = torch.randn(b, N, generator=g).to(dtype).to(DEV)
    C = torch.randn(b, N, generator=g).to(dtype).to(DEV)
    Dk = torch.randn(D, generator=g).to(DEV)
    z = torch.randn(b, D, generator=g).to(dtype).to(DEV)
    u = oracle.conv1d_silu(to64(x)[:, None, :], w, cb, cs)[:, 0, :]
    yr, sr = oracle.state_update(state, u, raw, A, B, C, D=Dk, z=z, delta_bias=bias, delta_softplus=True)
    csr = oracle.next_conv_state(to64(x)[:, None, :], cs)
    st, c = state.clone(), cs.clone()
    y = ssm.conv_state_update(c, st, x, w, raw, A, B, C, conv_bias=cb, D=Dk, z=z, delta_bias=bias,
                              delta_softplus=True)
    torch.cuda.synchronize()
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    check(y, yr, tol, dtype == torch.bfloat16, "y")
    check(st, sr, tol, False, "state")
    assert np.array_equal(to64(c), csr), "conv state"


def test_conv_decode_continues_forward():
    """conv forward over a prefix, then conv decode token by token, reproduces the conv
    forward over the whole sequence (prefill -> decode hand-off)."""
    b, L, D, N, P = 2, 40, 256, 16, 33
    d = conv_inputs(b, L, D, N, torch.bfloat16, seed=76)
    y_all, last_all = gpu(d, d["conv_state"].clone(), y_dtype=torch.float32)
    cs = d["conv_state"].clone()
    _, st = gpu(d, cs, sl=slice(0, P))
    for t in range(P, L):
        y = ssm.conv_state_update(cs, st, d["x"][:, t].contiguous(), d["conv_weight"], d["delta"][:, t].contiguous(),
                                  d["A"], d["B"][:, t].contiguous(), d["C"][:, t].contiguous(),
                                  conv_bias=d["conv_bias"], D=d["D"], z=d["z"][:, t].contiguous(),
                                  delta_bias=d["delta_bias"], delta_softplus=True, y_dtype=torch.float32)
        check(y, y_all[:, t], TOL_BF16, False, f"y t={t}")
    torch.cuda.synchronize()
    check(st, last_all, TOL_BF16, False, "state")


@pytest.mark.parametrize("with_conv_bias", [True, False], ids=["conv-bias", "no-conv-bias"])
def test_conv_decode_streamed_kernel(with_conv_bias, monkeypatch):
    """bf16, N = 16, D a multiple of 128: the conv decode step runs on the streamed kernel
    (conv state, weights and bias streamed with each tile, conv state shifted in place);
    three steps against the oracle, and bit for bit against the per-thread kernel
    (SSM_B300_DECODE=plain) on the same inputs."""
    b, D, N, T = 3, 384, 16, 3
    g = torch.Generator(device="cpu").manual_seed(77)
    cs0 = torch.randn(b, D, 3, generator=g).to(torch.bfloat16).to(DEV)
    s0 = torch.randn(b, D, N, generator=g).to(DEV)
    xs = torch.randn(T, b, D, generator=g).to(torch.bfloat16).to(DEV)
    w = (torch.randn(D, 4, generator=g) * 0.5).to(DEV)
    cb = (torch.randn(D, generator=g) * 0.1).to(DEV) if with_conv_bias else None
    raws = (torch.randn(T, b, D, generator=g) * 0.5 - 2.0).to(torch.bfloat16).to(DEV)
    bias = (torch.rand(D, generator=g) * 0.05).to(DEV)
    A = -(torch.rand(D, N, generator=g) * 4 + 0.1).to(DEV)
    Bs = torch.randn(T, b, N, generator=g).to(torch.bfloat16).to(DEV)
    Cs = torch.randn(T, b, N, generator=g).to(torch.bfloat16).to(DEV)
    Dk = torch.randn(D, generator=g).to(DEV)
    zs = torch.randn(T, b, D, generator=g).to(torch.bfloat16).to(DEV)
    runs = {}
    for mode in ("stream", "plain"):
        if mode == "plain":
            monkeypatch.setenv("SSM_B300_DECODE", "plain")
        st, c = s0.clone(), cs0.clone()
        ys = [ssm.conv_state_update(c, st, xs[t], w, raws[t], A, Bs[t], Cs[t], conv_bias=cb, D=Dk, z=zs[t],
                                    delta_bias=bias, delta_softplus=True, y_dtype=torch.float32) for t in range(T)]
        torch.cuda.synchronize()
        runs[mode] = (ys, st, c)
    monkeypatch.delenv("SSM_B300_DECODE")
    for t in range(T):
        assert torch.equal(runs["stream"][0][t], runs["plain"][0][t]), t
    assert torch.equal(runs["stream"][1], runs["plain"][1]) and torch.equal(runs["stream"][2], runs["plain"][2])
    st_ref, cs_ref = to64(s0), to64(cs0)
    for t in range(T):
        u = oracle.conv1d_silu(to64(xs[t])[:, None, :], w, cb, cs_ref)[:, 0, :]
        yr, st_ref = oracle.state_update(st_ref, u, raws[t], A, Bs[t], Cs[t], D=Dk, z=zs[t], delta_bias=bias,
                                         delta_softplus=True)
        cs_ref = oracle.next_conv_state(to64(xs[t])[:, None, :], cs_ref)
        check(runs["stream"][0][t], yr, TOL_BF16, False, f"y step {t}")
    check(runs["stream"][1], st_ref, TOL_BF16, False, "state")
    assert np.array_equal(to64(runs["stream"][2]), cs_ref), "conv state"
