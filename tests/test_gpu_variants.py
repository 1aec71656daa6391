"""GPU parity of the interface variants, against the fp64 oracle and against the plain
entry points: the forward pass from a given start state and with the zero-order-hold
B-bar (ssm_selective_scan_fwd_ex), and the decode step with the step-size map and the
zero-order-hold option applied inside (ssm_state_update_ex).

A start state continues a sequence ("Mamba and State Space Models", "Common Pitfalls":
the state after a prefix is reusable), so the strongest check is structural: a prefix
followed by the rest from the prefix's last_state must reproduce one call over the
whole sequence. Both passes run the same per-step arithmetic from the same fp32
state, so on the unsegmented kernels the two results are bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL_BF16, TOL_F32, check, to64
from selective_state_space_141_b300 import inputs, ssm

pytestmark = pytest.mark.gpu
DEV = "cuda"


def fwd(d, h0=None, sl=slice(None), last_state=None, y_dtype=None, use_workspace=True):
    y, last = ssm.selective_scan_fwd(d["u"][:, sl], d["delta"][:, sl], d["A"], d["B"][:, sl], d["C"][:, sl],
                                     D=d["D"], z=None if d["z"] is None else d["z"][:, sl],
                                     delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"], h0=h0,
                                     last_state=last_state, y_dtype=y_dtype, use_workspace=use_workspace)
    torch.cuda.synchronize()
    assert ssm.device_error() == 0
    return y, last


def contiguous_slice(d, sl):
    out = dict(d)
    for k in ("u", "delta", "z", "B", "C"):
        if d[k] is not None:
            out[k] = d[k][:, sl].contiguous()
    return out


def oracle_fwd(d, h0):
    return oracle.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"], h0=h0)


@pytest.mark.parametrize("shape", [(2, 77, 256, 16), (3, 45, 100, 8), (1, 130, 384, 16), (2, 33, 70, 4)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_fwd_h0_vs_oracle(shape, dtype):
    b, L, D, N = shape
    d = inputs.random_fwd(b, L, D, N, dtype, DEV, seed=41 + L)
    g = torch.Generator(device="cpu").manual_seed(42)
    h0 = torch.randn(b, D, N, generator=g).to(DEV)
    yr, lr = oracle_fwd(d, h0)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    y, last = fwd(d, h0=h0)
    check(y, yr, tol, dtype == torch.bfloat16, "y")
    check(last, lr, tol, False, "last_state")
    if dtype == torch.bfloat16:
        y32, _ = fwd(d, h0=h0, y_dtype=torch.float32)
        check(y32, yr, tol, False, "y (fp32 output)")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("split", [1, 37, 64, 199])
def test_chunked_prefill_is_bit_exact(dtype, split, monkeypatch):
    """prefix, then the rest from the prefix's last_state == one pass: bitwise with the
    sequence segments off (SSM_B300_SEGMENTS=0), within tolerance with them."""
    b, L, D, N = 2, 256, 256, 16
    d = inputs.random_fwd(b, L, D, N, dtype, DEV, seed=43)
    p = contiguous_slice(d, slice(0, split))
    r = contiguous_slice(d, slice(split, L))
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    y_seg, last_seg = fwd(d)
    y1, mid = fwd(p)
    y2, last2 = fwd(r, h0=mid)
    check(torch.cat([y1, y2], dim=1), y_seg, tol, False, "prefix + rest vs one pass")
    check(last2, last_seg, tol, False, "last_state")
    monkeypatch.setenv("SSM_B300_SEGMENTS", "0")
    y_all, last_all = fwd(d)
    y1, mid = fwd(p)
    y2, last2 = fwd(r, h0=mid)
    assert torch.equal(torch.cat([y1, y2], dim=1), y_all)
    assert torch.equal(last2, last_all)


def test_h0_in_place_state():
    """last_state may be the h0 buffer itself: the state is carried in one tensor."""
    b, L, D, N = 2, 96, 256, 16
    d = inputs.random_fwd(b, L, D, N, torch.bfloat16, DEV, seed=44)
    g = torch.Generator(device="cpu").manual_seed(45)
    h0 = torch.randn(b, D, N, generator=g).to(DEV)
    y_ref, last_ref = fwd(d, h0=h0.clone())
    st = h0.clone()
    y, last = fwd(d, h0=st, last_state=st)
    assert last.data_ptr() == st.data_ptr()
    assert torch.equal(y, y_ref) and torch.equal(st, last_ref)


def test_h0_zero_length_copies_state():
    g = torch.Generator(device="cpu").manual_seed(46)
    h0 = torch.randn(2, 64, 16, generator=g).to(DEV)
    d = inputs.random_fwd(2, 0, 64, 16, torch.bfloat16, DEV, seed=46)
    _, last = fwd(d, h0=h0)
    assert torch.equal(last, h0)


def test_h0_zeros_equals_plain_call():
    d = inputs.random_fwd(2, 150, 384, 16, torch.bfloat16, DEV, seed=47)
    y0, l0 = fwd(d)
    y1, l1 = fwd(d, h0=torch.zeros(2, 384, 16, device=DEV))
    assert torch.equal(y0, y1) and torch.equal(l0, l1)


def test_h0_segmented_schedule():
    """A long sequence over few channels takes the segmented schedule; the start state
    enters the carry scan as its first element. Sampled channels vs the oracle, and the
    whole output vs the unsegmented kernel."""
    b, L, D, N = 1, 16384, 256, 16
    assert ssm.workspace_size(b, L, D, N) > 0, "shape no longer takes the segmented schedule"
    d = inputs.random_fwd(b, L, D, N, torch.bfloat16, DEV, seed=48)
    g = torch.Generator(device="cpu").manual_seed(49)
    h0 = torch.randn(b, D, N, generator=g).to(DEV)
    y, last = fwd(d, h0=h0, y_dtype=torch.float32)
    y_u, last_u = fwd(d, h0=h0, y_dtype=torch.float32, use_workspace=False)
    check(y, y_u, TOL_BF16, False, "segmented vs unsegmented y")
    check(last, last_u, TOL_BF16, False, "segmented vs unsegmented last_state")
    ds = np.sort(np.random.default_rng(50).choice(D, size=12, replace=False))
    idx = torch.as_tensor(ds, device=DEV)
    sub = dict(d)
    for k in ("u", "delta", "z"):
        sub[k] = d[k].index_select(2, idx)
    sub["A"] = d["A"].index_select(0, idx)
    sub["D"] = d["D"].index_select(0, idx)
    sub["delta_bias"] = d["delta_bias"].index_select(0, idx)
    yr, lr = oracle_fwd(sub, h0.index_select(1, idx))
    check(y.index_select(2, idx), yr, TOL_BF16, False, "y sampled vs oracle")
    check(last.index_select(1, idx), lr, TOL_BF16, False, "last_state sampled vs oracle")


@pytest.mark.parametrize("N", [4, 8, 16])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("softplus", [True, False], ids=["softplus", "bias-only"])
def test_decode_ex_vs_oracle(N, dtype, softplus):
    b, D = 3, 150
    g = torch.Generator(device="cpu").manual_seed(51 + N)
    state = torch.randn(b, D, N, generator=g).to(DEV)
    x = torch.randn(b, D, generator=g).to(dtype).to(DEV)
    raw = (torch.randn(b, D, generator=g) * 0.5 - 2.0).to(dtype).to(DEV)
    if not softplus:
        raw = torch.rand(b, D, generator=g).to(dtype).to(DEV)  # dt = raw + bias stays positive
    bias = (torch.rand(D, generator=g) * 0.05 + 0.01).to(DEV)
    A = -(torch.rand(D, N, generator=g) * 4 + 0.1).to(DEV)
    B = torch.randn(b, N, generator=g).to(dtype).to(DEV)
    C = torch.randn(b, N, generator=g).to(dtype).to(DEV)
    Dk = torch.randn(D, generator=g).to(DEV)
    z = torch.randn(b, D, generator=g).to(dtype).to(DEV)
    yr, sr = oracle.state_update(state, x, raw, A, B, C, D=Dk, z=z, delta_bias=bias, delta_softplus=softplus)
    st = state.clone()
    y = ssm.state_update(st, x, raw, A, B, C, D=Dk, z=z, delta_bias=bias, delta_softplus=softplus)
    torch.cuda.synchronize()
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    check(y, yr, tol, dtype == torch.bfloat16, "y")
    check(st, sr, tol, False, "state")


def test_decode_ex_continues_forward():
    """forward over a prefix, then decode_ex token by token with the same bias and
    softplus, reproduces the forward pass over the whole sequence."""
    b, L, D, N, P = 2, 48, 256, 16, 40
    d = inputs.random_fwd(b, L, D, N, torch.bfloat16, DEV, seed=52)
    y_all, last_all = fwd(d, y_dtype=torch.float32)
    _, st = fwd(contiguous_slice(d, slice(0, P)))
    for t in range(P, L):
        y = ssm.state_update(st, d["u"][:, t].contiguous(), d["delta"][:, t].contiguous(), d["A"],
                             d["B"][:, t].contiguous(), d["C"][:, t].contiguous(), D=d["D"],
                             z=d["z"][:, t].contiguous(), delta_bias=d["delta_bias"], delta_softplus=True,
                             y_dtype=torch.float32)
        check(y, y_all[:, t], TOL_BF16, False, f"y t={t}")
    torch.cuda.synchronize()
    check(st, last_all, TOL_BF16, False, "state")


@pytest.mark.parametrize("shape", [(2, 77, 256, 16), (3, 45, 100, 8), (1, 70, 40, 4)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_fwd_zoh_vs_oracle(shape, dtype):
    """B-bar from the exact zero-order hold, from a random start state."""
    b, L, D, N = shape
    d = inputs.random_fwd(b, L, D, N, dtype, DEV, seed=61 + L)
    g = torch.Generator(device="cpu").manual_seed(62)
    h0 = torch.randn(b, D, N, generator=g).to(DEV)
    yr, lr = oracle.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                       delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"], h0=h0,
                                       zoh=True)
    y, last = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                     delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"], h0=h0,
                                     zoh=True)
    torch.cuda.synchronize()
    assert ssm.device_error() == 0
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    check(y, yr, tol, dtype == torch.bfloat16, "y")
    check(last, lr, tol, False, "last_state")
    # and it differs from the dt * B discretisation by more than the tolerance
    yd, _ = oracle.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                      delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"], h0=h0)
    assert np.max(np.abs(yd - yr)) > 10 * tol * np.sqrt(np.mean(yr * yr)) or dtype == torch.bfloat16


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_zoh_vs_oracle(dtype):
    b, D, N = 4, 96, 16
    g = torch.Generator(device="cpu").manual_seed(63)
    state = torch.randn(b, D, N, generator=g).to(DEV)
    x = torch.randn(b, D, generator=g).to(dtype).to(DEV)
    raw = (torch.randn(b, D, generator=g) * 0.5 - 1.0).to(dtype).to(DEV)
    bias = (torch.rand(D, generator=g) * 0.05).to(DEV)
    A = -(torch.rand(D, N, generator=g) * 4 + 0.1).to(DEV)
    A[3, 5] = 0.0  # the a = 0 limit
    B = torch.randn(b, N, generator=g).to(dtype).to(DEV)
    C = torch.randn(b, N, generator=g).to(dtype).to(DEV)
    z = torch.randn(b, D, generator=g).to(dtype).to(DEV)
    yr, sr = oracle.state_update(state, x, raw, A, B, C, z=z, delta_bias=bias, delta_softplus=True, zoh=True)
    st = state.clone()
    y = ssm.state_update(st, x, raw, A, B, C, z=z, delta_bias=bias, delta_softplus=True, zoh=True)
    torch.cuda.synchronize()
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    check(y, yr, tol, dtype == torch.bfloat16, "y")
    check(st, sr, tol, False, "state")


@pytest.mark.parametrize("case", ["long-segmented", "tiny-dt"])
def test_fwd_zoh_channel_kernel(case, monkeypatch):
    """The zero-order hold on the channel kernel (bf16, N = 16): phi(z) = (e^z - 1) / z from
    the step's own 2^x where |z| >= 1/64, the series below. A long sequence over few channels
    (the segmented schedule) and step sizes tiny enough that every z falls in the series
    branch (some exactly 0), each against the oracle and against the generic kernel."""
    if case == "long-segmented":
        b, L, D, N = 1, 6001, 64, 16
        d = inputs.random_fwd(b, L, D, N, torch.bfloat16, DEV, seed=63)
    else:
        b, L, D, N = 2, 333, 128, 16
        d = inputs.random_fwd(b, L, D, N, torch.bfloat16, DEV, seed=64, delta_softplus=False)
        g = torch.Generator(device="cpu").manual_seed(65)
        dl = torch.rand(b, L, D, generator=g) * 2e-3                    # |dt A| <= 2e-3 * 16 < 1/64
        dl[:, ::7] = 0.0                                                 # and z = 0 exactly
        d["delta"] = dl.to(torch.bfloat16).to(DEV)
        d["delta_bias"] = None
    kw = dict(D=d["D"], z=d["z"], delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"], zoh=True)
    yr, lr = oracle.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], **kw)
    y, last = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], y_dtype=torch.float32,
                                     use_workspace=False, **kw)
    monkeypatch.setenv("SSM_B300_FORWARD_KERNEL", "generic")
    yg, lg = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], y_dtype=torch.float32,
                                    use_workspace=False, **kw)
    monkeypatch.delenv("SSM_B300_FORWARD_KERNEL")
    torch.cuda.synchronize()
    assert ssm.device_error() == 0
    check(y, yr, TOL_BF16, False, "y (channel kernel)")
    check(last, lr, TOL_BF16, False, "last_state (channel kernel)")
    check(yg, yr, TOL_BF16, False, "y (generic kernel)")
