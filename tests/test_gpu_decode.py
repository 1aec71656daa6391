"""GPU decode step vs the fp64 oracle, and the decode/forward cross-checks."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL_BF16, TOL_F32, check, to64
from selective_state_space_141_b300 import inputs, ssm

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("N", [4, 8, 16])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_random(N, dtype):
    w = inputs.DecodeWorkload("t", 3, 70, N, 5, dtype, 21)
    d = inputs.decode_inputs(w, DEV)
    g = torch.Generator(device="cpu").manual_seed(22)
    state = torch.randn(3, 70, N, generator=g).to(DEV)  # start from a random state
    st_ref = to64(state)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    for t in range(w.steps):
        args = (d["x"][t], d["delta"][t], d["A"], d["B"][t], d["C"][t])
        yr, st_ref = oracle.state_update(st_ref, *args, D=d["D"], z=d["z"][t])
        y = ssm.state_update(state, *args, D=d["D"], z=d["z"][t])
        torch.cuda.synchronize()
        check(y, yr, tol, dtype == torch.bfloat16, f"y step {t}")
        check(state, st_ref, tol, False, f"state step {t}")


def test_decode_workload_sampled():
    """The 2.8B-shaped decode workload, 1024 steps, sampled channels vs the oracle."""
    w = inputs.DECODE
    d = inputs.decode_inputs(w, DEV)
    state = d["state"]
    rng = np.random.default_rng(31)
    rows = sorted(rng.choice(w.batch, size=4, replace=False).tolist())
    picks = {b: np.sort(rng.choice(w.D, size=64, replace=False)) for b in rows}  # 256 channels
    ref_state = {b: np.zeros((1, 64, w.N)) for b in rows}
    ys = []
    for t in range(w.steps):
        y = ssm.state_update(state, d["x"][t], d["delta"][t], d["A"], d["B"][t], d["C"][t], D=d["D"], z=d["z"][t])
        ys.append({b: y[b, torch.as_tensor(picks[b], device=DEV)] for b in rows})
    torch.cuda.synchronize()
    for b in rows:
        ds = torch.as_tensor(picks[b], device=DEV)
        A, Dk = d["A"].index_select(0, ds), d["D"].index_select(0, ds)
        x = to64(d["x"][:, b].index_select(1, ds))
        dl = to64(d["delta"][:, b].index_select(1, ds))
        z = to64(d["z"][:, b].index_select(1, ds))
        Bm, Cm = to64(d["B"][:, b]), to64(d["C"][:, b])
        st = ref_state[b]
        for t in range(w.steps):
            yr, st = oracle.state_update(st, x[t][None], dl[t][None], A, Bm[t][None], Cm[t][None], D=Dk, z=z[t][None])
            check(ys[t][b], yr[0], TOL_BF16, True, f"y b={b} t={t}")
        check(state[b].index_select(0, ds), st[0], TOL_BF16, False, f"state b={b}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_unaligned_B_C(dtype):
    """B and C at an element offset that is not 16-byte aligned take the scalar loads."""
    N = 16
    w = inputs.DecodeWorkload("t", 3, 96, N, 1, dtype, 23)
    d = inputs.decode_inputs(w, DEV)
    Bbuf = torch.empty(3 * N + 1, dtype=dtype, device=DEV)
    Cbuf = torch.empty(3 * N + 1, dtype=dtype, device=DEV)
    B = Bbuf[1:].view(3, N)
    C = Cbuf[1:].view(3, N)
    B.copy_(d["B"][0])
    C.copy_(d["C"][0])
    assert B.data_ptr() % 16 != 0
    state = torch.randn(3, 96, N, generator=torch.Generator().manual_seed(24)).to(DEV)
    st_ref = to64(state)
    yr, st_ref = oracle.state_update(st_ref, d["x"][0], d["delta"][0], d["A"], B, C, D=d["D"], z=d["z"][0])
    y = ssm.state_update(state, d["x"][0], d["delta"][0], d["A"], B, C, D=d["D"], z=d["z"][0])
    torch.cuda.synchronize()
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    check(y, yr, tol, dtype == torch.bfloat16, "y")
    check(state, st_ref, tol, False, "state")


def test_decode_delta_zero_keeps_state_bitwise():
    w = inputs.DecodeWorkload("t", 2, 64, 16, 1, torch.bfloat16, 5)
    d = inputs.decode_inputs(w, DEV)
    state = torch.randn(2, 64, 16, device=DEV)
    before = state.clone()
    ssm.state_update(state, d["x"][0], torch.zeros_like(d["delta"][0]), d["A"], d["B"][0], d["C"][0], D=d["D"],
                     z=d["z"][0])
    torch.cuda.synchronize()
    assert torch.equal(state, before)


def test_decode_iterated_equals_forward():
    """T decode steps from zero == one forward pass over the T steps (no softplus)."""
    b, T, D, N = 2, 40, 96, 16
    d = inputs.random_fwd(b, T, D, N, dtype=torch.bfloat16, device=DEV, seed=9, has_bias=False,
                          delta_softplus=False)
    d["delta"] = (d["delta"].float().abs() * 0.05).to(torch.bfloat16)
    y_f, last_f = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                         delta_softplus=False, y_dtype=torch.float32)
    state = torch.zeros(b, D, N, device=DEV)
    ys = []
    for t in range(T):
        ys.append(ssm.state_update(state, d["u"][:, t].contiguous(), d["delta"][:, t].contiguous(), d["A"],
                                   d["B"][:, t].contiguous(), d["C"][:, t].contiguous(), D=d["D"],
                                   z=d["z"][:, t].contiguous(), y_dtype=torch.float32))
    torch.cuda.synchronize()
    y_d = torch.stack(ys, 1)
    # bf16 inputs: the two kernels may use different fast SFU forms, so they agree to
    # the bf16 tolerance, and each matches the oracle.
    yr, sr = oracle.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                       delta_softplus=False)
    check(y_d, y_f, TOL_BF16, False, "decode vs forward y")
    check(state, last_f, TOL_BF16, False, "decode vs forward state")
    check(y_d, yr, TOL_BF16, False, "decode vs oracle y")
    check(y_f, yr, TOL_BF16, False, "forward vs oracle y")
    check(state, sr, TOL_BF16, False, "decode vs oracle state")


def test_prefix_state_then_decode():
    """forward(prefix).last_state continued by decode == forward(prefix + suffix)."""
    b, T, P, D, N = 2, 48, 30, 64, 16
    d = inputs.random_fwd(b, T, D, N, dtype=torch.float32, device=DEV, seed=10, has_bias=False,
                          delta_softplus=False)
    d["delta"] = d["delta"].abs() * 0.05
    y_all, _ = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                      delta_softplus=False)
    _, mid = ssm.selective_scan_fwd(d["u"][:, :P].contiguous(), d["delta"][:, :P].contiguous(), d["A"],
                                    d["B"][:, :P].contiguous(), d["C"][:, :P].contiguous(), D=d["D"],
                                    z=d["z"][:, :P].contiguous(), delta_softplus=False)
    for t in range(P, T):
        y = ssm.state_update(mid, d["u"][:, t].contiguous(), d["delta"][:, t].contiguous(), d["A"],
                             d["B"][:, t].contiguous(), d["C"][:, t].contiguous(), D=d["D"],
                             z=d["z"][:, t].contiguous())
        check(y, y_all[:, t], TOL_F32, False, f"y t={t}")
    torch.cuda.synchronize()


@pytest.mark.parametrize("step_map", [False, True], ids=["dt", "softplus-bias"])
@pytest.mark.parametrize("gate", [True, False], ids=["z-D", "bare"])
@pytest.mark.parametrize("y_dtype", [torch.bfloat16, torch.float32], ids=["y-bf16", "y-f32"])
def test_decode_streamed_kernel(gate, y_dtype, step_map, monkeypatch):
    """The streamed decode kernel (bf16, N = 16, D a multiple of its 128-channel tile)
    against the oracle over several steps, and bit for bit against the one-thread-per-8-
    states kernel (SSM_B300_DECODE=plain) on the same inputs."""
    b, Dm, N = 5, 256, 16
    w = inputs.DecodeWorkload("t", b, Dm, N, 4, torch.bfloat16, 41)
    d = inputs.decode_inputs(w, DEV)
    g = torch.Generator(device="cpu").manual_seed(42)
    s0 = torch.randn(b, Dm, N, generator=g).to(DEV)
    bias = (torch.rand(Dm, generator=g) * 2 - 3).to(DEV) if step_map else None  # softplus(delta + bias)
    mp = dict(delta_bias=bias, delta_softplus=True) if step_map else {}
    kw = lambda t: dict(D=d["D"] if gate else None, z=d["z"][t] if gate else None, y_dtype=y_dtype, **mp)
    runs = {}
    for mode in ("stream", "plain"):
        if mode == "plain":
            monkeypatch.setenv("SSM_B300_DECODE", "plain")
        state = s0.clone()
        ys = [ssm.state_update(state, d["x"][t], d["delta"][t], d["A"], d["B"][t], d["C"][t], **kw(t))
              for t in range(w.steps)]
        torch.cuda.synchronize()
        runs[mode] = (ys, state)
    monkeypatch.delenv("SSM_B300_DECODE")
    for t in range(w.steps):
        assert torch.equal(runs["stream"][0][t], runs["plain"][0][t]), t
    assert torch.equal(runs["stream"][1], runs["plain"][1])
    st_ref = to64(s0)
    for t in range(w.steps):
        args = (d["x"][t], d["delta"][t], d["A"], d["B"][t], d["C"][t])
        yr, st_ref = oracle.state_update(st_ref, *args, D=d["D"] if gate else None, z=d["z"][t] if gate else None,
                                         **mp)
        check(runs["stream"][0][t], yr, TOL_BF16, y_dtype == torch.bfloat16, f"y step {t}")
    check(runs["stream"][1], st_ref, TOL_BF16, False, "state")
