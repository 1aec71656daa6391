"""GPU backward pass vs the fp64 oracle's backward (itself pinned to finite differences
of the forward pass), called through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL_BF16, TOL_F32, check
from selective_state_space_141_b300 import inputs, ssm

pytestmark = pytest.mark.gpu
DEV = "cuda"


def case(b, L, D, N, dtype, seed, full=True, softplus=True):
    d = inputs.random_fwd(b, L, D, N, dtype, DEV, seed=seed, has_bias=full, has_D=full, has_z=full,
                          delta_softplus=softplus)
    g = torch.Generator(device="cpu").manual_seed(seed + 500)
    if not softplus:
        d["delta"] = (torch.rand(b, L, D, generator=g) * 0.5 + 0.01).to(dtype).to(DEV)
    d["h0"] = torch.randn(b, D, N, generator=g).to(DEV) if full else None
    d["dlast"] = torch.randn(b, D, N, generator=g).to(DEV) if full else None
    d["dy"] = torch.randn(b, L, D, generator=g).to(DEV)
    return d


def run(d, grad_dtype, want_dh0=True):
    g = ssm.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["dy"].to(grad_dtype), D=d["D"], z=d["z"],
                               delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"], h0=d["h0"],
                               dlast=d["dlast"], want_dh0=want_dh0)
    torch.cuda.synchronize()
    return g


def ref(d, grad_dtype):
    return oracle.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["dy"].to(grad_dtype), D=d["D"],
                                     z=d["z"], delta_bias=d["delta_bias"], delta_softplus=d["delta_softplus"],
                                     h0=d["h0"] if d["h0"] is not None else np.zeros((d["u"].shape[0],
                                                                                      d["u"].shape[2],
                                                                                      d["A"].shape[1])),
                                     dlast=d["dlast"])


# (2, 77, 104, 16): rows 16-byte aligned, so whole chunks of whole channel blocks take the
# unclamped staging while the last chunk (13 steps) and the last warp (8 channels) take the
# clamped one; (2, 77, 100, 16): rows not aligned, every chunk staged with plain loads
@pytest.mark.parametrize("shape", [(2, 77, 100, 16), (2, 77, 104, 16), (3, 45, 64, 8), (1, 33, 40, 4), (2, 16, 32, 16)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("full", [True, False], ids=["all-inputs", "bare"])
def test_bwd_vs_oracle(shape, dtype, full):
    b, L, D, N = shape
    d = case(b, L, D, N, dtype, seed=81 + L, full=full, softplus=full)
    r = ref(d, torch.float32)
    g = run(d, torch.float32)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    for k, v in r.items():
        check(g[k], v, tol, False, k)
    if dtype == torch.bfloat16:  # bf16 gradients: the same values rounded once
        gb = run(d, torch.bfloat16)
        rb = ref(d, torch.bfloat16)
        for k in ("du", "ddelta", "dB", "dC") + (("dz",) if full else ()):
            check(gb[k], rb[k], TOL_BF16, True, k + " (bf16)")


def test_bwd_medium_shape():
    """Several chunks, warps and a ragged tail, every gradient against the oracle."""
    d = case(2, 333, 200, 16, torch.bfloat16, seed=91)
    r = ref(d, torch.float32)
    g = run(d, torch.float32)
    for k, v in r.items():
        check(g[k], v, TOL_BF16, False, k)


def test_bwd_is_deterministic():
    d = case(2, 100, 256, 16, torch.bfloat16, seed=92)
    g1, g2 = run(d, torch.float32), run(d, torch.float32)
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


def test_bwd_empty_sequence():
    d = case(2, 0, 64, 16, torch.bfloat16, seed=93)
    g = run(d, torch.float32)
    assert torch.count_nonzero(g["dA"]) == 0 and torch.count_nonzero(g["dD"]) == 0
    assert torch.equal(g["dh0"], d["dlast"])


def test_bwd_layer_workload_sampled():
    """The Mamba-1.4B layer (4 x 4096 x 4096, N = 16) in the bench's launch configuration
    (bf16 dy and gradients, caller workspace): the per-channel gradients (du, ddelta, dz,
    dA, dD, dbias) of sampled channels against the oracle run on those channels alone.
    (dB and dC sum over every channel; the smaller shapes above check them whole.)"""
    w = inputs.FWD_WORKLOADS["m1p4b"]
    d = inputs.fwd_inputs(w, DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    dy = torch.randn(d["u"].shape, generator=g, device=DEV).to(d["u"].dtype)
    wsp = torch.empty(ssm.bwd_workspace_size(w.batch, w.L, w.D, w.N), dtype=torch.uint8, device=DEV)
    gr = ssm.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy, D=d["D"], z=d["z"],
                                delta_bias=d["delta_bias"], delta_softplus=True, workspace=wsp)
    torch.cuda.synchronize()
    assert ssm.device_error() == 0
    rng = np.random.default_rng(94)
    ds = np.unique(np.concatenate([[0, 15, 16, w.D - 1], rng.choice(w.D, size=8, replace=False)]))
    idx = torch.as_tensor(ds, device=DEV)
    pick = lambda t: t.index_select(-1, idx)
    r = oracle.selective_scan_bwd(pick(d["u"]), pick(d["delta"]), d["A"].index_select(0, idx), d["B"], d["C"],
                                  pick(dy), D=d["D"].index_select(0, idx), z=pick(d["z"]),
                                  delta_bias=d["delta_bias"].index_select(0, idx), delta_softplus=True,
                                  h0=np.zeros((w.batch, len(ds), w.N)))
    for k in ("du", "ddelta", "dz"):
        check(pick(gr[k]), r[k], TOL_BF16, True, k)
    check(gr["dA"].index_select(0, idx), r["dA"], TOL_BF16, False, "dA")
    for k in ("dD", "dbias"):
        check(gr[k].index_select(0, idx), r[k], TOL_BF16, False, k)


@pytest.mark.parametrize("shape", [(2, 333, 200, 16), (3, 45, 64, 8), (2, 77, 100, 16), (1, 40, 48, 4)])
def test_fwd_train_checkpoints_feed_bwd(shape):
    """ssm_selective_scan_fwd_train: y and last_state bit for bit those of the forward pass
    with the same h0; it writes the checkpoints exactly where the channel kernel runs (bf16,
    N = 8 or 16, D % 8 == 0), and the backward pass given them (SSM_BWD_CHECKPOINTS) returns
    the same gradients, bit for bit, as the backward pass that makes its own."""
    b, L, Dm, N = shape
    d = case(b, L, Dm, N, torch.bfloat16, seed=97 + L)
    ws = torch.empty(ssm.bwd_workspace_size(b, L, Dm, N), dtype=torch.uint8, device=DEV)
    kw = dict(D=d["D"], z=d["z"], delta_bias=d["delta_bias"], delta_softplus=True, h0=d["h0"])
    y, last, written = ssm.selective_scan_fwd_train(d["u"], d["delta"], d["A"], d["B"], d["C"], ws, **kw)
    y0, last0 = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], use_workspace=False, **kw)
    torch.cuda.synchronize()
    assert torch.equal(y, y0) and torch.equal(last, last0)
    assert written == (N in (8, 16) and Dm % 8 == 0)
    g_own = run(d, torch.float32)
    g_ck = ssm.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["dy"].to(torch.float32), D=d["D"],
                                  z=d["z"], delta_bias=d["delta_bias"], delta_softplus=True, h0=d["h0"],
                                  dlast=d["dlast"], want_dh0=True, workspace=ws, checkpoints_ready=written)
    torch.cuda.synchronize()
    for k in g_own:
        assert torch.equal(g_own[k], g_ck[k]), k


def test_fwd_train_checkpoints_on_the_segmented_schedule():
    """A long sequence over few channels runs the forward pass as segments (carries kept in
    y). Each segment's full pass starts from the carried state, which equals the sequential
    one up to rounding (the carry scan reassociates the recurrence), so its checkpoints do
    too: the backward pass given them agrees with the one that makes its own to rounding,
    and both match the oracle."""
    b, L, Dm, N = 1, 12001, 64, 16
    d = case(b, L, Dm, N, torch.bfloat16, seed=98)
    ws = torch.empty(ssm.bwd_workspace_size(b, L, Dm, N), dtype=torch.uint8, device=DEV)
    kw = dict(D=d["D"], z=d["z"], delta_bias=d["delta_bias"], delta_softplus=True, h0=d["h0"])
    y, last, written = ssm.selective_scan_fwd_train(d["u"], d["delta"], d["A"], d["B"], d["C"], ws, **kw)
    assert written
    g_own = run(d, torch.float32)
    g_ck = ssm.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["dy"].to(torch.float32), D=d["D"],
                                  z=d["z"], delta_bias=d["delta_bias"], delta_softplus=True, h0=d["h0"],
                                  dlast=d["dlast"], want_dh0=True, workspace=ws, checkpoints_ready=True)
    torch.cuda.synchronize()
    # the segmented forward's states differ from the sequential ones by ~2e-4 of their rms
    # (the long-sequence bench line's oracle check); dA, a sum over all 12001 steps, shows
    # ~2.3e-4: 1e-3 bounds that rounding, well inside the bf16 tolerance checked below
    for k in g_own:
        diff = (g_own[k].double() - g_ck[k].double()).abs().max().item()
        rms = g_own[k].double().pow(2).mean().sqrt().item()
        assert diff <= 1e-3 * max(rms, 1e-30), (k, diff, rms)
    r = ref(d, torch.float32)
    for k, v in r.items():
        check(g_ck[k], v, TOL_BF16, False, k + " (segmented forward's checkpoints)")
