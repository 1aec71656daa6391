"""GPU Mamba-2 SSD forward (chunked, tensor cores) vs the fp64 sequential oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL_BF16, check
from selective_state_space_141_b300 import inputs, ssm

pytestmark = pytest.mark.gpu
DEV = "cuda"


def case(b, L, H, P, N, G, seed):
    return inputs.ssd_inputs(inputs.SsdWorkload("t", b, L, H, P, N, G, seed), DEV)


def gpu(d, h0=None, y_dtype=None, use_workspace=True):
    y, last = ssm.ssd_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], dt_bias=d["dt_bias"],
                          dt_softplus=d["dt_softplus"], h0=h0, y_dtype=y_dtype, use_workspace=use_workspace)
    torch.cuda.synchronize()
    return y, last


def ref(d, h0=None):
    return oracle.ssd_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], dt_bias=d["dt_bias"],
                          dt_softplus=d["dt_softplus"], h0=h0)


@pytest.mark.parametrize("shape", [(2, 200, 3, 128, 128, 1), (1, 130, 4, 64, 64, 2), (2, 64, 2, 64, 128, 1),
                                   (1, 257, 2, 128, 64, 2), (1, 5, 2, 64, 64, 1)])
@pytest.mark.parametrize("schedule", ["chunk-parallel", "sequential"])
def test_ssd_vs_oracle(shape, schedule):
    b, L, H, P, N, G = shape
    d = case(b, L, H, P, N, G, seed=101 + L)
    g = torch.Generator(device="cpu").manual_seed(102)
    h0 = torch.randn(b, H, P, N, generator=g).to(DEV)
    yr, lr = ref(d, h0)
    ws = schedule == "chunk-parallel"
    y32, last = gpu(d, h0, y_dtype=torch.float32, use_workspace=ws)
    check(y32, yr, TOL_BF16, False, "y (fp32 output)")
    check(last, lr, TOL_BF16, False, "last_state")
    y, _ = gpu(d, h0, use_workspace=ws)
    check(y, yr, TOL_BF16, True, "y (bf16)")


def test_ssd_continuation():
    """prefix, then the rest from the prefix's last_state == one pass (within tolerance:
    the chunk boundaries differ)."""
    d = case(2, 300, 3, 128, 128, 1, seed=103)
    y_all, l_all = gpu(d, y_dtype=torch.float32)
    cut = lambda k, sl: d[k][:, sl].contiguous()
    p1 = dict(d, x=cut("x", slice(0, 100)), delta=cut("delta", slice(0, 100)), B=cut("B", slice(0, 100)),
              C=cut("C", slice(0, 100)))
    p2 = dict(d, x=cut("x", slice(100, 300)), delta=cut("delta", slice(100, 300)), B=cut("B", slice(100, 300)),
              C=cut("C", slice(100, 300)))
    y1, mid = gpu(p1, y_dtype=torch.float32)
    y2, l2 = gpu(p2, h0=mid, y_dtype=torch.float32)
    check(torch.cat([y1, y2], dim=1), y_all, TOL_BF16, False, "y")
    check(l2, l_all, TOL_BF16, False, "last_state")


def test_ssd_empty_sequence():
    d = case(2, 0, 3, 64, 64, 1, seed=104)
    h0 = torch.randn(2, 3, 64, 64, device=DEV)
    _, last = gpu(d, h0)
    assert torch.equal(last, h0)


def test_ssd_workload_sampled_heads():
    """The bench's Mamba-2 layer, two sampled (batch, head) pairs vs the oracle, and the
    two schedules against each other over the whole output."""
    w = inputs.SSD_M2
    d = inputs.ssd_inputs(w, DEV)
    y, last = gpu(d, y_dtype=torch.float32)
    y_s, last_s = gpu(d, y_dtype=torch.float32, use_workspace=False)
    check(y, y_s, TOL_BF16, False, "chunk-parallel vs sequential y")
    check(last, last_s, TOL_BF16, False, "chunk-parallel vs sequential last_state")
    for bi, h in ((0, 5), (3, 23)):
        sub = dict(x=d["x"][bi:bi + 1, :, h:h + 1], delta=d["delta"][bi:bi + 1, :, h:h + 1], A=d["A"][h:h + 1],
                   B=d["B"][bi:bi + 1], C=d["C"][bi:bi + 1], D=d["D"][h:h + 1], dt_bias=d["dt_bias"][h:h + 1],
                   dt_softplus=True)
        yr, lr = ref(sub)
        check(y[bi:bi + 1, :, h:h + 1], yr, TOL_BF16, False, f"y b={bi} h={h}")
        check(last[bi:bi + 1, h:h + 1], lr, TOL_BF16, False, f"last_state b={bi} h={h}")


@pytest.mark.parametrize("shape", [(2, 70, 2, 128, 128, 1), (3, 77, 2, 128, 64, 2), (2, 70, 2, 64, 64, 1)])
def test_ssd_ragged_chunk_ignores_next_row(shape):
    """A batch row's last chunk is ragged; its copies reach into the next row (or past the
    tensor). Filling the next row with inf must not change this row's outputs."""
    b, L, H, P, N, G = shape
    d = case(b, L, H, P, N, G, seed=105 + L)
    inf = torch.tensor(float("inf"), dtype=torch.bfloat16, device=DEV)
    for k in ("x", "B", "C", "delta"):
        d[k][1:] = inf
    y, last = gpu(d, y_dtype=torch.float32)
    sub = {k: (v[:1] if k in ("x", "delta", "B", "C") else v) for k, v in d.items()}
    yr, lr = ref(sub)
    check(y[:1], yr, TOL_BF16, False, "y of row 0")
    check(last[:1], lr, TOL_BF16, False, "last_state of row 0")
    assert np.isfinite(y[:1].double().cpu().numpy()).all()
