"""The C-ABI library on a machine without a GPU: it loads, exports every entry point
include/ssm.h declares, and rejects bad arguments on the host before any CUDA call.
Only argument-validation paths run here (fake, never-dereferenced pointers)."""
import ctypes
import os
import re

import pytest

from selective_state_space_141_b300 import ssm
from selective_state_space_141_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return ssm.load_library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "ssm.h")).read()
    return sorted(set(re.findall(r"SSM_API\s+[\w\s\*]+?\b(ssm_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert {"ssm_selective_scan_fwd", "ssm_state_update", "ssm_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in ssm.STATUS.items():
        assert lib.ssm_status_string(code).decode().startswith(name)


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: validation fails before any launch


def T(shape, dtype=ssm.SSM_BF16, addr=None):
    t = ssm.SsmTensor()
    n = 1
    for s in shape:
        n *= s
    global FAKE
    if addr is None:
        addr = FAKE
        FAKE += ((n * 4 + 255) // 256 + 1) * 256
    t.data = addr if n > 0 else None
    t.dtype = dtype
    t.ndim = len(shape)
    for i, s in enumerate(shape):
        t.shape[i] = s
    return t


def fwd_args(b=2, L=5, D=8, N=16, io=ssm.SSM_BF16):
    return dict(u=T((b, L, D), io), delta=T((b, L, D), io), A=T((D, N), ssm.SSM_F32), B=T((b, L, N), io),
                C=T((b, L, N), io), D=T((D,), ssm.SSM_F32), z=T((b, L, D), io), bias=T((D,), ssm.SSM_F32),
                y=T((b, L, D), io), last=T((b, D, N), ssm.SSM_F32))


def call_fwd(lib, a, softplus=1):
    r = lambda k: None if a[k] is None else ctypes.byref(a[k])
    return lib.ssm_selective_scan_fwd(r("u"), r("delta"), r("A"), r("B"), r("C"), r("D"), r("z"), r("bias"),
                                      softplus, r("y"), r("last"), None)


def test_fwd_null(lib):
    for k in ("u", "delta", "A", "B", "C", "y"):
        a = fwd_args()
        a[k] = None
        assert call_fwd(lib, a) == 1, k
    a = fwd_args()
    a["u"].data = None
    assert call_fwd(lib, a) == 1


def test_fwd_shape(lib):
    a = fwd_args()
    a["delta"] = T((2, 5, 9))
    assert call_fwd(lib, a) == 2
    a = fwd_args()
    a["B"] = T((2, 4, 16))
    assert call_fwd(lib, a) == 2
    a = fwd_args()
    a["last"] = T((2, 8, 8), ssm.SSM_F32)
    assert call_fwd(lib, a) == 2
    a = fwd_args()
    a["u"].ndim = 2
    assert call_fwd(lib, a) == 2


def test_fwd_dtype(lib):
    a = fwd_args()
    a["z"].dtype = ssm.SSM_F32
    assert call_fwd(lib, a) == 3
    a = fwd_args()
    a["A"].dtype = ssm.SSM_BF16
    assert call_fwd(lib, a) == 3
    a = fwd_args(io=ssm.SSM_F32)
    a["y"].dtype = ssm.SSM_BF16  # f32 call cannot write bf16 y
    assert call_fwd(lib, a) == 3
    a = fwd_args()
    a["u"].dtype = 7
    assert call_fwd(lib, a) == 3


def test_fwd_layout(lib):
    a = fwd_args()
    a["u"].data = a["u"].data + 1  # not aligned to its 2-byte elements
    assert call_fwd(lib, a) == 4
    a = fwd_args()
    a["y"].data = a["u"].data  # y aliases u
    assert call_fwd(lib, a) == 4
    a = fwd_args()
    a["last"].data = a["z"].data + 16  # last_state overlaps z
    assert call_fwd(lib, a) == 4


def test_fwd_unsupported(lib):
    a = fwd_args(N=5)
    assert call_fwd(lib, a) == 5
    a = fwd_args(N=32)
    assert call_fwd(lib, a) == 5
    assert call_fwd(lib, fwd_args(), softplus=2) == 5


def test_fwd_empty_batch_is_noop(lib):
    assert call_fwd(lib, fwd_args(b=0)) == 0
    assert call_fwd(lib, fwd_args(D=0)) == 0


def dec_args(b=3, D=8, N=16, io=ssm.SSM_BF16):
    return dict(state=T((b, D, N), ssm.SSM_F32), x=T((b, D), io), delta=T((b, D), io), A=T((D, N), ssm.SSM_F32),
                B=T((b, N), io), C=T((b, N), io), D=T((D,), ssm.SSM_F32), z=T((b, D), io), y=T((b, D), io))


def call_dec(lib, a):
    r = lambda k: None if a[k] is None else ctypes.byref(a[k])
    return lib.ssm_state_update(r("state"), r("x"), r("delta"), r("A"), r("B"), r("C"), r("D"), r("z"), r("y"),
                                None)


def test_decode_validation(lib):
    for k in ("state", "x", "delta", "A", "B", "C", "y"):
        a = dec_args()
        a[k] = None
        assert call_dec(lib, a) == 1, k
    a = dec_args()
    a["x"] = T((3, 9))
    assert call_dec(lib, a) == 2
    a = dec_args()
    a["state"].dtype = ssm.SSM_BF16
    assert call_dec(lib, a) == 3
    a = dec_args()
    a["y"].data = a["state"].data
    assert call_dec(lib, a) == 4
    assert call_dec(lib, dec_args(N=12)) == 5
    assert call_dec(lib, dec_args(b=0)) == 0


def test_binding_refuses_noncontiguous():
    import torch
    t = torch.zeros(4, 6)[:, ::2]
    with pytest.raises(ssm.SsmError):
        ssm.describe(t)


def test_workspace_size_validation(lib):
    n = ctypes.c_size_t(123)
    assert lib.ssm_selective_scan_fwd_workspace_size(1, 10, 8, 16, None) == 1
    assert lib.ssm_selective_scan_fwd_workspace_size(-1, 10, 8, 16, ctypes.byref(n)) == 2
    assert lib.ssm_selective_scan_fwd_workspace_size(0, 10, 8, 16, ctypes.byref(n)) == 0 and n.value == 0


def test_fwd_ws_validation(lib):
    a = fwd_args()
    r = lambda k: None if a[k] is None else ctypes.byref(a[k])
    args = [r(k) for k in ("u", "delta", "A", "B", "C", "D", "z", "bias")]
    # bytes > 0 with a NULL workspace; then a misaligned workspace
    assert lib.ssm_selective_scan_fwd_ws(*args, 1, r("y"), r("last"), None, ctypes.c_size_t(64), None) == 1
    assert lib.ssm_selective_scan_fwd_ws(*args, 1, r("y"), r("last"), ctypes.c_void_p(FAKE + 8),
                                         ctypes.c_size_t(64), None) == 4
    # a workspace overlapping u
    assert lib.ssm_selective_scan_fwd_ws(*args, 1, r("y"), r("last"), ctypes.c_void_p(a["u"].data),
                                         ctypes.c_size_t(64), None) == 4


def call_fwd_ex(lib, a, h0, softplus=1, flags=0):
    r = lambda k: None if a[k] is None else ctypes.byref(a[k])
    return lib.ssm_selective_scan_fwd_ex(r("u"), r("delta"), r("A"), r("B"), r("C"), r("D"), r("z"), r("bias"),
                                         softplus, None if h0 is None else ctypes.byref(h0), ctypes.c_uint32(flags),
                                         r("y"), r("last"), None, ctypes.c_size_t(0), None)


def test_fwd_ex_validation(lib):
    a = fwd_args()
    assert call_fwd_ex(lib, a, T((2, 8, 8), ssm.SSM_F32)) == 2          # wrong N
    assert call_fwd_ex(lib, a, T((2, 8, 16), ssm.SSM_BF16)) == 3        # start state must be f32
    h = T((2, 8, 16), ssm.SSM_F32, addr=a["y"].data)                    # overlaps the output y
    assert call_fwd_ex(lib, a, h) == 4
    h = T((2, 8, 16), ssm.SSM_F32, addr=a["last"].data + 16)            # partial overlap with last_state
    assert call_fwd_ex(lib, a, h) == 4
    e = fwd_args(b=0)                                                    # h0 == last_state exactly: allowed
    e["last"] = T((0, 8, 16), ssm.SSM_F32)
    assert call_fwd_ex(lib, e, e["last"]) == 0
    assert call_fwd_ex(lib, fwd_args(), None, softplus=3) == 5
    assert call_fwd_ex(lib, fwd_args(), None, flags=2) == 5             # unknown flag bit
    assert call_fwd_ex(lib, fwd_args(b=0), None, flags=ssm.SSM_FWD_ZOH) == 0


def call_dec_ex(lib, a, bias, softplus, flags=0):
    r = lambda k: None if a[k] is None else ctypes.byref(a[k])
    return lib.ssm_state_update_ex(r("state"), r("x"), r("delta"), r("A"), r("B"), r("C"), r("D"), r("z"),
                                   None if bias is None else ctypes.byref(bias), softplus, ctypes.c_uint32(flags),
                                   r("y"), None)


def test_decode_ex_validation(lib):
    a = dec_args()
    assert call_dec_ex(lib, a, T((9,), ssm.SSM_F32), 1) == 2            # bias is (D)
    assert call_dec_ex(lib, a, T((8,), ssm.SSM_BF16), 1) == 3           # bias must be f32
    assert call_dec_ex(lib, a, T((8,), ssm.SSM_F32, addr=a["y"].data), 1) == 4
    assert call_dec_ex(lib, a, None, 2) == 5
    assert call_dec_ex(lib, dec_args(b=0), T((8,), ssm.SSM_F32), 1) == 0
    assert call_dec_ex(lib, dec_args(), None, 0, flags=4) == 5


def call_conv_fwd(lib, a, w, cb, cs, softplus=1):
    r = lambda k: None if a[k] is None else ctypes.byref(a[k])
    o = lambda t: None if t is None else ctypes.byref(t)
    return lib.ssm_conv_selective_scan_fwd(r("u"), o(w), o(cb), o(cs), r("delta"), r("A"), r("B"), r("C"), r("D"),
                                           r("z"), r("bias"), softplus, None, ctypes.c_uint32(0), r("y"), r("last"),
                                           None, ctypes.c_size_t(0), None)


def test_conv_fwd_validation(lib):
    a = fwd_args()  # batch 2, L 5, D 8, bf16
    w, cb, cs = T((8, 4), ssm.SSM_F32), T((8,), ssm.SSM_F32), T((2, 8, 3))
    assert call_conv_fwd(lib, a, None, cb, cs) == 1                          # weights are required
    assert call_conv_fwd(lib, a, T((8, 3), ssm.SSM_F32), cb, cs) == 2       # width must be 4
    assert call_conv_fwd(lib, a, w, T((9,), ssm.SSM_F32), cs) == 2
    assert call_conv_fwd(lib, a, w, cb, T((2, 8, 4))) == 2                  # state holds 3 inputs
    assert call_conv_fwd(lib, a, T((8, 4), ssm.SSM_BF16), cb, cs) == 3      # weights are f32
    assert call_conv_fwd(lib, a, w, cb, T((2, 8, 3), ssm.SSM_F32)) == 3     # state has the I/O type
    assert call_conv_fwd(lib, a, w, cb, T((2, 8, 3), addr=a["y"].data)) == 4   # state overlaps y
    assert call_conv_fwd(lib, a, w, cb, T((2, 8, 3), addr=a["u"].data)) == 4   # state overlaps x
    assert call_conv_fwd(lib, fwd_args(b=0), w, cb, T((0, 8, 3))) == 0


def test_conv_decode_validation(lib):
    a = dec_args()  # batch 3, D 8, bf16
    w, cs = T((8, 4), ssm.SSM_F32), T((3, 8, 3))
    r = lambda k: ctypes.byref(a[k])
    call = lambda cs_, w_: lib.ssm_conv_state_update(None if cs_ is None else ctypes.byref(cs_), r("state"), r("x"),
                                                     None if w_ is None else ctypes.byref(w_), None, r("delta"),
                                                     r("A"), r("B"), r("C"), r("D"), r("z"), None, 1,
                                                     ctypes.c_uint32(0), r("y"), None)
    assert call(None, w) == 1
    assert call(cs, None) == 1
    assert call(T((3, 8, 2)), w) == 2
    assert call(cs, T((8, 5), ssm.SSM_F32)) == 2
    assert call(T((3, 8, 3), addr=a["state"].data), w) == 4


def bwd_args(b=2, L=5, D=8, N=16, io=ssm.SSM_BF16, gt=None):
    gt = io if gt is None else gt
    a = fwd_args(b, L, D, N, io)
    a.update(dy=T((b, L, D), gt), du=T((b, L, D), gt), ddelta=T((b, L, D), gt), dA=T((D, N), ssm.SSM_F32),
             dB=T((b, L, N), gt), dC=T((b, L, N), gt), dD=T((D,), ssm.SSM_F32), dz=T((b, L, D), gt),
             dbias=T((D,), ssm.SSM_F32), ws=T((1 << 16,), ssm.SSM_F32))
    return a


def call_bwd(lib, a, ws_bytes=None, ws_addr=None):
    r = lambda k: None if a[k] is None else ctypes.byref(a[k])
    n = ctypes.c_size_t(0)
    assert lib.ssm_selective_scan_bwd_workspace_size(a["u"].shape[0], a["u"].shape[1], a["u"].shape[2],
                                                      a["A"].shape[1], ctypes.byref(n)) == 0
    wb = n.value if ws_bytes is None else ws_bytes
    wa = ((a["ws"].data + 255) // 256 * 256) if ws_addr is None else ws_addr
    return lib.ssm_selective_scan_bwd(r("u"), r("delta"), r("A"), r("B"), r("C"), r("D"), r("z"), r("bias"), 1, None,
                                      r("dy"), None, r("du"), r("ddelta"), r("dA"), r("dB"), r("dC"), r("dD"), r("dz"),
                                      r("dbias"), None, ctypes.c_void_p(wa), ctypes.c_size_t(wb), None)


def test_bwd_validation(lib):
    for k in ("dD", "dz", "dbias"):        # a gradient output for each optional input given
        a = bwd_args()
        a[k] = None
        assert call_bwd(lib, a) == 1, k
    a = bwd_args()
    a["D"] = None                           # and none for an absent one
    assert call_bwd(lib, a) == 1
    a = bwd_args()
    assert call_bwd(lib, a, ws_addr=0, ws_bytes=1024) == 1           # no workspace
    assert call_bwd(lib, a, ws_bytes=16) == 2                         # too small
    assert call_bwd(lib, a, ws_addr=a["ws"].data + 256 + 16) == 4     # not 256-byte aligned
    a = bwd_args()
    a["du"].dtype = ssm.SSM_F32                                       # gradient types must agree with dy
    assert call_bwd(lib, a) == 3
    a = bwd_args()
    a["dA"].dtype = ssm.SSM_BF16
    assert call_bwd(lib, a) == 3
    a = bwd_args()
    a["du"] = T((2, 5, 8), addr=a["u"].data)                          # an output over an input
    assert call_bwd(lib, a) == 4
    a = bwd_args()
    a["dC"] = T((2, 5, 16), addr=a["dB"].data)                        # two outputs overlapping
    assert call_bwd(lib, a) == 4
    a = bwd_args()
    a["dB"] = T((2, 5, 8))
    assert call_bwd(lib, a) == 2


def test_ssd_validation(lib):
    b, L, H, P, N, G = 2, 5, 4, 64, 64, 2
    x, dl, A = T((b, L, H * P)), T((b, L, H)), T((H,), ssm.SSM_F32)
    Bm, Cm, y = T((b, L, G * N)), T((b, L, G * N)), T((b, L, H * P))
    call = lambda g, x_=x, A_=A, B_=Bm, C_=Cm, y_=y, sp=1: lib.ssm_ssd_fwd(
        ctypes.c_int64(g), ctypes.byref(x_), ctypes.byref(dl), ctypes.byref(A_), ctypes.byref(B_), ctypes.byref(C_),
        None, None, sp, None, ctypes.byref(y_), None, None, ctypes.c_size_t(0), None)
    assert call(3) == 2                                              # groups must divide H
    assert call(G, A_=T((3,), ssm.SSM_F32)) == 2                     # H must divide H*P
    assert call(G, B_=T((b, L, G * 32)), C_=T((b, L, G * 32))) == 5  # N = 32 is not supported
    assert call(G, x_=T((b, L, H * P), ssm.SSM_F32)) == 3            # bf16 inputs
    assert call(G, y_=T((b, L, H * P), addr=x.data)) == 4            # y over x
    assert call(G, x_=T((b, L, H * P), addr=x.data + 2)) == 4        # x not 16-byte aligned
    assert call(G, sp=2) == 5
    n = ctypes.c_size_t(0)
    assert lib.ssm_ssd_fwd_workspace_size(2, 100, 4, 2, 64, 64, ctypes.byref(n)) == 0
    # per (b, c, h): entering state (bf16 P x N) + dt, cs (64 floats each); per (b, c, g): C B^T
    items, cbs = 2 * 2 * 4, 2 * 2 * 2
    r256 = lambda v: (v + 255) // 256 * 256
    assert n.value == r256(items * 64 * 64 * 2) + 2 * r256(items * 64 * 4) + r256(cbs * 64 * 72 * 4)
    assert lib.ssm_ssd_fwd_workspace_size(2, 100, 4, 0, 64, 64, ctypes.byref(n)) == 2
    assert lib.ssm_ssd_fwd_workspace_size(2, 100, 4, 2, 64, 64, None) == 1


def call_fwd_train(lib, a, ws_addr, ws_bytes, with_flag=True):
    r = lambda k: None if a[k] is None else ctypes.byref(a[k])
    written = ctypes.c_int32(7)
    st = lib.ssm_selective_scan_fwd_train(r("u"), r("delta"), r("A"), r("B"), r("C"), r("D"), r("z"), r("bias"), 1,
                                          None, r("y"), r("last"), ctypes.c_void_p(ws_addr), ctypes.c_size_t(ws_bytes),
                                          ctypes.byref(written) if with_flag else None, None)
    return st, written.value


def test_fwd_train_validation(lib):
    """ssm_selective_scan_fwd_train: the checkpoints_written out-pointer and the backward
    workspace are checked before anything runs; the flag reads 0 on every error."""
    a = fwd_args()
    ws = T((1 << 16,), ssm.SSM_F32)
    n = ctypes.c_size_t(0)
    assert lib.ssm_selective_scan_bwd_workspace_size(2, 5, 8, 16, ctypes.byref(n)) == 0
    wa = (ws.data + 255) // 256 * 256
    assert call_fwd_train(lib, a, wa, n.value, with_flag=False)[0] == 1   # no out-pointer
    assert call_fwd_train(lib, a, 0, n.value) == (1, 0)                    # no workspace
    assert call_fwd_train(lib, a, wa + 16, n.value) == (4, 0)              # not 256-byte aligned
    assert call_fwd_train(lib, a, wa, 16) == (2, 0)                        # too small
    assert call_fwd_train(lib, a, a["u"].data, n.value) == (4, 0)          # over an input
    b = fwd_args()
    b["y"].dtype = 99                                                      # the forward pass's own checks follow
    assert call_fwd_train(lib, b, wa, n.value) == (3, 0)


def test_bwd_ex_flags(lib):
    """ssm_selective_scan_bwd_ex: only SSM_BWD_CHECKPOINTS is a known flag."""
    a = bwd_args()
    r = lambda k: None if a[k] is None else ctypes.byref(a[k])
    n = ctypes.c_size_t(0)
    assert lib.ssm_selective_scan_bwd_workspace_size(2, 5, 8, 16, ctypes.byref(n)) == 0
    wa = (a["ws"].data + 255) // 256 * 256
    call = lambda flags: lib.ssm_selective_scan_bwd_ex(
        r("u"), r("delta"), r("A"), r("B"), r("C"), r("D"), r("z"), r("bias"), 1, None, r("dy"), None, r("du"),
        r("ddelta"), r("dA"), r("dB"), r("dC"), r("dD"), r("dz"), r("dbias"), None, ctypes.c_uint32(flags),
        ctypes.c_void_p(wa), ctypes.c_size_t(n.value), None)
    assert call(2) == 5
    assert call(ssm.SSM_BWD_CHECKPOINTS | 4) == 5
    a["dD"] = None                                                         # the usual checks with the flag set
    assert call(ssm.SSM_BWD_CHECKPOINTS) == 1
