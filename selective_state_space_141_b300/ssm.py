"""ctypes binding over libssm_b300.so (the C ABI in include/ssm.h).

Argument marshalling only: torch tensors become ssm_tensor_t descriptors (device
pointer, element type, shape) and the current torch stream is passed through. Every
step of the computation runs in the library's CUDA kernels. There is no fallback: if
the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssm_b300.so")

SSM_F32, SSM_BF16 = 0, 1
SSM_FWD_ZOH = 1  # flag of the extended entry points (include/ssm.h)
SSM_BWD_CHECKPOINTS = 1  # the backward workspace holds the training forward's checkpoints
_BAD_DTYPE = 99  # forwarded for any other torch dtype so the library reports SSM_ERR_DTYPE
_DTYPES = {torch.float32: SSM_F32, torch.bfloat16: SSM_BF16}

STATUS = {0: "SSM_OK", 1: "SSM_ERR_NULL", 2: "SSM_ERR_SHAPE", 3: "SSM_ERR_DTYPE", 4: "SSM_ERR_LAYOUT",
          5: "SSM_ERR_UNSUPPORTED", 6: "SSM_ERR_CUDA", 7: "SSM_ERR_DEVICE_TIMEOUT"}


class SsmTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 3)]


class SsmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


_lib = None
_P = ctypes.POINTER(SsmTensor)


def library_path() -> str:
    return LIB_PATH


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle of the CUDA library."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise SsmError(6, f"CUDA library not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    lib.ssm_selective_scan_fwd.restype = ctypes.c_int
    lib.ssm_selective_scan_fwd.argtypes = [_P] * 8 + [ctypes.c_int, _P, _P, ctypes.c_void_p]
    lib.ssm_selective_scan_fwd_ws.restype = ctypes.c_int
    lib.ssm_selective_scan_fwd_ws.argtypes = [_P] * 8 + [ctypes.c_int, _P, _P, ctypes.c_void_p, ctypes.c_size_t,
                                                          ctypes.c_void_p]
    lib.ssm_selective_scan_fwd_workspace_size.restype = ctypes.c_int
    lib.ssm_selective_scan_fwd_workspace_size.argtypes = [ctypes.c_int64] * 4 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.ssm_selective_scan_fwd_ex.restype = ctypes.c_int
    lib.ssm_selective_scan_fwd_ex.argtypes = [_P] * 8 + [ctypes.c_int, _P, ctypes.c_uint32, _P, _P, ctypes.c_void_p,
                                                          ctypes.c_size_t, ctypes.c_void_p]
    lib.ssm_state_update.restype = ctypes.c_int
    lib.ssm_state_update.argtypes = [_P] * 9 + [ctypes.c_void_p]
    lib.ssm_conv_selective_scan_fwd.restype = ctypes.c_int
    lib.ssm_conv_selective_scan_fwd.argtypes = [_P] * 11 + [ctypes.c_int, _P, ctypes.c_uint32, _P, _P, ctypes.c_void_p,
                                                            ctypes.c_size_t, ctypes.c_void_p]
    lib.ssm_conv_state_update.restype = ctypes.c_int
    lib.ssm_conv_state_update.argtypes = [_P] * 12 + [ctypes.c_int, ctypes.c_uint32, _P, ctypes.c_void_p]
    lib.ssm_selective_scan_bwd.restype = ctypes.c_int
    lib.ssm_selective_scan_bwd.argtypes = [_P] * 8 + [ctypes.c_int] + [_P] * 12 + [ctypes.c_void_p, ctypes.c_size_t,
                                                                                ctypes.c_void_p]
    lib.ssm_selective_scan_bwd_ex.restype = ctypes.c_int
    lib.ssm_selective_scan_bwd_ex.argtypes = [_P] * 8 + [ctypes.c_int] + [_P] * 12 + [ctypes.c_uint32, ctypes.c_void_p,
                                                                                   ctypes.c_size_t, ctypes.c_void_p]
    lib.ssm_selective_scan_fwd_train.restype = ctypes.c_int
    lib.ssm_selective_scan_fwd_train.argtypes = [_P] * 8 + [ctypes.c_int, _P, _P, _P, ctypes.c_void_p, ctypes.c_size_t,
                                                             ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]
    lib.ssm_selective_scan_bwd_workspace_size.restype = ctypes.c_int
    lib.ssm_selective_scan_bwd_workspace_size.argtypes = [ctypes.c_int64] * 4 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.ssm_ssd_fwd.restype = ctypes.c_int
    lib.ssm_ssd_fwd.argtypes = [ctypes.c_int64] + [_P] * 7 + [ctypes.c_int, _P, _P, _P, ctypes.c_void_p,
                                                              ctypes.c_size_t, ctypes.c_void_p]
    lib.ssm_ssd_fwd_workspace_size.restype = ctypes.c_int
    lib.ssm_ssd_fwd_workspace_size.argtypes = [ctypes.c_int64] * 6 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.ssm_state_update_ex.restype = ctypes.c_int
    lib.ssm_state_update_ex.argtypes = [_P] * 9 + [ctypes.c_int, ctypes.c_uint32, _P, ctypes.c_void_p]
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_status_string.argtypes = [ctypes.c_int]
    lib.ssm_device_error.restype = ctypes.c_int
    lib.ssm_device_error.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    _lib = lib
    return lib


def describe(t: torch.Tensor | None):
    """ssm_tensor_t for a dense tensor (None -> NULL). Non-contiguous tensors are refused
    here because the descriptor carries no strides."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise SsmError(4, "tensor is not contiguous")
    if t.dim() > 3:
        raise SsmError(2, "tensor has more than 3 dimensions")
    d = SsmTensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _DTYPES.get(t.dtype, _BAD_DTYPE)
    d.ndim = t.dim()
    for i, s in enumerate(t.shape):
        d.shape[i] = s
    return d


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def workspace_size(batch, L, D, N) -> int:
    """Bytes of workspace ``ssm_selective_scan_fwd_ws`` can use for this shape (0: none)."""
    lib = load_library()
    n = ctypes.c_size_t(0)
    st = lib.ssm_selective_scan_fwd_workspace_size(int(batch), int(L), int(D), int(N), ctypes.byref(n))
    if st != 0:
        raise SsmError(st, "ssm_selective_scan_fwd_workspace_size")
    return int(n.value)


def selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True, y=None,
                       last_state=None, return_last_state=True, y_dtype=None, stream=None, workspace=None,
                       use_workspace=True, h0=None, zoh=False):
    """Fused selective-scan forward pass.

    u, delta, z: (batch, L, D); A: (D, N) fp32; B, C: (batch, L, N); D, delta_bias: (D) fp32.
    h0 (batch, D, N) fp32: start state; None = zeros. ``last_state`` may be the h0 tensor
    itself (the state is carried in place). zoh: B-bar from the exact zero-order hold,
    (exp(dt A) - 1) / A B, instead of dt B. Either option goes through
    ``ssm_selective_scan_fwd_ex``.
    Outputs are allocated with torch on u's device unless given. Returns (y, last_state);
    last_state is None when ``return_last_state`` is False and none was passed.
    With ``use_workspace`` (default) the call goes through ``ssm_selective_scan_fwd_ws``
    with a workspace of ``workspace_size(...)`` bytes (allocated here with torch unless
    given), which lets long sequences over few channels run as parallel segments;
    ``use_workspace=False`` calls ``ssm_selective_scan_fwd``.
    """
    lib = load_library()
    if y is None:
        y = torch.empty(u.shape, dtype=y_dtype or u.dtype, device=u.device)
    if last_state is None and return_last_state:
        last_state = torch.empty((u.shape[0], u.shape[2], A.shape[-1]), dtype=torch.float32, device=u.device)
    ds = [describe(t) for t in (u, delta, A, B, C, D, z, delta_bias, y, last_state)]
    extended = h0 is not None or zoh
    if not use_workspace and not extended:
        st = lib.ssm_selective_scan_fwd(*[_ref(x) for x in ds[:8]], int(bool(delta_softplus)), _ref(ds[8]),
                                        _ref(ds[9]), _stream(stream))
        if st != 0:
            raise SsmError(st, "ssm_selective_scan_fwd")
        return y, last_state
    if workspace is None and use_workspace:
        nbytes = workspace_size(u.shape[0], u.shape[1], u.shape[2], A.shape[-1])
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=u.device)
    ws_ptr = workspace.data_ptr() if workspace is not None and workspace.numel() > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if ws_ptr else 0
    if extended:
        st = lib.ssm_selective_scan_fwd_ex(*[_ref(x) for x in ds[:8]], int(bool(delta_softplus)),
                                           _ref(describe(h0)), ctypes.c_uint32(SSM_FWD_ZOH if zoh else 0),
                                           _ref(ds[8]), _ref(ds[9]), ctypes.c_void_p(ws_ptr),
                                           ctypes.c_size_t(ws_bytes), _stream(stream))
        if st != 0:
            raise SsmError(st, "ssm_selective_scan_fwd_ex")
        return y, last_state
    st = lib.ssm_selective_scan_fwd_ws(*[_ref(x) for x in ds[:8]], int(bool(delta_softplus)), _ref(ds[8]),
                                       _ref(ds[9]), ctypes.c_void_p(ws_ptr), ctypes.c_size_t(ws_bytes),
                                       _stream(stream))
    if st != 0:
        raise SsmError(st, "ssm_selective_scan_fwd_ws")
    return y, last_state


def bwd_workspace_size(batch, L, D, N) -> int:
    """Bytes of workspace ``ssm_selective_scan_bwd`` needs for this shape."""
    lib = load_library()
    n = ctypes.c_size_t(0)
    st = lib.ssm_selective_scan_bwd_workspace_size(int(batch), int(L), int(D), int(N), ctypes.byref(n))
    if st != 0:
        raise SsmError(st, "ssm_selective_scan_bwd_workspace_size")
    return int(n.value)


def selective_scan_fwd_train(u, delta, A, B, C, workspace, D=None, z=None, delta_bias=None, delta_softplus=True,
                             h0=None, y=None, last_state=None, y_dtype=None, stream=None):
    """Forward pass of a training step (``ssm_selective_scan_fwd_train``): y and last_state
    as ``selective_scan_fwd`` and, into ``workspace`` (a uint8 tensor of
    ``bwd_workspace_size(...)`` bytes, handed on to ``selective_scan_bwd``), the state
    checkpoints of the backward pass. Returns (y, last_state, checkpoints_written)."""
    lib = load_library()
    if y is None:
        y = torch.empty(u.shape, dtype=y_dtype or u.dtype, device=u.device)
    if last_state is None:
        last_state = torch.empty((u.shape[0], u.shape[2], A.shape[-1]), dtype=torch.float32, device=u.device)
    ds = [describe(t) for t in (u, delta, A, B, C, D, z, delta_bias)]
    written = ctypes.c_int32(0)
    ws_ptr = workspace.data_ptr() if workspace is not None and workspace.numel() > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if ws_ptr else 0
    st = lib.ssm_selective_scan_fwd_train(*[_ref(x) for x in ds], int(bool(delta_softplus)), _ref(describe(h0)),
                                          _ref(describe(y)), _ref(describe(last_state)), ctypes.c_void_p(ws_ptr),
                                          ctypes.c_size_t(ws_bytes), ctypes.byref(written), _stream(stream))
    if st != 0:
        raise SsmError(st, "ssm_selective_scan_fwd_train")
    return y, last_state, bool(written.value)


def selective_scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, delta_softplus=True, h0=None,
                       dlast=None, want_dh0=False, workspace=None, stream=None, checkpoints_ready=False):
    """Backward pass (``ssm_selective_scan_bwd_ex``): gradients of sum(dy * y) +
    sum(dlast * last_state). dy's dtype (the I/O dtype or fp32) is the dtype of du,
    ddelta, dz, dB, dC; dA, dD, dbias, dh0 are fp32. Returns a dict with du, ddelta, dA,
    dB, dC and, for the optional inputs given, dD, dz, dbias (dh0 when h0 is given or
    ``want_dh0``). ``checkpoints_ready``: ``workspace`` holds the checkpoints that
    ``selective_scan_fwd_train`` wrote for these inputs (it returned True)."""
    lib = load_library()
    batch, L, Dm = u.shape
    N = A.shape[-1]
    dev, gt = u.device, dy.dtype
    f32 = torch.float32
    g = dict(du=torch.empty(u.shape, dtype=gt, device=dev), ddelta=torch.empty(u.shape, dtype=gt, device=dev),
             dA=torch.empty(A.shape, dtype=f32, device=dev), dB=torch.empty(B.shape, dtype=gt, device=dev),
             dC=torch.empty(C.shape, dtype=gt, device=dev))
    g["dD"] = torch.empty(D.shape, dtype=f32, device=dev) if D is not None else None
    g["dz"] = torch.empty(z.shape, dtype=gt, device=dev) if z is not None else None
    g["dbias"] = torch.empty(delta_bias.shape, dtype=f32, device=dev) if delta_bias is not None else None
    g["dh0"] = torch.empty((batch, Dm, N), dtype=f32, device=dev) if (h0 is not None or want_dh0) else None
    if workspace is None:
        nbytes = bwd_workspace_size(batch, L, Dm, N)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
    ws_ptr = workspace.data_ptr() if workspace is not None and workspace.numel() > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if ws_ptr else 0
    ins = [describe(t) for t in (u, delta, A, B, C, D, z, delta_bias)]
    rest = [describe(t) for t in (h0, dy, dlast, g["du"], g["ddelta"], g["dA"], g["dB"], g["dC"], g["dD"], g["dz"],
                                  g["dbias"], g["dh0"])]
    if checkpoints_ready:
        st = lib.ssm_selective_scan_bwd_ex(*[_ref(d) for d in ins], int(bool(delta_softplus)), *[_ref(d) for d in rest],
                                           ctypes.c_uint32(SSM_BWD_CHECKPOINTS), ctypes.c_void_p(ws_ptr),
                                           ctypes.c_size_t(ws_bytes), _stream(stream))
        name = "ssm_selective_scan_bwd_ex"
    else:
        st = lib.ssm_selective_scan_bwd(*[_ref(d) for d in ins], int(bool(delta_softplus)), *[_ref(d) for d in rest],
                                        ctypes.c_void_p(ws_ptr), ctypes.c_size_t(ws_bytes), _stream(stream))
        name = "ssm_selective_scan_bwd"
    if st != 0:
        raise SsmError(st, name)
    return {k: v for k, v in g.items() if v is not None}


def ssd_workspace_size(batch, L, H, P, N, groups=1) -> int:
    """Bytes of workspace for the chunk-parallel ``ssm_ssd_fwd`` schedule."""
    lib = load_library()
    n = ctypes.c_size_t(0)
    st = lib.ssm_ssd_fwd_workspace_size(int(batch), int(L), int(H), int(groups), int(P), int(N), ctypes.byref(n))
    if st != 0:
        raise SsmError(st, "ssm_ssd_fwd_workspace_size")
    return int(n.value)


def ssd_fwd(x, delta, A, B, C, D=None, dt_bias=None, dt_softplus=True, h0=None, y=None, last_state=None,
            return_last_state=True, y_dtype=None, stream=None, workspace=None, use_workspace=True):
    """Mamba-2 SSD forward (``ssm_ssd_fwd``). x: (batch, L, H, P) bf16; delta: (batch, L, H)
    bf16; A, D, dt_bias: (H) fp32; B, C: (batch, L, G, N) bf16; h0: (batch, H, P, N) fp32.
    With ``use_workspace`` (default) a workspace of ``ssd_workspace_size`` bytes is passed
    (allocated here unless given): the chunk-parallel schedule; without, one CTA per
    (batch, head). Returns (y (batch, L, H, P), last_state (batch, H, P, N))."""
    lib = load_library()
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if workspace is None and use_workspace:
        nbytes = ssd_workspace_size(b, L, H, P, N, groups=G)
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    ws_ptr = workspace.data_ptr() if use_workspace and workspace is not None and workspace.numel() > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if ws_ptr else 0
    if y is None:
        y = torch.empty(x.shape, dtype=y_dtype or x.dtype, device=x.device)
    if last_state is None and return_last_state:
        last_state = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device)
    v3 = lambda t, shape: None if t is None else t.view(shape)
    ds = [describe(t) for t in (v3(x, (b, L, H * P)), delta, A, v3(B, (b, L, G * N)), v3(C, (b, L, G * N)), D, dt_bias)]
    st = lib.ssm_ssd_fwd(ctypes.c_int64(G), *[_ref(d) for d in ds], int(bool(dt_softplus)),
                         _ref(describe(v3(h0, (b, H, P * N)))), _ref(describe(v3(y, (b, L, H * P)))),
                         _ref(describe(v3(last_state, (b, H, P * N)))), ctypes.c_void_p(ws_ptr),
                         ctypes.c_size_t(ws_bytes), _stream(stream))
    if st != 0:
        raise SsmError(st, "ssm_ssd_fwd")
    return y, last_state


def conv_selective_scan_fwd(x, conv_weight, delta, A, B, C, conv_bias=None, conv_state=None, D=None, z=None,
                            delta_bias=None, delta_softplus=True, h0=None, zoh=False, y=None, last_state=None,
                            return_last_state=True, y_dtype=None, stream=None, workspace=None, use_workspace=True):
    """The block's causal width-4 depthwise conv + SiLU fused in front of the forward pass
    (``ssm_conv_selective_scan_fwd``): x (batch, L, D) is the conv input, conv_weight (D, 4)
    fp32, conv_bias (D) fp32. ``conv_state`` (batch, D, 3), I/O dtype, holds the three
    inputs before x[:, 0] and is overwritten with the three before step L (None: zeros, not
    returned). Other arguments as ``selective_scan_fwd``. Returns (y, last_state)."""
    lib = load_library()
    if y is None:
        y = torch.empty(x.shape, dtype=y_dtype or x.dtype, device=x.device)
    if last_state is None and return_last_state:
        last_state = torch.empty((x.shape[0], x.shape[2], A.shape[-1]), dtype=torch.float32, device=x.device)
    if workspace is None and use_workspace:
        nbytes = workspace_size(x.shape[0], x.shape[1], x.shape[2], A.shape[-1])
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    ws_ptr = workspace.data_ptr() if workspace is not None and workspace.numel() > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if ws_ptr else 0
    ds = [describe(t) for t in (x, conv_weight, conv_bias, conv_state, delta, A, B, C, D, z, delta_bias)]
    st = lib.ssm_conv_selective_scan_fwd(*[_ref(d) for d in ds], int(bool(delta_softplus)), _ref(describe(h0)),
                                         ctypes.c_uint32(SSM_FWD_ZOH if zoh else 0), _ref(describe(y)),
                                         _ref(describe(last_state)), ctypes.c_void_p(ws_ptr), ctypes.c_size_t(ws_bytes),
                                         _stream(stream))
    if st != 0:
        raise SsmError(st, "ssm_conv_selective_scan_fwd")
    return y, last_state


def conv_state_update(conv_state, state, x, conv_weight, delta, A, B, C, conv_bias=None, D=None, z=None,
                      delta_bias=None, delta_softplus=True, zoh=False, y=None, y_dtype=None, stream=None):
    """One decode step with the conv prologue (``ssm_conv_state_update``): conv_state
    (batch, D, 3) and state (batch, D, N) are updated in place; x (batch, D) is the conv
    input of this token. Returns y (batch, D)."""
    lib = load_library()
    if y is None:
        y = torch.empty(x.shape, dtype=y_dtype or x.dtype, device=x.device)
    ds = [describe(t) for t in (conv_state, state, x, conv_weight, conv_bias, delta, A, B, C, D, z, delta_bias)]
    st = lib.ssm_conv_state_update(*[_ref(d) for d in ds], int(bool(delta_softplus)),
                                   ctypes.c_uint32(SSM_FWD_ZOH if zoh else 0), _ref(describe(y)), _stream(stream))
    if st != 0:
        raise SsmError(st, "ssm_conv_state_update")
    return y


def state_update(state, x, delta, A, B, C, D=None, z=None, y=None, y_dtype=None, stream=None, delta_bias=None,
                 delta_softplus=False, zoh=False):
    """One decode step; ``state`` (batch, D, N) fp32 is updated in place. x, delta, z:
    (batch, D); B, C: (batch, N). Returns y (batch, D). With ``delta_bias`` (D) fp32 or
    ``delta_softplus`` the step size is softplus(delta + bias) as in the forward pass
    (``ssm_state_update_ex``); otherwise delta is the final step size (``ssm_state_update``).
    zoh: B-bar from the exact zero-order hold, as in ``selective_scan_fwd``."""
    lib = load_library()
    if y is None:
        y = torch.empty(x.shape, dtype=y_dtype or x.dtype, device=x.device)
    ds = [describe(t) for t in (state, x, delta, A, B, C, D, z, y)]
    if delta_bias is None and not delta_softplus and not zoh:
        st = lib.ssm_state_update(*[_ref(d) for d in ds], _stream(stream))
        name = "ssm_state_update"
    else:
        st = lib.ssm_state_update_ex(*[_ref(d) for d in ds[:8]], _ref(describe(delta_bias)), int(bool(delta_softplus)),
                                     ctypes.c_uint32(SSM_FWD_ZOH if zoh else 0), _ref(ds[8]), _stream(stream))
        name = "ssm_state_update_ex"
    if st != 0:
        raise SsmError(st, name)
    return y


def device_error(stream=None) -> int:
    """Synchronise and read/clear the library's device error word (0 = none)."""
    lib = load_library()
    code = ctypes.c_int32(0)
    st = lib.ssm_device_error(_stream(stream), ctypes.byref(code))
    if st != 0:
        raise SsmError(st, "ssm_device_error")
    return int(code.value)
