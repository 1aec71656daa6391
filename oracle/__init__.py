"""fp64 CPU oracle for the Mamba selective scan and the recurrent state update.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package. It shares
no code with the CUDA library and never imports it.

The arithmetic lives in ``ssm_oracle.c`` (plain C, fp64, sequential); this module
only marshals numpy arrays into it. Definitions and their sources (page title and
section) are in the C header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libssm_oracle.so"
_dp = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(out_dir: str | None = None, plant: int = 0, force: bool = False) -> str:
    """Compile ssm_oracle.c into a shared library; returns its path.

    ``plant`` > 0 compiles a deliberately wrong variant (see ssm_oracle.c) used only by
    the pin tests to show that each planted mistake is caught.
    """
    out_dir = out_dir or _HERE
    name = LIB_NAME if plant == 0 else f"libssm_oracle_plant{plant}.so"
    out = os.path.join(out_dir, name)
    src = os.path.join(_HERE, "ssm_oracle.c")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(
        os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "ssm_oracle.h"))
    ):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           f"-DSSM_ORACLE_PLANT={plant}", "-o", out, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _f64(a, shape=None):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor -> numpy (CPU), exact widening to fp64
        a = a.detach().to("cpu").double().numpy()
    a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None and tuple(a.shape) != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {tuple(a.shape)}")
    return a


class Oracle:
    """ctypes front end over one build of the oracle library."""

    def __init__(self, lib_path: str | None = None):
        self.path = lib_path or build()
        lib = ctypes.CDLL(self.path)
        lib.ssm_oracle_softplus.restype = ctypes.c_double
        lib.ssm_oracle_softplus.argtypes = [ctypes.c_double]
        lib.ssm_oracle_silu.restype = ctypes.c_double
        lib.ssm_oracle_silu.argtypes = [ctypes.c_double]
        lib.ssm_oracle_fwd.restype = ctypes.c_int
        lib.ssm_oracle_fwd.argtypes = [_i64, _i64, _i64, _i64] + [_dp] * 8 + [ctypes.c_int, _dp, _dp, _dp,
                                                                               ctypes.c_int]
        lib.ssm_oracle_state_update.restype = ctypes.c_int
        lib.ssm_oracle_state_update.argtypes = [_i64, _i64, _i64] + [_dp] * 9
        lib.ssm_oracle_state_update_ex.restype = ctypes.c_int
        lib.ssm_oracle_state_update_ex.argtypes = [_i64, _i64, _i64] + [_dp] * 9 + [ctypes.c_int, ctypes.c_int, _dp]
        lib.ssm_oracle_conv1d_silu.restype = ctypes.c_int
        lib.ssm_oracle_conv1d_silu.argtypes = [_i64, _i64, _i64] + [_dp] * 5
        lib.ssm_oracle_bwd.restype = ctypes.c_int
        lib.ssm_oracle_bwd.argtypes = [_i64, _i64, _i64, _i64] + [_dp] * 8 + [ctypes.c_int] + [_dp] * 12
        lib.ssm_oracle_ssd_fwd.restype = ctypes.c_int
        lib.ssm_oracle_ssd_fwd.argtypes = [_i64] * 6 + [_dp] * 7 + [ctypes.c_int, _dp, _dp, _dp]
        lib.ssm_oracle_fwd_ex.restype = ctypes.c_int
        lib.ssm_oracle_fwd_ex.argtypes = [_i64, _i64, _i64, _i64] + [_dp] * 8 + [ctypes.c_int, ctypes.c_int, _dp, _dp,
                                                                                 _dp, ctypes.c_int]
        self.lib = lib

    def softplus(self, r: float) -> float:
        return self.lib.ssm_oracle_softplus(float(r))

    def silu(self, z: float) -> float:
        return self.lib.ssm_oracle_silu(float(z))

    def selective_scan_fwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                           delta_softplus=True, h0=None, nthreads=0, zoh=False):
        """Returns (y, last_state) as fp64 numpy arrays.

        u, delta, z: (batch, L, D); A: (D, N); B, C: (batch, L, N); D, delta_bias: (D);
        h0: (batch, D, N) initial state (zeros if None). zoh: B-bar from the exact
        zero-order hold, (exp(dt A) - 1) / A * B, instead of dt * B.
        """
        u = _f64(u)
        batch, L, Dm = u.shape
        A = _f64(A)
        N = A.shape[1]
        delta = _f64(delta, (batch, L, Dm))
        B = _f64(B, (batch, L, N))
        C = _f64(C, (batch, L, N))
        A = _f64(A, (Dm, N))
        D = _f64(D, (Dm,))
        z = _f64(z, (batch, L, Dm))
        delta_bias = _f64(delta_bias, (Dm,))
        h0 = _f64(h0, (batch, Dm, N))
        y = np.empty((batch, L, Dm), np.float64)
        last = np.empty((batch, Dm, N), np.float64)
        rc = self.lib.ssm_oracle_fwd_ex(batch, L, Dm, N, _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                        _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)),
                                        int(bool(zoh)), _ptr(h0), _ptr(y), _ptr(last), int(nthreads))
        if rc != 0:
            raise RuntimeError("ssm_oracle_fwd rejected its arguments")
        return y, last

    def selective_scan_bwd(self, u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, delta_softplus=True,
                           h0=None, dlast=None):
        """Gradients of sum(dy * y) + sum(dlast * last_state) of selective_scan_fwd (dt B
        discretisation). Returns a dict of fp64 arrays: du, ddelta, dA, dB, dC and, when
        the matching input is given, dD, dz, dbias, dh0."""
        u = _f64(u)
        batch, L, Dm = u.shape
        A = _f64(A)
        N = A.shape[1]
        delta = _f64(delta, (batch, L, Dm))
        B = _f64(B, (batch, L, N))
        C = _f64(C, (batch, L, N))
        D = _f64(D, (Dm,))
        z = _f64(z, (batch, L, Dm))
        delta_bias = _f64(delta_bias, (Dm,))
        h0 = _f64(h0, (batch, Dm, N))
        dy = _f64(dy, (batch, L, Dm))
        dlast = _f64(dlast, (batch, Dm, N))
        out = dict(du=np.empty((batch, L, Dm)), ddelta=np.empty((batch, L, Dm)), dA=np.empty((Dm, N)),
                   dB=np.empty((batch, L, N)), dC=np.empty((batch, L, N)))
        out["dD"] = np.empty(Dm) if D is not None else None
        out["dz"] = np.empty((batch, L, Dm)) if z is not None else None
        out["dbias"] = np.empty(Dm) if delta_bias is not None else None
        out["dh0"] = np.empty((batch, Dm, N)) if h0 is not None else None
        rc = self.lib.ssm_oracle_bwd(batch, L, Dm, N, _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                     _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(h0), _ptr(dy),
                                     _ptr(dlast), _ptr(out["du"]), _ptr(out["ddelta"]), _ptr(out["dA"]),
                                     _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dz"]),
                                     _ptr(out["dbias"]), _ptr(out["dh0"]))
        if rc != 0:
            raise RuntimeError("ssm_oracle_bwd rejected its arguments")
        return {k: v for k, v in out.items() if v is not None}

    def ssd_fwd(self, x, delta, A, B, C, D=None, dt_bias=None, dt_softplus=True, h0=None):
        """Mamba-2 SSD forward (sequential). x: (batch, L, H, P); delta: (batch, L, H);
        A, D, dt_bias: (H); B, C: (batch, L, G, N); h0: (batch, H, P, N). Returns
        (y (batch, L, H, P), last_state (batch, H, P, N)) as fp64 arrays."""
        x = _f64(x)
        batch, L, H, P = x.shape
        B = _f64(B)
        G, N = B.shape[2], B.shape[3]
        delta = _f64(delta, (batch, L, H))
        A = _f64(A, (H,))
        C = _f64(C, (batch, L, G, N))
        D = _f64(D, (H,))
        dt_bias = _f64(dt_bias, (H,))
        h0 = _f64(h0, (batch, H, P, N))
        y = np.empty((batch, L, H, P))
        last = np.empty((batch, H, P, N))
        rc = self.lib.ssm_oracle_ssd_fwd(batch, L, H, P, N, G, _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                         _ptr(D), _ptr(dt_bias), int(bool(dt_softplus)), _ptr(h0), _ptr(y),
                                         _ptr(last))
        if rc != 0:
            raise RuntimeError("ssm_oracle_ssd_fwd rejected its arguments")
        return y, last

    def conv1d_silu(self, x, w, bias=None, conv_state=None):
        """u = silu(causal depthwise conv of width 4 (+ bias)) as an fp64 array.

        x: (batch, L, D); w: (D, 4); bias: (D); conv_state: (batch, D, 3), the three
        inputs before x[:, 0], oldest first (zeros if None).
        """
        x = _f64(x)
        batch, L, Dm = x.shape
        w = _f64(w, (Dm, 4))
        bias = _f64(bias, (Dm,))
        conv_state = _f64(conv_state, (batch, Dm, 3))
        u = np.empty((batch, L, Dm), np.float64)
        if self.lib.ssm_oracle_conv1d_silu(batch, L, Dm, _ptr(x), _ptr(w), _ptr(bias), _ptr(conv_state), _ptr(u)):
            raise RuntimeError("ssm_oracle_conv1d_silu rejected its arguments")
        return u

    @staticmethod
    def next_conv_state(x, conv_state=None):
        """The three inputs before step L (what follows x[:, L-1]): the last three of
        conv_state followed by x, as (batch, D, 3), oldest first."""
        x = _f64(x)
        batch, L, Dm = x.shape
        prev = np.zeros((batch, Dm, 3)) if conv_state is None else _f64(conv_state, (batch, Dm, 3))
        seq = np.concatenate([prev, np.transpose(x, (0, 2, 1))], axis=2)
        return np.ascontiguousarray(seq[:, :, -3:])

    def conv_selective_scan_fwd(self, x, conv_weight, A, B, C, delta, conv_bias=None, conv_state=None, **kw):
        """The conv + SiLU prologue, then selective_scan_fwd on its output. Returns
        (y, last_state, next_conv_state)."""
        u = self.conv1d_silu(x, conv_weight, conv_bias, conv_state)
        y, last = self.selective_scan_fwd(u, delta, A, B, C, **kw)
        return y, last, self.next_conv_state(x, conv_state)

    def state_update(self, state, x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
                     zoh=False):
        """One decode step. Returns (y, new_state); the input state is not modified.

        state: (batch, D, N); x, delta, z: (batch, D); A: (D, N); B, C: (batch, N); D: (D).
        delta_bias (D) / delta_softplus: the forward pass's step-size map applied to delta
        first (dt = softplus(delta + bias)); by default delta is the final step size.
        zoh: B-bar from the exact zero-order hold (as in selective_scan_fwd).
        """
        st = _f64(state).copy()
        batch, Dm, N = st.shape
        x = _f64(x, (batch, Dm))
        delta = _f64(delta, (batch, Dm))
        A = _f64(A, (Dm, N))
        B = _f64(B, (batch, N))
        C = _f64(C, (batch, N))
        D = _f64(D, (Dm,))
        z = _f64(z, (batch, Dm))
        delta_bias = _f64(delta_bias, (Dm,))
        y = np.empty((batch, Dm), np.float64)
        rc = self.lib.ssm_oracle_state_update_ex(batch, Dm, N, _ptr(st), _ptr(x), _ptr(delta), _ptr(A),
                                                 _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
                                                 int(bool(delta_softplus)), int(bool(zoh)), _ptr(y))
        if rc != 0:
            raise RuntimeError("ssm_oracle_state_update rejected its arguments")
        return y, st


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def selective_scan_fwd(*args, **kwargs):
    return default().selective_scan_fwd(*args, **kwargs)


def state_update(*args, **kwargs):
    return default().state_update(*args, **kwargs)


def conv1d_silu(*args, **kwargs):
    return default().conv1d_silu(*args, **kwargs)


def selective_scan_bwd(*args, **kwargs):
    return default().selective_scan_bwd(*args, **kwargs)


def ssd_fwd(*args, **kwargs):
    return default().ssd_fwd(*args, **kwargs)


def conv_selective_scan_fwd(*args, **kwargs):
    return default().conv_selective_scan_fwd(*args, **kwargs)


def next_conv_state(*args, **kwargs):
    return Oracle.next_conv_state(*args, **kwargs)
