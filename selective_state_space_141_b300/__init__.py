"""B300-native (sm_103a) Mamba selective scan: fused forward pass and decode step.

The compute runs in hand-written CUDA kernels inside ``libssm_b300.so`` behind the C
ABI declared in ``include/ssm.h``; ``ssm.py`` is a thin ctypes binding over it (device
memory and streams come from PyTorch). ``inputs`` holds the seeded workload generators.
There is no CPU fallback: calling an op without the built library raises.
"""
from . import inputs  # noqa: F401

_BINDING = ("selective_scan_fwd", "state_update", "device_error", "library_path", "load_library",
            "SsmError")


def __getattr__(name):
    if name in _BINDING:
        from . import ssm
        return getattr(ssm, name)
    raise AttributeError(name)
