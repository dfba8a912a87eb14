"""graph_replay_gb300: the constant-shape small-batch decode step, captured once
into a CUDA graph and replayed per token, as hand-written sm_103a kernels behind
a C ABI (include/graphdec.h, libgraphdec.so).

The package holds only the path: ``csrc/`` (kernels + C ABI), ``_binding``
(ctypes, same names as the header) and ``decoder`` (torch-owned device memory
around one handle).  Importing ``Decoder`` requires the built library; there is
no CPU fallback.
"""
from . import build  # noqa: F401


def __getattr__(name):
    if name in ("Decoder", "StepResult", "make_config"):
        import importlib
        return getattr(importlib.import_module(".decoder", __name__), name)
    raise AttributeError(name)
