"""Chunked Kimi Delta Attention (KDA) forward for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libkda.so`` built from ``csrc/``
(hand-written CUDA kernels).  ``kda_fwd`` (Python, in ``binding.py``) only
marshals torch tensors into that C call; importing it loads the library and
fails loudly when it is missing.  ``inputs`` (synthetic workloads) is
importable without the library.
"""

__all__ = ["fwd", "kda_fwd", "load_library"]


def __getattr__(name):
    if name in ("fwd", "kda_fwd", "load_library", "workspace_bytes", "KdaError"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
