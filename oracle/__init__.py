"""KDA forward oracle (fp64, CPU).

TEST INFRASTRUCTURE ONLY.  The oracle is what the CUDA path is checked
against.  It shares no code with ``chunked_gated_delta_kda_gb300`` (no kernels,
headers, helpers, tables or constants) and neither imports the other.  Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import it; the product path never does.

Independent forms:
  * ``kda_recurrent``: the per-token recurrence in plain C, fp64, OpenMP over
    (sequence, head) units (``kda_recurrent.c``).  This is the definition of
    the result.
  * ``kda_chunked``: the chunked M1-M4 form in numpy fp64 with an explicit
    triangular solve (``chunked.py``).  It equals the recurrence up to rounding
    order and serves to pin the chunked reading of the page.
  * ``fused_recurrent``: the token-by-token recurrence with an in-place state
    pool, slot indices and speculative-decoding checkpoints, numpy fp64
    (``decode.py``): the oracle of the decode entry point.
  * ``kcp_forward``: the KCP forward simulated rank by rank (``kcp.py``).
  * ``backward.kda_backward``: gradients of <do, o> + <dht, ht> by fp64
    torch autograd through the per-token recurrence (``backward.py``): the
    oracle of the backward entry point.

Parity pins live in ``tests/test_oracle*.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .chunked import kda_chunked  # noqa: F401
from .decode import fused_recurrent  # noqa: F401
from .kcp import kcp_forward  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_recurrent.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libkda_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/libkda_oracle.so`` with gcc.

    -ffp-contract=off keeps the fp64 rounding identical on x86 and Arm hosts.
    """
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.kda_oracle_recurrent.restype = ctypes.c_int
        lib.kda_oracle_recurrent.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p]
        lib.kda_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    """Host threads the C oracle's OpenMP loop uses."""
    return int(_load().kda_oracle_max_threads())


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def kda_recurrent(q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None,
                  l2norm=False, units=None, want_state=True):
    """Per-token fp64 recurrence.

    q, k, g: (B, T, H, K); v: (B, T, H, V); beta: (B, T, H) -- any array
    convertible to float32 exactly (bf16 data widened by the caller);
    h0: (N, H, V, K) or None; cu_seqlens: (N+1,) int or None.  ``scale``
    None means K**-0.5.  ``units``: optional iterable of (n, h) to compute;
    the rest of o / ht is NaN.  Returns (o float64 (B, T, H, V),
    ht float64 (N, H, V, K) or None).
    """
    q, k, v, g, beta = _f32(q), _f32(k), _f32(v), _f32(g), _f32(beta)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = K ** -0.5
    if cu_seqlens is None:
        N = B
        cu = None
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = cu.shape[0] - 1
    h0a = None if h0 is None else _f32(h0)
    mask = None
    if units is not None:
        mask = np.zeros(N * H, dtype=np.uint8)
        for n, h in units:
            mask[n * H + h] = 1
    o = np.full((B, T, H, V), np.nan)
    ht = np.full((N, H, V, K), np.nan) if want_state else None
    rc = _load().kda_oracle_recurrent(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(h0a),
        _ptr(cu), B, T, H, K, V, N, int(bool(l2norm)), _ptr(mask), _ptr(o), _ptr(ht))
    if rc != 0:
        raise ValueError(f"kda_oracle_recurrent failed with code {rc}")
    return o, ht
