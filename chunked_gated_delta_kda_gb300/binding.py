"""Python binding of ``libkda.so`` (argument marshalling only).

Every step of the forward runs in the library's CUDA kernels; this module
checks torch tensors, allocates outputs and the workspace with torch on the
tensors' device, and passes raw device pointers and torch's current stream to
the C entry points declared in ``include/kda.h``.  If the library is missing
or fails to load, every call raises: there is no fallback path.

``fwd`` mirrors the operator page's host wrapper signature
(``chunk_kda_wrapper(q, k, v, g, beta, scale=None, initial_state=None,
output_final_state=False, use_qk_l2norm_in_kernel=False, cu_seqlens=None)``,
page "PyPTO-Gym chunk_kda operator", section "算子签名与 I/O 规格").
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import build as _build

KDA_FLAG_QK_L2NORM = 1
KDA_FLAG_BWD_TOKEN_EXACT = 2
KDA_FLAG_BWD_CHUNK_FP32 = 4
KDA_FLAG_SAVE_FOR_BWD = 8
KDA_FLAG_BWD_REUSE_FWD = 16
KDA_FLAG_BWD_UMMA = 32
KDA_FLAG_FWD_TOKEN_EXACT = 64

KDA_DEBUG_WAIT_LIMIT = 1
KDA_DEBUG_DROP_SCAN_LOAD = 2

_STATUS = {
    0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error",
    4: "invalid cu_seqlens", 5: "device wait timed out", 6: "too large for the no-alloc scratch",
    7: "state slot index or accepted-token count out of range",
}

RECURRENT_WORKSPACE_BYTES = 256

_lib = None


class KdaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_STATUS.get(code, 'unknown')} ({code})")


def load_library(path: Optional[str] = None):
    """Load (building first if needed) and return the ctypes handle."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = _build.LIB if _build.up_to_date() else _build.build()
    lib = ctypes.CDLL(path)
    vp, i, f, sz, u = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint
    lib.kda_fwd.restype = ctypes.c_int
    lib.kda_fwd.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp, vp, i, i, i, i, i, i, u, vp, sz, vp]
    lib.kda_fwd_timed.restype = ctypes.c_int
    lib.kda_fwd_timed.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp, vp, i, i, i, i, i, i, u, vp, sz, vp, vp]
    lib.kda_fwd_noalloc.restype = ctypes.c_int
    lib.kda_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp, vp, i, i, i, i, i, i, u, vp]
    lib.kda_fwd_workspace_bytes.restype = sz
    lib.kda_fwd_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.kda_get_status.restype = ctypes.c_int
    lib.kda_get_status.argtypes = [vp, vp]
    lib.kda_fused_recurrent.restype = ctypes.c_int
    lib.kda_fused_recurrent.argtypes = [vp, vp, vp, vp, vp, f, vp, i, vp, i, vp, vp, vp,
                                        i, i, i, i, i, i, u, vp, vp]
    lib.kda_kcp_workspace_bytes.restype = sz
    lib.kda_kcp_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.kda_kcp_fwd.restype = ctypes.c_int
    lib.kda_kcp_fwd.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp, vp, i, i, i, i, i, i, u, vp, sz, vp]
    lib.kda_bwd_workspace_bytes.restype = sz
    lib.kda_bwd_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.kda_bwd.restype = ctypes.c_int
    lib.kda_bwd.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                            i, i, i, i, i, i, u, vp, sz, vp]
    lib.kda_bwd_timed.restype = ctypes.c_int
    lib.kda_bwd_timed.argtypes = lib.kda_bwd.argtypes + [vp]
    lib.kda_debug_set.restype = ctypes.c_int
    lib.kda_debug_set.argtypes = [i, u]
    lib.kda_status_str.restype = ctypes.c_char_p
    lib.kda_status_str.argtypes = [i]
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def workspace_bytes(B: int, T: int, H: int, N: int, K: int = 128, V: int = 128) -> int:
    return int(load_library().kda_fwd_workspace_bytes(B, T, H, K, V, N))


def kda_fwd(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, N: int, flags: int,
            workspace: torch.Tensor) -> None:
    """Direct call of the C entry point on caller-provided tensors (all on one
    CUDA device, contiguous).  Raises KdaError on a non-zero status."""
    lib = load_library()
    B, T, H, K = q.shape
    V = v.shape[-1]
    rc = lib.kda_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                     float(scale if scale is not None else -1.0), _ptr(h0), _ptr(cu_seqlens),
                     _ptr(o), _ptr(ht), B, T, H, K, V, N, flags, _ptr(workspace),
                     workspace.numel() * workspace.element_size(), _stream_handle(q.device))
    if rc != 0:
        raise KdaError(rc, "kda_fwd")


def kda_fwd_timed(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, N: int, flags: int,
                  workspace: torch.Tensor, events) -> None:
    """kda_fwd that also records three torch.cuda.Event objects (created with
    enable_timing=True) around the two stages on torch's current stream."""
    lib = load_library()
    B, T, H, K = q.shape
    V = v.shape[-1]
    ev = (ctypes.c_void_p * 3)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    rc = lib.kda_fwd_timed(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           float(scale if scale is not None else -1.0), _ptr(h0), _ptr(cu_seqlens),
                           _ptr(o), _ptr(ht), B, T, H, K, V, N, flags, _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream_handle(q.device), ev)
    if rc != 0:
        raise KdaError(rc, "kda_fwd_timed")


def kda_fwd_noalloc(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, N: int, flags: int) -> None:
    """The no-allocation entry point: like kda_fwd but the library supplies
    the workspace from its static device scratch (for callers that cannot
    allocate device memory).  Raises KdaError (code 6) if the problem does
    not fit the scratch."""
    lib = load_library()
    B, T, H, K = q.shape
    V = v.shape[-1]
    rc = lib.kda_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                             float(scale if scale is not None else -1.0), _ptr(h0), _ptr(cu_seqlens),
                             _ptr(o), _ptr(ht), B, T, H, K, V, N, flags, _stream_handle(q.device))
    if rc != 0:
        raise KdaError(rc, "kda_fwd_noalloc")


def debug_set(what: int, value: int) -> None:
    """Test hook of the bounded device waits (``kda_debug_set``): the poll
    limit (``KDA_DEBUG_WAIT_LIMIT``, 0 = default) or a one-shot dropped scan
    load (``KDA_DEBUG_DROP_SCAN_LOAD``) for the next forward."""
    rc = load_library().kda_debug_set(int(what), int(value))
    if rc != 0:
        raise KdaError(rc, "kda_debug_set")


def get_status(workspace: torch.Tensor) -> int:
    """Synchronise torch's current stream and return the device status code."""
    lib = load_library()
    return int(lib.kda_get_status(_ptr(workspace), _stream_handle(workspace.device)))


def _check(name, t, dtype, ndim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
        scale: Optional[float] = None, initial_state: Optional[torch.Tensor] = None,
        output_final_state: bool = False, use_qk_l2norm_in_kernel: bool = False,
        cu_seqlens: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
        save_for_backward: bool = False, token_exact: bool = False) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunked KDA forward.  ``token_exact`` computes every (sequence, head)
    token by token with an fp32 state instead (``KDA_FLAG_FWD_TOKEN_EXACT``:
    for very slowly decaying heads; slower).  ``save_for_backward`` (training) also stores the
    chunk states in ``workspace`` (which must then be a caller tensor of at
    least ``bwd_workspace_bytes`` bytes) for ``bwd(..., reuse_forward=True,
    workspace=<the same tensor>)``.  q, k: bf16 [B,T,H,K]; v: bf16 [B,T,H,V]; g: fp32
    [B,T,H,K]; beta: fp32 [B,T,H]; initial_state: fp32 [N,H,V,K] or None;
    cu_seqlens: int32 [N+1] on the device (varlen, B == 1) or None (fixed
    length, T % 128 == 0).  Returns (o bf16 [B,T,H,V], final state fp32
    [N,H,V,K] or None)."""
    _check("q", q, torch.bfloat16, 4)
    _check("k", k, torch.bfloat16, 4)
    _check("v", v, torch.bfloat16, 4)
    _check("g", g, torch.float32, 4)
    _check("beta", beta, torch.float32, 3)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape or v.shape[:3] != q.shape[:3] or beta.shape != q.shape[:3]:
        raise ValueError("shape mismatch among q, k, v, g, beta")
    if cu_seqlens is not None:
        _check("cu_seqlens", cu_seqlens, torch.int32, 1)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if initial_state is not None:
        _check("initial_state", initial_state, torch.float32, 4)
        if tuple(initial_state.shape) != (N, H, V, K):
            raise ValueError(f"initial_state must be {(N, H, V, K)}, got {tuple(initial_state.shape)}")
    dev = q.device
    tensors = [q, k, v, g, beta] + [t for t in (initial_state, cu_seqlens) if t is not None]
    if any(t.device != dev for t in tensors):
        raise ValueError("all tensors must be on the same device")
    q, k, v, g, beta = (t.contiguous() for t in (q, k, v, g, beta))
    h0 = initial_state.contiguous() if initial_state is not None else None
    o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=dev)
    ht = torch.empty((N, H, V, K), dtype=torch.float32, device=dev) if output_final_state else None
    need = bwd_workspace_bytes(B, T, H, N, K, V) if save_for_backward else workspace_bytes(B, T, H, N, K, V)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        if save_for_backward:
            raise ValueError("save_for_backward needs a workspace of at least bwd_workspace_bytes(...) bytes")
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    flags = ((KDA_FLAG_QK_L2NORM if use_qk_l2norm_in_kernel else 0) | (KDA_FLAG_SAVE_FOR_BWD if save_for_backward else 0)
             | (KDA_FLAG_FWD_TOKEN_EXACT if token_exact else 0))
    with torch.cuda.device(dev):
        kda_fwd(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, N, flags, workspace)
    return o, ht


def kda_fused_recurrent(q, k, v, g, beta, scale, state_pool, ssm_state_indices, num_accepted_tokens,
                        cu_seqlens, o, N: int, flags: int, workspace: torch.Tensor) -> None:
    """Direct call of the token-by-token entry point on caller-provided
    tensors.  ``state_pool`` fp32 [P,H,V,K] is updated in place;
    ``ssm_state_indices`` is int32 [N, stride].  Raises KdaError on a
    non-zero status."""
    lib = load_library()
    B, T, H, K = q.shape
    V = v.shape[-1]
    stride = ssm_state_indices.shape[1] if ssm_state_indices.dim() == 2 else 1
    rc = lib.kda_fused_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                 float(scale if scale is not None else -1.0), _ptr(state_pool),
                                 int(state_pool.shape[0]), _ptr(ssm_state_indices), stride,
                                 _ptr(num_accepted_tokens), _ptr(cu_seqlens), _ptr(o), B, T, H, K, V, N,
                                 flags, _ptr(workspace), _stream_handle(q.device))
    if rc != 0:
        raise KdaError(rc, "kda_fused_recurrent")


def fused_recurrent(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                    state_pool: torch.Tensor, ssm_state_indices: torch.Tensor, scale: Optional[float] = None,
                    num_accepted_tokens: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None,
                    use_qk_l2norm_in_kernel: bool = False, workspace: Optional[torch.Tensor] = None
                    ) -> torch.Tensor:
    """Token-by-token KDA with an in-place state pool (the decode sibling of
    ``fwd``).  q, k: bf16 [B,T,H,K]; v: bf16 [B,T,H,V]; g fp32 [B,T,H,K];
    beta fp32 [B,T,H]; state_pool fp32 [P,H,V,K] (updated in place);
    ssm_state_indices int32 [N] or [N, S]; num_accepted_tokens int32 [N] or
    None; cu_seqlens int32 [N+1] (B == 1) or None.  Returns o bf16
    [B,T,H,V]."""
    _check("q", q, torch.bfloat16, 4)
    _check("k", k, torch.bfloat16, 4)
    _check("v", v, torch.bfloat16, 4)
    _check("g", g, torch.float32, 4)
    _check("beta", beta, torch.float32, 3)
    _check("state_pool", state_pool, torch.float32, 4)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape or v.shape[:3] != q.shape[:3] or beta.shape != q.shape[:3]:
        raise ValueError("shape mismatch among q, k, v, g, beta")
    if tuple(state_pool.shape[1:]) != (H, V, K) or not state_pool.is_contiguous():
        raise ValueError(f"state_pool must be a contiguous [P, {H}, {V}, {K}] tensor")
    idx = ssm_state_indices
    if idx.dtype != torch.int32 or not idx.is_cuda or idx.dim() not in (1, 2):
        raise ValueError("ssm_state_indices must be a CUDA int32 tensor [N] or [N, S]")
    idx = idx.reshape(idx.shape[0], -1).contiguous()
    N = idx.shape[0]
    if cu_seqlens is not None:
        _check("cu_seqlens", cu_seqlens, torch.int32, 1)
        if cu_seqlens.numel() != N + 1:
            raise ValueError("cu_seqlens must have N + 1 entries")
    if num_accepted_tokens is not None:
        _check("num_accepted_tokens", num_accepted_tokens, torch.int32, 1)
        if num_accepted_tokens.numel() != N:
            raise ValueError("num_accepted_tokens must have N entries")
    dev = q.device
    q, k, v, g, beta = (t.contiguous() for t in (q, k, v, g, beta))
    o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=dev)
    if workspace is None or workspace.numel() * workspace.element_size() < RECURRENT_WORKSPACE_BYTES:
        workspace = torch.empty(RECURRENT_WORKSPACE_BYTES, dtype=torch.uint8, device=dev)
    flags = KDA_FLAG_QK_L2NORM if use_qk_l2norm_in_kernel else 0
    with torch.cuda.device(dev):
        kda_fused_recurrent(q, k, v, g, beta, scale, state_pool, idx, num_accepted_tokens, cu_seqlens, o, N,
                            flags, workspace)
    return o


def kcp_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
            cu_seqlens, world_size: int, scale: Optional[float] = None,
            initial_state: Optional[torch.Tensor] = None, output_final_state: bool = False,
            use_qk_l2norm_in_kernel: bool = False) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """KCP forward with ``world_size`` ranks simulated on q's device.
    Packed inputs (B == 1) as for ``fwd``; ``cu_seqlens`` is a host sequence
    of N + 1 offsets (list, numpy array or CPU tensor).  Returns (o, final
    state or None)."""
    _check("q", q, torch.bfloat16, 4)
    _check("k", k, torch.bfloat16, 4)
    _check("v", v, torch.bfloat16, 4)
    _check("g", g, torch.float32, 4)
    _check("beta", beta, torch.float32, 3)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if B != 1:
        raise ValueError("kcp_fwd takes packed inputs (B == 1)")
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu().contiguous()
    N = cu.numel() - 1
    dev = q.device
    q, k, v, g, beta = (t.contiguous() for t in (q, k, v, g, beta))
    h0 = initial_state.contiguous() if initial_state is not None else None
    if h0 is not None and (h0.dtype != torch.float32 or tuple(h0.shape) != (N, H, V, K)):
        raise ValueError(f"initial_state must be fp32 {(N, H, V, K)}")
    o = torch.empty((1, T, H, V), dtype=torch.bfloat16, device=dev)
    ht = torch.empty((N, H, V, K), dtype=torch.float32, device=dev) if output_final_state else None
    lib = load_library()
    nbytes = int(lib.kda_kcp_workspace_bytes(T, H, K, V, N, world_size))
    if nbytes == 0:
        raise KdaError(1, "kda_kcp_workspace_bytes")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    flags = KDA_FLAG_QK_L2NORM if use_qk_l2norm_in_kernel else 0
    with torch.cuda.device(dev):
        rc = lib.kda_kcp_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                             float(scale if scale is not None else -1.0), _ptr(h0),
                             ctypes.c_void_p(cu.data_ptr()), _ptr(o), _ptr(ht), T, H, K, V, N, world_size, flags,
                             _ptr(ws), nbytes, _stream_handle(dev))
    if rc != 0:
        raise KdaError(rc, "kda_kcp_fwd")
    return o, ht


def bwd_workspace_bytes(B: int, T: int, H: int, N: int, K: int = 128, V: int = 128) -> int:
    return int(load_library().kda_bwd_workspace_bytes(B, T, H, K, V, N))


def kda_bwd(q, k, v, g, beta, scale, h0, cu_seqlens, dout, dht, dq, dk, dv, dg, dbeta, dh0, N: int, flags: int,
            workspace: torch.Tensor) -> None:
    """Direct call of the backward entry point on caller-provided tensors.
    Raises KdaError on a non-zero status."""
    lib = load_library()
    B, T, H, K = q.shape
    V = v.shape[-1]
    rc = lib.kda_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale if scale is not None else -1.0),
                     _ptr(h0), _ptr(cu_seqlens), _ptr(dout), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                     _ptr(dbeta), _ptr(dh0), B, T, H, K, V, N, flags, _ptr(workspace),
                     workspace.numel() * workspace.element_size(), _stream_handle(q.device))
    if rc != 0:
        raise KdaError(rc, "kda_bwd")


def kda_bwd_timed(q, k, v, g, beta, scale, h0, cu_seqlens, dout, dht, dq, dk, dv, dg, dbeta, dh0, N: int,
                  flags: int, workspace: torch.Tensor, events) -> None:
    """kda_bwd that also records six torch.cuda.Event objects at its stage
    boundaries on torch's current stream."""
    lib = load_library()
    B, T, H, K = q.shape
    V = v.shape[-1]
    ev = (ctypes.c_void_p * 6)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    rc = lib.kda_bwd_timed(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           float(scale if scale is not None else -1.0), _ptr(h0), _ptr(cu_seqlens), _ptr(dout),
                           _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0), B, T, H, K, V,
                           N, flags, _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream_handle(q.device), ev)
    if rc != 0:
        raise KdaError(rc, "kda_bwd_timed")


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
        do: torch.Tensor, scale: Optional[float] = None, initial_state: Optional[torch.Tensor] = None,
        dht: Optional[torch.Tensor] = None, use_qk_l2norm_in_kernel: bool = False,
        cu_seqlens: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
        token_exact: bool = False, chunk_fp32: bool = False, reuse_forward: bool = False, umma: bool = False):
    """KDA backward of ``fwd`` with the same arguments: the gradients of
    <do, o> + <dht, ht>.  do: bf16 [B,T,H,V]; dht: fp32 [N,H,V,K] or None.
    ``token_exact`` selects the token-by-token backward for every unit;
    ``chunk_fp32`` the per-token fp32 chain rule inside every chunk (instead
    of the chunked form on the tensor cores); ``reuse_forward`` skips the
    forward replay, using what ``fwd(..., save_for_backward=True)`` left in
    ``workspace`` for the same inputs; ``umma`` the per-chunk chain rule on
    tcgen05 products instead of the warp-level TF32 ones.
    Returns fp32 (dq, dk, dv, dg, dbeta, dh0) with the shapes of q, k, v, g,
    beta and the state [N,H,V,K]."""
    for name, t, dt, nd in (("q", q, torch.bfloat16, 4), ("k", k, torch.bfloat16, 4), ("v", v, torch.bfloat16, 4),
                            ("g", g, torch.float32, 4), ("beta", beta, torch.float32, 3),
                            ("do", do, torch.bfloat16, 4)):
        _check(name, t, dt, nd)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if (k.shape != q.shape or g.shape != q.shape or v.shape[:3] != q.shape[:3] or beta.shape != q.shape[:3]
            or do.shape != v.shape):
        raise ValueError("shape mismatch among q, k, v, g, beta, do")
    if cu_seqlens is not None:
        _check("cu_seqlens", cu_seqlens, torch.int32, 1)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    for name, t in (("initial_state", initial_state), ("dht", dht)):
        if t is not None:
            _check(name, t, torch.float32, 4)
            if tuple(t.shape) != (N, H, V, K):
                raise ValueError(f"{name} must be {(N, H, V, K)}, got {tuple(t.shape)}")
    dev = q.device
    q, k, v, g, beta, do = (t.contiguous() for t in (q, k, v, g, beta, do))
    h0 = initial_state.contiguous() if initial_state is not None else None
    dht = dht.contiguous() if dht is not None else None
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk, dg = (torch.empty((B, T, H, K), **f32) for _ in range(3))
    dv = torch.empty((B, T, H, V), **f32)
    dbeta = torch.empty((B, T, H), **f32)
    dh0 = torch.empty((N, H, V, K), **f32)
    need = bwd_workspace_bytes(B, T, H, N, K, V)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        if reuse_forward:
            raise ValueError("reuse_forward needs the workspace the saving forward used")
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    flags = ((KDA_FLAG_QK_L2NORM if use_qk_l2norm_in_kernel else 0) | (KDA_FLAG_BWD_TOKEN_EXACT if token_exact else 0)
             | (KDA_FLAG_BWD_CHUNK_FP32 if chunk_fp32 else 0) | (KDA_FLAG_BWD_REUSE_FWD if reuse_forward else 0)
             | (KDA_FLAG_BWD_UMMA if umma else 0))
    with torch.cuda.device(dev):
        kda_bwd(q, k, v, g, beta, scale, h0, cu_seqlens, do, dht, dq, dk, dv, dg, dbeta, dh0, N, flags, workspace)
    return dq, dk, dv, dg, dbeta, dh0
