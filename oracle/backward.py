"""Gradients of the KDA forward, fp64 (plain PyTorch CPU autograd).

TEST INFRASTRUCTURE ONLY: the oracle of the library's backward entry point.
It shares no code with the CUDA path.

The forward it differentiates is the per-token rule of the page "PyPTO-Gym
chunk_kda operator: an NPU forward of chunked gated delta-rule linear
attention" (section "算子定位与算法背景": decay S <- diag(exp(g)) S, delta
update S <- S + beta k (v - S^T k)^T, read-out o = S^T (scale q); the
optional per-token q/k normalisation x / sqrt(sum x^2 + 1e-6) of section
"测试与验证体系"), written with torch fp64 tensors so that autograd gives the
vector-Jacobian product.  The gradients are those of the scalar

    L = sum_t <do_t, o_t> + sum_n <dht_n, ht_n>

with respect to q, k, v, g, beta and h0 (states in the [N, H, V, K] layout of
section "算子签名与 I/O 规格").  The pages name the backward kernels of the
training path but give no formulas for them; the plain definition of what they
compute is this vector-Jacobian product.

``normalise``, ``token_step`` and ``objective`` are separate so the tests can
plant a mistake in each.  Pins: ``tests/test_oracle_backward.py`` (central
finite differences of the C recurrence, closed forms, invariances).
"""

from __future__ import annotations

import numpy as np
import torch


def normalise(x):
    """Per-token L2 normalisation of the last axis with eps 1e-6 in the root."""
    return x / torch.sqrt((x * x).sum(-1, keepdim=True) + 1e-6)


def token_step(S, qt, kt, vt, gt, bt, scale):
    """One token for every head.  S: [H, K, V]; qt, kt, gt: [H, K]; vt: [H, V];
    bt: [H].  Returns (S after the token, o_t [H, V])."""
    S = S * torch.exp(gt)[:, :, None]
    pred = torch.einsum("hk,hkv->hv", kt, S)
    S = S + bt[:, None, None] * torch.einsum("hk,hv->hkv", kt, vt - pred)
    return S, torch.einsum("hk,hkv->hv", scale * qt, S)


def objective(o, ht, do, dht):
    """The scalar whose gradient is taken: <do, o> + <dht, ht>."""
    L = (o * do).sum()
    return L if dht is None else L + (ht * dht).sum()


def _forward(q, k, v, g, beta, scale, h0, bounds, l2norm):
    """q, k, g: [T, H, K]; v: [T, H, V]; beta: [T, H]; h0: [N, H, V, K].
    Returns (o [T, H, V], ht [N, H, V, K])."""
    T, H, K = q.shape
    V = v.shape[-1]
    outs = [None] * T
    finals = []
    for n, (bos, eos) in enumerate(bounds):
        S = h0[n].transpose(1, 2)
        for t in range(bos, eos):
            qt, kt = (normalise(q[t]), normalise(k[t])) if l2norm else (q[t], k[t])
            S, outs[t] = token_step(S, qt, kt, v[t], g[t], beta[t], scale)
        finals.append(S.transpose(1, 2))
    for t in range(T):                        # tokens outside every sequence
        if outs[t] is None:
            outs[t] = torch.zeros((H, V), dtype=torch.float64)
    o = torch.stack(outs) if T > 0 else torch.zeros((0, H, V), dtype=torch.float64)
    ht = torch.stack(finals) if finals else torch.zeros((0, H, V, K), dtype=torch.float64)
    return o, ht


def _bounds(B, T, cu_seqlens):
    if cu_seqlens is None:
        return [(n * T, (n + 1) * T) for n in range(B)]
    cu = [int(c) for c in cu_seqlens]
    return [(cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


def _flat(x, B, T):
    a = np.asarray(x, np.float64)
    return torch.tensor(a.reshape((B * T,) + a.shape[2:]))


def kda_forward_fp64(q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None, l2norm=False):
    """The forward alone (no gradients).  Shapes as ``kda_backward``;
    returns (o [B, T, H, V], ht [N, H, V, K]) as float64 numpy."""
    B, T, H, K = np.shape(q)
    V = np.shape(v)[-1]
    bounds = _bounds(B, T, cu_seqlens)
    h = torch.zeros((len(bounds), H, V, K), dtype=torch.float64) if h0 is None else \
        torch.tensor(np.asarray(h0, np.float64))
    with torch.no_grad():
        o, ht = _forward(*(_flat(x, B, T) for x in (q, k, v, g, beta)), K ** -0.5 if scale is None else scale,
                         h, bounds, l2norm)
    return o.reshape(B, T, H, V).numpy(), ht.numpy()


def kda_backward(q, k, v, g, beta, do, scale=None, h0=None, dht=None, cu_seqlens=None, l2norm=False):
    """Gradients (dq, dk, dv, dg, dbeta, dh0) of <do, o> + <dht, ht>, float64.

    q, k, g: [B, T, H, K]; v, do: [B, T, H, V]; beta: [B, T, H]; h0, dht:
    [N, H, V, K] or None (zero); cu_seqlens: N+1 offsets (B == 1) or None;
    scale None means K**-0.5.  dh0 is returned even when h0 is None (the
    gradient at a zero initial state).
    """
    B, T, H, K = np.shape(q)
    V = np.shape(v)[-1]
    bounds = _bounds(B, T, cu_seqlens)
    N = len(bounds)
    leaves = [_flat(x, B, T).requires_grad_(True) for x in (q, k, v, g, beta)]
    h = torch.tensor(np.zeros((N, H, V, K)) if h0 is None else np.asarray(h0, np.float64), requires_grad=True)
    o, ht = _forward(*leaves, K ** -0.5 if scale is None else scale, h, bounds, l2norm)
    L = objective(o, ht, _flat(do, B, T), None if dht is None else torch.tensor(np.asarray(dht, np.float64)))
    grads = torch.autograd.grad(L, leaves + [h], allow_unused=True)
    dq, dk, dv, dg, db, dh0 = (np.zeros(x.shape) if gr is None else gr.numpy() for x, gr in zip(leaves + [h], grads))
    return (dq.reshape(B, T, H, K), dk.reshape(B, T, H, K), dv.reshape(B, T, H, V), dg.reshape(B, T, H, K),
            db.reshape(B, T, H), dh0)
