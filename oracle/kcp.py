"""Kimi Context Parallel (KCP) forward, simulated rank by rank, fp64.

TEST INFRASTRUCTURE ONLY: the oracle of the library's KCP entry point
(``kda_kcp_fwd``).  It shares no code with the CUDA path; it composes the C
per-token recurrence (``kda_recurrent``) in the KCP structure.

Page "flash-linear-attention KCP precision-debugging guide":
  * section "背景：KCP 调试的特殊性": KCP cuts the sequence dimension across
    ranks; each rank processes its local tokens; a pre-process computes the
    transition M and the accumulated state S_ext, and a merge chains the
    ranks' contributions;
  * section "h与dh的跨 rank 语义": the merge of rank r yields the initial state
    of its first local sequence (the state at the first token it owns);
  * section "陷阱 4": the forward pre-process works on the rank's LAST local
    piece (the one whose tail passes to rank r + 1).
Reading used where the page leaves it open: rank r owns the packed tokens
[T r / W, T (r + 1) / W) (integer division); the state leaving a rank is
M_r S_start + S_ext,r with M_r the linear map of the last piece's
recurrence (obtained by running it with v = 0 from the identity, so that in
the [V, K] layout it is M_r^T) and S_ext,r its state from a zero start.

``merge`` and ``piece_initial`` are separate so the tests can plant mistakes.
"""

from __future__ import annotations

import numpy as np


def rank_bounds(T, W):
    return [T * r // W for r in range(W + 1)]


def pieces(cu, T, W):
    """Per rank, the (sequence, a, b) pieces of the sequences it owns."""
    b = rank_bounds(T, W)
    out = []
    for r in range(W):
        pr = []
        for n in range(len(cu) - 1):
            a0, b0 = max(cu[n], b[r]), min(cu[n + 1], b[r + 1])
            if a0 < b0:
                pr.append((n, a0, b0))
        out.append(pr)
    return out


def merge(start_vk, mt_vk, ext_vk):
    """State leaving a rank, [H, V, K] layout: S_start^T M^T + S_ext^T."""
    if start_vk is None:
        return ext_vk.copy()
    return np.einsum("hvj,hjk->hvk", start_vk, mt_vk) + ext_vk


def piece_initial(n, a, cu, h0, incoming):
    """Initial state of a local piece: the merged incoming state when the
    piece continues its sequence from an earlier rank, else the sequence's
    own initial state (or None for zero)."""
    if a > cu[n]:
        return incoming
    return None if h0 is None else h0[n]


def kcp_forward(q, k, v, g, beta, cu_seqlens, world_size, scale=None, h0=None, l2norm=False):
    """q, k, g: [1,T,H,K]; v: [1,T,H,V]; beta: [1,T,H]; cu_seqlens: N+1
    offsets; h0: [N,H,V,K] or None.  Returns (o float64 [1,T,H,V],
    ht float64 [N,H,V,K])."""
    from . import kda_recurrent
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    _, T, H, K = q.shape
    V = v.shape[-1]
    cu = [int(c) for c in cu_seqlens]
    N = len(cu) - 1
    W = int(world_size)
    h0 = None if h0 is None else np.asarray(h0, dtype=np.float64)
    pc = pieces(cu, T, W)

    def run(a, b, vv, init):
        sl = slice(a, b)
        return kda_recurrent(q[:, sl], k[:, sl], vv, g[:, sl], beta[:, sl], scale=scale,
                             h0=None if init is None else init[None], cu_seqlens=[0, b - a], l2norm=l2norm)

    # pre-process: every rank whose last piece continues into the next rank
    carry = {}
    for r in range(W - 1):
        if not pc[r]:
            continue
        n, a, b = pc[r][-1]
        if b >= cu[n + 1]:
            continue
        eye = np.broadcast_to(np.eye(K), (H, K, K)).copy()
        _, mt = run(a, b, np.zeros((1, b - a, H, K)), eye)    # V = K probe: M^T in [V, K] layout
        _, ext = run(a, b, v[:, a:b], None)
        carry[r] = (n, a, mt[0], ext[0])

    # merge in rank order
    incoming = [None] * W
    for r in range(W - 1):
        if not pc[r]:
            incoming[r + 1] = incoming[r]
            continue
        if r not in carry:
            continue
        n, a, mt, ext = carry[r]
        start = piece_initial(n, a, cu, h0, incoming[r])
        incoming[r + 1] = merge(start, mt, ext)

    # local forwards
    o = np.zeros((1, T, H, V))
    ht = np.zeros((N, H, V, K))
    for n in range(N):
        if cu[n] == cu[n + 1] and h0 is not None:
            ht[n] = h0[n]
    for r in range(W):
        for n, a, b in pc[r]:
            init = piece_initial(n, a, cu, h0, incoming[r])
            o_p, ht_p = run(a, b, v[:, a:b], init)
            o[:, a:b] = o_p
            if b == cu[n + 1]:
                ht[n] = ht_p[0]
    return o, ht
