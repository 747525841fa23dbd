"""Token-by-token KDA with an in-place state pool, fp64 (numpy).

TEST INFRASTRUCTURE ONLY: the oracle for the library's decode entry point
(``kda_fused_recurrent``).  It shares no code with the CUDA path; only tests,
the smoke check and the benchmark's CPU legs use it.

Page "PyPTO-Gym chunk_kda operator: an NPU forward of chunked gated delta-rule
linear attention":
  * section "算子定位与算法背景": the per-token update, in the K x V
    orientation: S <- diag(exp(g)) S; S <- S + beta k (v - S^T k)^T;
    o = S^T q (q multiplied by ``scale`` first, section "算法原理" M1);
  * section "算子签名与 I/O 规格": states are stored as [.., H, V, K], the
    transpose of the K x V state;
  * section "测试与验证体系": the optional q/k normalisation
    x / sqrt(sum(x^2) + 1e-6) over K;
  * section "与其他 KDA 算子的关系": fused_recurrent_kda steps an fp32 state
    per sequence one token at a time, in place at slots named by
    ``ssm_state_indices``, with speculative decoding via
    ``num_accepted_tokens``.  The page names these two arguments without
    defining them; the reading implemented here (and by the library) is:
      - no ``num_accepted_tokens``: sequence n starts from slot idx[n][0] and
        its final state is written back there; a negative slot is a padding
        entry (no state read or written, output rows zero);
      - with ``num_accepted_tokens``: sequence n starts from slot
        idx[n][num_accepted[n] - 1] and the state after its token t is stored
        at slot idx[n][t] (skipped where that slot is negative).

The helpers ``read_slot``, ``write_slots`` and ``token_step`` are separate so
that the tests can plant mistakes in each and check that a pin catches them.
"""

from __future__ import annotations

import numpy as np


def token_step(S, q, k, v, g, beta):
    """One token of the recurrence on the K x V state S (fp64, in place).
    Returns the output row o = S^T q after the update."""
    S *= np.exp(g)[:, None]                 # per-dimension decay
    pred = k @ S                            # S^T k
    S += beta * np.outer(k, v - pred)       # delta update
    return q @ S                            # read-out


def read_slot(row, num_accepted):
    """Slot the sequence's state is read from."""
    return int(row[0]) if num_accepted is None else int(row[num_accepted - 1])


def write_slots(row, num_accepted, L):
    """(token index, slot) pairs at which the state is stored: the final
    state only in plain decode, every token's state in speculative mode."""
    if num_accepted is None:
        return [(L - 1, int(row[0]))]
    return [(t, int(row[t])) for t in range(L)]


def _norm(x):
    return x / np.sqrt(np.sum(x * x) + 1e-6)


def fused_recurrent(q, k, v, g, beta, pool, indices, scale=None, num_accepted=None, cu_seqlens=None,
                    l2norm=False):
    """Run the decode recurrence.

    q, k [B,T,H,K]; v [B,T,H,V]; g [B,T,H,K]; beta [B,T,H]; pool [P,H,V,K];
    indices int [N] or [N, S]; num_accepted int [N] or None; cu_seqlens int
    [N+1] (B == 1) or None (N = B sequences of T tokens).
    Returns (o float64 [B,T,H,V], new pool float64 [P,H,V,K]).  Raises
    ValueError on a slot or accepted count out of range.
    """
    q, k, v, g = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g))
    beta = np.asarray(beta, dtype=np.float64)
    pool = np.array(pool, dtype=np.float64, copy=True)
    B, T, H, K = q.shape
    V = v.shape[-1]
    idx = np.asarray(indices).reshape(len(indices), -1)
    N = idx.shape[0]
    if scale is None:
        scale = K ** -0.5
    if cu_seqlens is None:
        if N != B:
            raise ValueError("fixed length needs one index row per batch entry")
        bounds = [(n * T, T) for n in range(N)]
    else:
        cu = [int(c) for c in cu_seqlens]
        bounds = [(cu[n], cu[n + 1] - cu[n]) for n in range(N)]
    P = pool.shape[0]
    qf, kf, vf, gf = (x.reshape(B * T, H, -1) for x in (q, k, v, g))
    bf = beta.reshape(B * T, H)
    o = np.zeros((B * T, H, V))
    for n, (bos, L) in enumerate(bounds):
        if L == 0:
            continue
        acc = None if num_accepted is None else int(num_accepted[n])
        row = idx[n]
        if acc is not None and not (1 <= acc <= len(row) and L <= len(row)):
            raise ValueError("accepted-token count out of range")
        rs = read_slot(row, acc)
        writes = dict(write_slots(row, acc, L))
        if rs >= P or any(s >= P for s in writes.values()):
            raise ValueError("state slot out of range")
        if rs < 0:
            continue
        for h in range(H):
            S = pool[rs, h].T.copy()          # [V,K] -> K x V
            for t in range(L):
                qt, kt = qf[bos + t, h], kf[bos + t, h]
                if l2norm:
                    qt, kt = _norm(qt), _norm(kt)
                o[bos + t, h] = token_step(S, scale * qt, kt, vf[bos + t, h], gf[bos + t, h], bf[bos + t, h])
                if t in writes and writes[t] >= 0:
                    pool[writes[t], h] = S.T
    return o.reshape(B, T, H, V), pool
