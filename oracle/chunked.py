"""Naive chunked KDA forward in fp64 (numpy) -- the oracle's second form.

TEST INFRASTRUCTURE ONLY.  Nothing under ``oracle/`` is used by the product
path; only tests, the smoke check and the benchmark's CPU-baseline leg call it.

This restates the four steps M1-M4 of the page "PyPTO-Gym chunk_kda operator:
an NPU forward of chunked gated delta-rule linear attention", section "算法原理" (algorithm), literally and without
blocking or fusion, so that it can be compared with the per-token recurrence
(``oracle.kda_recurrent``), which it must equal up to rounding order:

  M1  split the sequence into chunks of BT rows, multiply q by ``scale``, and
      take the inclusive prefix sum of g inside each chunk, written as a
      product with the inclusive lower-triangular all-ones matrix.
  M2  A_full[c, i] = sum_d k[c, d] k[i, d] exp(G[c, d] - G[i, d]); keep the
      strictly lower part, scale row c by beta[c], and invert (I + A) with an
      explicit triangular solve.
  M3  w = (I + A)^-1 diag(beta) (exp(G) * k),  u = (I + A)^-1 diag(beta) v.
  M4  v_new = u - w S;  o = (q * exp(G)) S + A2 v_new;
      S <- diag(exp(G_last)) S + (exp(G_last - G) * k)^T v_new.

Readings of the page taken here (the page is silent or terse on them):
  * beta enters w and u as diag(beta) on the right-hand side (the M3 formula is
    printed without beta; M2 puts beta on the rows of A).  This is the only
    placement under which M4's state update, which carries no beta, equals the
    per-token rule.
  * A2 (named in M4, not defined) is the inclusive lower-triangular q-k
    matrix A2[c, i] = sum_d qs[c, d] k[i, d] exp(G[c, d] - G[i, d]) for i <= c,
    because the per-token read-out happens after token t's own update.
  * The tail chunk of a sequence is zero-padded (q, k, v, g, beta all 0), per
    section "尾部 chunk 的零填充" (tail-chunk zero padding); padded rows
    produce no output.
"""

from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def _l2norm(x: np.ndarray) -> np.ndarray:
    """Per-row L2 normalisation with eps 1e-6 inside the root (section "测试与验证体系")."""
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + 1e-6)


def chunk_step(S, qs, k, v, g, beta, BT, return_terms=False):
    """One chunk of M1-M4 for one (sequence, head).

    S: (K, V) state entering the chunk.  qs, k: (L, K); v: (L, V); g: (L, K);
    beta: (L,), with L <= BT valid rows.  Returns (o (L, V), S_next (K, V)),
    and with ``return_terms`` also the two operands of M4's subtraction
    v_new = u - w S as a third element (u, w S).
    """
    L = qs.shape[0]
    K = k.shape[1]
    V = v.shape[1]

    def pad(x):
        out = np.zeros((BT,) + x.shape[1:], dtype=np.float64)
        out[:L] = x
        return out

    qs_, k_, v_, g_, b_ = pad(qs), pad(k), pad(v), pad(g), pad(beta)

    # M1: inclusive prefix sum as a product with tril(ones).
    tril_incl = np.tril(np.ones((BT, BT)))
    G = tril_incl @ g_                                   # (BT, K)

    # M2: A_full[c, i] = sum_d k_c,d k_i,d exp(G_c,d - G_i,d), only i <= c is
    # ever used; the exponent is masked above the diagonal so it cannot overflow.
    c_idx = np.arange(BT)[:, None]
    i_idx = np.arange(BT)[None, :]
    lower_incl = i_idx <= c_idx
    diff = G[:, None, :] - G[None, :, :]                  # (c, i, d)
    diff = np.where(lower_incl[:, :, None], diff, -np.inf)
    decay = np.exp(diff)
    A_full = np.einsum("cd,id,cid->ci", k_, k_, decay)
    A = np.where(i_idx < c_idx, A_full, 0.0) * b_[:, None]
    I = np.eye(BT)
    A_inv = solve_triangular(I + A, I, lower=True, unit_diagonal=True)

    # M3: WY projections with beta on the right-hand side.
    w = A_inv @ (b_[:, None] * np.exp(G) * k_)            # (BT, K)
    u = A_inv @ (b_[:, None] * v_)                        # (BT, V)

    # M4: inter-chunk recurrence and output.
    A2 = np.where(lower_incl, np.einsum("cd,id,cid->ci", qs_, k_, decay), 0.0)
    v_new = u - w @ S
    o = (qs_ * np.exp(G)) @ S + A2 @ v_new
    g_last = G[BT - 1]
    S_next = np.exp(g_last)[:, None] * S + (np.exp(g_last[None, :] - G) * k_).T @ v_new
    if return_terms:
        return o[:L], S_next, (u[:L], (w @ S)[:L])
    return o[:L], S_next


def cancellation_ratio(S, k, v, g, beta, BT=128):
    """How much of M4's subtraction v_new = u - w S cancels on one chunk:
    ||u - w S|| / max(||u||, ||w S||) (Frobenius norms; near 0 = severe
    cancellation).  Used to search for adversarial inputs (section "测试与验证
    体系": the input generator's cancellation_stress mode searches random
    scalings for this cancellation)."""
    K = k.shape[1]
    _, _, (u, wS) = chunk_step(S, np.zeros_like(k), k, v, g, beta, BT, return_terms=True)
    den = max(np.linalg.norm(u), np.linalg.norm(wS), 1e-300)
    return float(np.linalg.norm(u - wS) / den)


def kda_chunked(q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None,
                l2norm=False, BT=128, units=None):
    """Chunked KDA forward for all (or the selected) (sequence, head) units.

    Shapes follow the page's I/O table: q, k, g (B, T, H, K); v (B, T, H, V);
    beta (B, T, H); h0 (N, H, V, K) or None; cu_seqlens (N+1,) or None.
    ``units`` is an optional iterable of (n, h) pairs.  Returns
    (o (B, T, H, V) float64 with NaN for units not computed, ht (N, H, V, K)).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = K ** -0.5
    if cu_seqlens is None:
        N = B
        bounds = [(n, n * T, (n + 1) * T) for n in range(N)]
    else:
        assert B == 1
        cu = [int(x) for x in np.asarray(cu_seqlens)]
        N = len(cu) - 1
        bounds = [(n, cu[n], cu[n + 1]) for n in range(N)]
    qf = q.reshape(B * T, H, K)
    kf = k.reshape(B * T, H, K)
    vf = v.reshape(B * T, H, V)
    gf = g.reshape(B * T, H, K)
    bf = beta.reshape(B * T, H)
    o = np.full((B * T, H, V), np.nan)
    ht = np.full((N, H, V, K), np.nan)
    todo = set(units) if units is not None else {(n, h) for n in range(N) for h in range(H)}
    for n, bos, eos in bounds:
        for h in range(H):
            if (n, h) not in todo:
                continue
            S = np.zeros((K, V)) if h0 is None else np.asarray(h0[n, h], np.float64).T.copy()
            for s in range(bos, eos, BT):
                e = min(s + BT, eos)
                qq, kk = qf[s:e, h], kf[s:e, h]
                if l2norm:
                    qq, kk = _l2norm(qq), _l2norm(kk)
                o_c, S = chunk_step(S, scale * qq, kk, vf[s:e, h], gf[s:e, h], bf[s:e, h], BT)
                o[s:e, h] = o_c
            ht[n, h] = S.T
    return o.reshape(B, T, H, V), ht
