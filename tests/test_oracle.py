"""Pins for the fp64 oracle (CPU only).

The oracle is the definition the CUDA path is graded against, so it is pinned
here to things other than itself: closed forms of the per-token rule, the
delta rule's retrieval property, pure-decay special cases, a brute-force
expansion into explicit transition matrices, agreement between its two
independently written forms (per-token C recurrence and chunked numpy M1-M4),
varlen packing, head independence, and the chunk-boundary worked example of
the KCP debugging guide.  ``test_pins_catch_mutants`` shows that each pin
set fails for a family of plausible mistakes planted in a small numpy copy of
the recurrence.

Page cited throughout: "PyPTO-Gym chunk_kda operator: an NPU forward of
chunked gated delta-rule linear attention".
"""

import json
import os

import numpy as np
import pytest

import oracle
from oracle.chunked import chunk_step, kda_chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, shape, scale=1.0):
    return (scale * rng.standard_normal(shape)).astype(np.float32)


def _unit_rows(rng, shape):
    x = rng.standard_normal(shape)
    return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)


def _problem(seed, B=1, T=9, H=2, K=4, V=3, N=None, gate=0.3, with_h0=True):
    rng = np.random.default_rng(seed)
    q = _rand(rng, (B, T, H, K))
    k = _unit_rows(rng, (B, T, H, K))
    v = _rand(rng, (B, T, H, V))
    g = (-gate * np.abs(rng.standard_normal((B, T, H, K)))).astype(np.float32)
    beta = rng.uniform(0.05, 0.95, (B, T, H)).astype(np.float32)
    n = B if N is None else N
    h0 = _rand(rng, (n, H, V, K), 0.5) if with_h0 else None
    return q, k, v, g, beta, h0


# ---------------------------------------------------------------------------
# Pins, written against a generic runner so that mutants can be fed through
# the same checks.  run(q, k, v, g, beta, scale, h0, cu, l2norm) -> (o, ht).
# ---------------------------------------------------------------------------

def pin_single_token_closed_form(run):
    """T = 1, zero initial state: S = beta k v^T and o = beta * scale * (q.k) v,
    whatever the gate (the decay of a zero state is zero)."""
    q, k, v, g, beta, _ = _problem(1, T=1, H=1, K=5, V=4)
    scale = 0.37
    o, ht = run(q, k, v, g, beta, scale, None, None, False)
    qk = float(np.dot(q[0, 0, 0].astype(np.float64), k[0, 0, 0].astype(np.float64)))
    b = float(beta[0, 0, 0])
    o_ref = b * scale * qk * v[0, 0, 0].astype(np.float64)
    S_ref = b * np.outer(k[0, 0, 0].astype(np.float64), v[0, 0, 0].astype(np.float64))  # K x V
    return np.allclose(o[0, 0, 0], o_ref, rtol=1e-12, atol=1e-14) and \
        np.allclose(ht[0, 0], S_ref.T, rtol=1e-12, atol=1e-14)


def pin_retrieval(run):
    """Delta rule with g = 0, beta = 1 and unit keys: right after writing
    (k_t, v_t) the memory returns v_t for k_t, from any prior state; writing
    the same key again overwrites.  With q_t = k_t and scale = 1, o_t = v_t."""
    rng = np.random.default_rng(7)
    K, V, T = 6, 5, 7
    keys = _unit_rows(rng, (T, K))
    keys[4] = keys[1]                       # rewrite an earlier key
    q = keys[None, :, None, :].copy()
    k = keys[None, :, None, :].copy()
    v = _rand(rng, (1, T, 1, V))
    g = np.zeros((1, T, 1, K), np.float32)
    beta = np.ones((1, T, 1), np.float32)
    h0 = _rand(rng, (1, 1, V, K))
    o, ht = run(q, k, v, g, beta, 1.0, h0, None, False)
    ok = np.allclose(o[0, :, 0], v[0, :, 0], atol=2e-6)
    # after the last write of key 1 (t = 4), reading key 1 at the end returns
    # v_4 only if no later key interfered; check t = 6 directly instead:
    S_T = ht[0, 0].T                         # K x V
    ok &= np.allclose(S_T.T @ keys[6].astype(np.float64), v[0, 6, 0], atol=2e-6)
    return bool(ok)


def pin_pure_decay(run):
    """beta = 0: the state only decays, S_t = diag(exp(G_t)) S_0 with
    G_t = sum_{s<=t} g_s, and o_t = S_t^T (scale q_t).  h0 is not symmetric,
    so this also fixes the [V, K] layout of the state at the ABI."""
    q, k, v, g, beta, h0 = _problem(3, T=6, H=1, K=4, V=4)
    beta[:] = 0
    scale = 0.8
    o, ht = run(q, k, v, g, beta, scale, h0, None, False)
    G = np.cumsum(g[0, :, 0].astype(np.float64), axis=0)      # (T, K)
    S0 = h0[0, 0].astype(np.float64).T                         # K x V
    ok = True
    for t in range(6):
        St = np.exp(G[t])[:, None] * S0
        ok &= np.allclose(o[0, t, 0], St.T @ (scale * q[0, t, 0].astype(np.float64)),
                          rtol=1e-12, atol=1e-14)
    ok &= np.allclose(ht[0, 0], (np.exp(G[-1])[:, None] * S0).T, rtol=1e-12, atol=1e-14)
    return bool(ok)


def pin_frozen_state(run):
    """g = 0 and beta = 0: the state is unchanged and o_t = h0 (scale q_t),
    with h0 in its [V, K] layout."""
    q, k, v, g, beta, h0 = _problem(4, T=5, H=1, K=4, V=4)
    g[:] = 0
    beta[:] = 0
    o, ht = run(q, k, v, g, beta, 0.5, h0, None, False)
    ok = np.array_equal(ht[0, 0], h0[0, 0].astype(np.float64))
    for t in range(5):
        ok &= np.allclose(o[0, t, 0], h0[0, 0].astype(np.float64) @ (0.5 * q[0, t, 0]),
                          rtol=1e-12, atol=1e-14)
    return bool(ok)


def pin_l2norm_eps(run):
    """The in-kernel normalisation divides by sqrt(sum x^2 + 1e-6): for a
    vector with sum x^2 = 1e-6 the factor is exactly 1/sqrt(2e-6).  T = 1,
    zero state, so o = beta * scale * (qn . kn) v."""
    K, V = 4, 2
    q = np.zeros((1, 1, 1, K), np.float32)
    q[..., 0] = 1e-3                       # sum q^2 = 1e-6
    k = np.zeros((1, 1, 1, K), np.float32)
    k[..., 0] = 2.0                        # sum k^2 = 4
    v = np.array([1.0, -2.0], np.float32).reshape(1, 1, 1, V)
    g = np.zeros((1, 1, 1, K), np.float32)
    beta = np.full((1, 1, 1), 0.5, np.float32)
    o, _ = run(q, k, v, g, beta, 1.0, None, None, True)
    qn = np.float64(np.float32(1e-3)) / np.sqrt(np.float64(np.float32(1e-3)) ** 2 + 1e-6)
    kn = 2.0 / np.sqrt(4.0 + 1e-6)
    o_ref = 0.5 * qn * kn * np.array([1.0, -2.0])
    return bool(np.allclose(o[0, 0, 0], o_ref, rtol=1e-12))


PINS = [pin_single_token_closed_form, pin_retrieval, pin_pure_decay,
        pin_frozen_state, pin_l2norm_eps]


def _oracle_run(q, k, v, g, beta, scale, h0, cu, l2norm):
    return oracle.kda_recurrent(q, k, v, g, beta, scale=scale, h0=h0, cu_seqlens=cu,
                                l2norm=l2norm)


def _chunked_run(BT):
    def run(q, k, v, g, beta, scale, h0, cu, l2norm):
        return kda_chunked(q, k, v, g, beta, scale=scale, h0=h0, cu_seqlens=cu,
                           l2norm=l2norm, BT=BT)
    return run


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_recurrent_oracle_pins(pin):
    assert pin(_oracle_run)


@pytest.mark.parametrize("BT", [1, 2, 4, 16, 128])
@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_chunked_oracle_pins(pin, BT):
    assert pin(_chunked_run(BT))


# ---------------------------------------------------------------------------
# Brute force: explicit transition matrices on tiny problems.
# ---------------------------------------------------------------------------

def _brute_force(q, k, v, g, beta, scale, h0):
    """S_t = M_t S_{t-1} + beta_t k_t v_t^T with M_t = (I - beta_t k_t k_t^T)
    diag(exp(g_t)) -- the per-token rule written as an affine map of the whole
    state -- and o_t = S_t^T (scale q_t).  Products of the M_t, not rank-1
    loops, so an index slip in the oracle's loops shows up."""
    _, T, H, K = q.shape
    V = v.shape[-1]
    o = np.zeros((1, T, H, V))
    ht = np.zeros((1, H, V, K))
    for h in range(H):
        S0 = np.zeros((K, V)) if h0 is None else h0[0, h].astype(np.float64).T
        Ms, Bs = [], []
        for t in range(T):
            kt = k[0, t, h].astype(np.float64)
            Mt = (np.eye(K) - beta[0, t, h] * np.outer(kt, kt)) @ np.diag(np.exp(g[0, t, h].astype(np.float64)))
            Ms.append(Mt)
            Bs.append(beta[0, t, h] * np.outer(kt, v[0, t, h].astype(np.float64)))
        for t in range(T):
            # S_t = (M_t ... M_0) S0 + sum_{s<=t} (M_t ... M_{s+1}) B_s
            P = np.eye(K)
            St = np.zeros((K, V))
            for s in range(t, -1, -1):
                St += P @ Bs[s]
                P = P @ Ms[s]
            St += P @ S0
            o[0, t, h] = St.T @ (scale * q[0, t, h].astype(np.float64))
            if t == T - 1:
                ht[0, h] = St.T
    return o, ht


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_expansion(seed):
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(1, 9))
    K = int(rng.integers(1, 5))
    V = int(rng.integers(1, 5))
    q, k, v, g, beta, h0 = _problem(200 + seed, T=T, H=2, K=K, V=V)
    if seed % 2:
        h0 = None
    scale = float(rng.uniform(0.2, 1.5))
    o_ref, ht_ref = _brute_force(q, k, v, g, beta, scale, h0)
    o, ht = oracle.kda_recurrent(q, k, v, g, beta, scale=scale, h0=h0)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(ht, ht_ref, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------------------
# The two forms agree (chunked re-association == per-token rule).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("BT", [1, 2, 4, 16, 128])
@pytest.mark.parametrize("T", [7, 37, 129, 300])
def test_chunked_equals_recurrent(BT, T):
    q, k, v, g, beta, h0 = _problem(T * 1000 + BT, B=2, T=T, H=2, K=8, V=6)
    o_r, ht_r = oracle.kda_recurrent(q, k, v, g, beta, h0=h0)
    o_c, ht_c = kda_chunked(q, k, v, g, beta, h0=h0, BT=BT)
    np.testing.assert_allclose(o_c, o_r, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ht_c, ht_r, rtol=1e-10, atol=1e-12)


def test_chunked_equals_recurrent_varlen_strong_gates():
    """Varlen with tails of every kind and gates far stronger than the named
    workloads (cumulative decay of tens of nats inside a chunk)."""
    cu = [0, 1, 130, 130, 257, 400]
    T = cu[-1]
    q, k, v, g, beta, h0 = _problem(55, B=1, T=T, H=2, K=8, V=4, N=len(cu) - 1, gate=1.5)
    o_r, ht_r = oracle.kda_recurrent(q, k, v, g, beta, h0=h0, cu_seqlens=cu, l2norm=True)
    o_c, ht_c = kda_chunked(q, k, v, g, beta, h0=h0, cu_seqlens=cu, l2norm=True, BT=64)
    np.testing.assert_allclose(o_c, o_r, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ht_c, ht_r, rtol=1e-10, atol=1e-12)


def test_chunked_equals_recurrent_tiny_workload():
    """The tiny named workload (B=1, T=256, H=1, K=V=128) at BT = 128."""
    import torch
    from chunked_gated_delta_kda_gb300.inputs import WORKLOADS, make_inputs
    x = make_inputs(WORKLOADS["tiny"])
    args = [x[n].float().numpy() for n in ("q", "k", "v", "g", "beta")]
    o_r, ht_r = oracle.kda_recurrent(*args)
    o_c, ht_c = kda_chunked(*args, BT=128)
    np.testing.assert_allclose(o_c, o_r, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(ht_c, ht_r, rtol=1e-9, atol=1e-12)
    assert torch.isfinite(torch.from_numpy(o_r)).all()


def test_inverse_identity():
    """(I + A) (I + A)^-1 = I inside the chunked form, and beta = 0 gives
    (I + A)^-1 = I so w = 0, u = 0."""
    rng = np.random.default_rng(9)
    L, K, V, BT = 20, 8, 5, 32
    qs = rng.standard_normal((L, K))
    k = rng.standard_normal((L, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((L, V))
    g = -0.2 * np.abs(rng.standard_normal((L, K)))
    S = rng.standard_normal((K, V))
    # beta = 0: state only decays, output is the gated read-out alone
    o, S1 = chunk_step(S, qs, k, v, g, np.zeros(L), BT)
    G = np.cumsum(g, axis=0)
    np.testing.assert_allclose(S1, np.exp(G[-1])[:, None] * S, rtol=1e-13)
    np.testing.assert_allclose(o, (qs * np.exp(G)) @ S, rtol=1e-12)


# ---------------------------------------------------------------------------
# Packing and independence.
# ---------------------------------------------------------------------------

def test_varlen_equals_per_sequence():
    lens = [5, 0, 17, 1, 30]
    cu = np.cumsum([0] + lens).tolist()
    T = cu[-1]
    q, k, v, g, beta, h0 = _problem(77, B=1, T=T, H=3, K=6, V=5, N=len(lens))
    o, ht = oracle.kda_recurrent(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    for n, L in enumerate(lens):
        s, e = cu[n], cu[n + 1]
        if L == 0:
            np.testing.assert_array_equal(ht[n], h0[n].astype(np.float64))
            continue
        o1, ht1 = oracle.kda_recurrent(q[:, s:e], k[:, s:e], v[:, s:e], g[:, s:e],
                                       beta[:, s:e], h0=h0[n:n + 1])
        np.testing.assert_array_equal(o[:, s:e], o1)
        np.testing.assert_array_equal(ht[n], ht1[0])


def test_fixed_equals_uniform_varlen():
    q, k, v, g, beta, h0 = _problem(78, B=3, T=11, H=2, K=4, V=4)
    o_f, ht_f = oracle.kda_recurrent(q, k, v, g, beta, h0=h0)
    flat = [x.reshape((1, 33) + x.shape[2:]) for x in (q, k, v, g, beta)]
    o_v, ht_v = oracle.kda_recurrent(*flat, h0=h0, cu_seqlens=[0, 11, 22, 33])
    np.testing.assert_array_equal(o_v.reshape(o_f.shape), o_f)
    np.testing.assert_array_equal(ht_v, ht_f)


def test_heads_independent_and_unit_selection():
    q, k, v, g, beta, h0 = _problem(79, B=1, T=12, H=3, K=4, V=4)
    o, ht = oracle.kda_recurrent(q, k, v, g, beta, h0=h0)
    q2, v2 = q.copy(), v.copy()
    q2[:, :, 1] += 1.0
    v2[:, :, 2] *= -3.0
    o2, ht2 = oracle.kda_recurrent(q2, k, v2, g, beta, h0=h0)
    np.testing.assert_array_equal(o2[:, :, 0], o[:, :, 0])
    np.testing.assert_array_equal(ht2[:, 0], ht[:, 0])
    o3, ht3 = oracle.kda_recurrent(q, k, v, g, beta, h0=h0, units=[(0, 2)])
    np.testing.assert_array_equal(o3[:, :, 2], o[:, :, 2])
    assert np.isnan(o3[:, :, 0]).all()


def test_bad_cu_rejected():
    q, k, v, g, beta, _ = _problem(80, B=1, T=10, H=1, K=4, V=4)
    with pytest.raises(ValueError):
        oracle.kda_recurrent(q, k, v, g, beta, cu_seqlens=[0, 6, 4, 10])
    with pytest.raises(ValueError):
        oracle.kda_recurrent(q, k, v, g, beta, cu_seqlens=[0, 6, 9])


def test_kcp_chunk_boundary_worked_example():
    """The KCP debugging guide's worked example (lengths [400, 624], chunk 64):
    the single-device path cuts sequence 1 at global tokens 400, 464, 528,
    592, ...  The oracle's chunked form walks each sequence from its own start
    in steps of BT; this pins that walk to the printed boundaries."""
    with open(os.path.join(GOLDEN, "kcp_chunk_boundaries.json")) as f:
        gold = json.load(f)
    cu = np.cumsum([0] + gold["lengths"]).tolist()
    BT = gold["chunk_size"]
    seq = gold["sequence"]
    starts = list(range(cu[seq], cu[seq + 1], BT))
    assert starts[:len(gold["global_chunk_starts"])] == gold["global_chunk_starts"]
    # rank 1's local slice [0, 512) of sequence 1 starts at global 512 and is
    # cut at 512, 576, 640, ... -- none of which is a boundary of the
    # single-device walk after 464, the guide's point about per-chunk compares.
    r1 = list(range(gold["rank1_global_start"], cu[seq + 1], BT))
    assert r1[:3] == gold["rank1_global_chunk_starts"]
    assert not set(r1) & set(s for s in starts if s > 464)


# ---------------------------------------------------------------------------
# The pins catch planted mistakes (mutants of a small numpy recurrence).
# ---------------------------------------------------------------------------

def _mutant(kind):
    def run(q, k, v, g, beta, scale, h0, cu, l2norm):
        assert cu is None
        B, T, H, K = q.shape
        V = v.shape[-1]
        o = np.zeros((B, T, H, V))
        ht = np.zeros((B, H, V, K))
        for b in range(B):
            for h in range(H):
                S = np.zeros((K, V)) if h0 is None else h0[b, h].astype(np.float64)
                if kind != "h0_not_transposed" and h0 is not None:
                    S = S.T.copy()
                for t in range(T):
                    x_q = q[b, t, h].astype(np.float64)
                    x_k = k[b, t, h].astype(np.float64)
                    if l2norm:
                        if kind == "eps_outside_sqrt":
                            x_q = x_q / (np.sqrt(x_q @ x_q) + 1e-6)
                            x_k = x_k / (np.sqrt(x_k @ x_k) + 1e-6)
                        else:
                            x_q = x_q / np.sqrt(x_q @ x_q + 1e-6)
                            x_k = x_k / np.sqrt(x_k @ x_k + 1e-6)
                    sgn = -1.0 if kind == "exp_neg_g" else 1.0
                    a = np.exp(sgn * g[b, t, h].astype(np.float64))
                    bt = 1.0 if kind == "no_beta" else float(beta[b, t, h])
                    vt = v[b, t, h].astype(np.float64)
                    if kind == "readout_first":
                        o[b, t, h] = S.T @ (scale * x_q)
                    if kind != "decay_after_delta":
                        S = a[:, None] * S
                    delta = vt - S.T @ x_k
                    if kind == "delta_sign":
                        delta = -delta
                    S = S + bt * np.outer(x_k, delta)
                    if kind == "decay_after_delta":
                        S = a[:, None] * S
                    if kind != "readout_first":
                        s_eff = 1.0 if kind == "no_scale" else scale
                        o[b, t, h] = S.T @ (s_eff * x_q)
                ht[b, h] = S.T
        return o, ht
    return run


MUTANTS = ["decay_after_delta", "no_beta", "delta_sign", "h0_not_transposed",
           "no_scale", "readout_first", "exp_neg_g", "eps_outside_sqrt"]


def test_mutant_harness_is_faithful():
    """With no mutation the numpy copy passes every pin."""
    assert all(p(_mutant("none")) for p in PINS)


def _passes(pin, run):
    try:
        return bool(pin(run))
    except (ValueError, FloatingPointError):
        return False


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_mutants(kind):
    failed = [p.__name__ for p in PINS if not _passes(p, _mutant(kind))]
    assert failed, f"no pin catches mutant {kind}"


# ---------------------------------------------------------------------------
# The two operands of M4's subtraction (u and w S) and the cancellation ratio
# built on them (section "测试与验证体系": the cancellation_stress search).
#
# Unrolling the per-token rule inside one chunk gives the meaning of
# v_new = u - w S without any chunked algebra: with the decayed state
# S'_t = diag(exp(g_t)) S_{t-1}, the per-token rule adds k_t d_t^T where
#   d_t = beta_t (v_t - S'_t^T k_t),
# so S_T = diag(exp(G_T)) S_0 + sum_t diag(exp(G_T - G_t)) k_t d_t^T, which is
# M4's state update with v_new[t] = d_t.  Hence, recorded from a plain
# token loop: u - w S = d (any S_0), u = d at S_0 = 0 (u does not depend on
# S_0), and w S = u - d.  With beta = 0 both operands vanish.
# ---------------------------------------------------------------------------

def _token_deltas(S0, k, v, g, beta):
    """d_t of the per-token rule over one chunk (plain loop, fp64)."""
    S = np.array(S0, dtype=np.float64)
    d = np.zeros((k.shape[0], v.shape[1]))
    for t in range(k.shape[0]):
        S = np.exp(g[t])[:, None] * S
        d[t] = beta[t] * (v[t] - S.T @ k[t])
        S = S + np.outer(k[t], d[t])
    return d


def _terms_problem(seed, L=23, K=6, V=6):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((L, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((L, V))
    g = -0.3 * np.abs(rng.standard_normal((L, K)))
    beta = rng.uniform(0.1, 0.9, L)
    S = rng.standard_normal((K, V))
    return S, k, v, g, beta


def pin_terms(step):
    """u and w S returned by ``step`` (a chunk_step-like callable) against the
    token deltas; also the ratio helper built from them."""
    S, k, v, g, beta = _terms_problem(5)
    qs = np.zeros_like(k)
    BT = 32
    _, _, (u0, wS0) = step(np.zeros_like(S), qs, k, v, g, beta, BT, return_terms=True)
    _, _, (u, wS) = step(S, qs, k, v, g, beta, BT, return_terms=True)
    d0 = _token_deltas(np.zeros_like(S), k, v, g, beta)
    d = _token_deltas(S, k, v, g, beta)
    ok = np.allclose(u0, d0, rtol=0, atol=1e-12) and np.allclose(wS0, 0.0, atol=1e-12)
    ok = ok and np.allclose(u, d0, rtol=0, atol=1e-12)
    ok = ok and np.allclose(wS, d0 - d, rtol=0, atol=1e-12)
    ok = ok and np.allclose(u - wS, d, rtol=0, atol=1e-12)
    _, _, (ub, wSb) = step(S, qs, k, v, g, np.zeros_like(beta), BT, return_terms=True)
    ok = ok and np.array_equal(ub, np.zeros_like(ub)) and np.array_equal(wSb, np.zeros_like(wSb))
    return bool(ok)


def test_cancellation_terms_equal_token_deltas():
    assert pin_terms(chunk_step)


def test_cancellation_terms_with_tail_and_full_chunk():
    """The same identity on a ragged tail (L < BT) and on a full 128-row chunk."""
    for L, BT in ((37, 128), (128, 128)):
        S, k, v, g, beta = _terms_problem(6 + L, L=L, K=8, V=5)
        _, _, (u, wS) = chunk_step(S, np.zeros_like(k), k, v, g, beta, BT, return_terms=True)
        np.testing.assert_allclose(u - wS, _token_deltas(S, k, v, g, beta), rtol=0, atol=1e-11)


def test_cancellation_ratio_value():
    """cancellation_ratio = ||d|| / max(||u||, ||u - d||) with u the deltas
    from a zero state and d those from S; 0 when v is chosen so that every
    token's prediction is exact (d = 0 with S = 0, v = 0)."""
    from oracle.chunked import cancellation_ratio
    S, k, v, g, beta = _terms_problem(8)
    d0 = _token_deltas(np.zeros_like(S), k, v, g, beta)
    d = _token_deltas(S, k, v, g, beta)
    want = np.linalg.norm(d) / max(np.linalg.norm(d0), np.linalg.norm(d0 - d))
    assert abs(cancellation_ratio(S, k, v, g, beta, BT=32) - want) < 1e-12
    assert cancellation_ratio(np.zeros_like(S), k, np.zeros_like(v), g, beta, BT=32) == 0.0


def _terms_mutant(kind):
    """chunk_step with a plausible mistake planted in its returned terms."""
    def step(S, qs, k, v, g, beta, BT, return_terms=False):
        o, S1, (u, wS) = chunk_step(S, qs, k, v, g, beta, BT, return_terms=True)
        if kind == "w_not_times_S":
            # w itself instead of w S (K == V here, so the shapes agree)
            _, _, (_, w) = chunk_step(np.eye(S.shape[0]), qs, k, v, g, beta, BT, return_terms=True)
            wS = w
        elif kind == "wS_sign":
            wS = -wS
        elif kind == "u_without_inverse":
            u = beta[:, None] * v
        elif kind == "terms_swapped":
            u, wS = wS, u
        return o, S1, (u, wS)
    return step


@pytest.mark.parametrize("kind", ["w_not_times_S", "wS_sign", "u_without_inverse", "terms_swapped"])
def test_terms_pin_catches_mutants(kind):
    assert not pin_terms(_terms_mutant(kind))
