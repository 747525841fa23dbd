"""Pins of the gradient oracle (``oracle.backward``), CPU only.

The gradient oracle differentiates the per-token recurrence with fp64 torch
autograd.  It is pinned to things other than itself:
  * its forward equals the C recurrence (``kda_recurrent``, pinned in
    ``test_oracle.py``; the two share no code);
  * every gradient equals a central finite difference of the C recurrence
    (Richardson-extrapolated; inputs on a dyadic grid so that the
    perturbed values are exact in the C recurrence's float32 inputs);
  * closed forms derived by hand: one token from a given state, and a frozen
    state (beta = 0, g = 0);
  * the chain rule across a split point (the state gradient carried from the
    tail of a sequence into its head), which is how a chunked backward
    composes, and independence of packed sequences;
  * with q/k normalisation, each dq_t / dk_t is orthogonal to q_t / k_t up
    to the eps in the root (the page "PyPTO-Gym chunk_kda operator", section
    "测试与验证体系", normalises per token).
``test_pins_catch_planted_mistakes`` plants a mistake in each piece of the
oracle in turn and checks that at least one pin fails.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import backward as bw

GRID = 64.0                  # inputs are multiples of 1/64
H_FD = 2.0 ** -9             # finite-difference steps h and h/2 stay on a 2^-10 grid


def _dyadic(rng, shape, scale=1.0):
    return np.round(scale * rng.standard_normal(shape) * GRID) / GRID


def _problem(seed, lens=(4, 3), B=None, H=2, K=3, V=2, h0=True, dht=True):
    rng = np.random.default_rng(seed)
    if B is None:
        B, T = 1, int(sum(lens))
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        N = len(lens)
    else:
        T, cu, N = int(lens), None, B
    x = dict(q=_dyadic(rng, (B, T, H, K)), k=_dyadic(rng, (B, T, H, K), 0.7),
             v=_dyadic(rng, (B, T, H, V)),
             g=-np.abs(_dyadic(rng, (B, T, H, K), 0.3)),
             beta=np.round(rng.uniform(0.05, 0.95, (B, T, H)) * GRID) / GRID,
             h0=_dyadic(rng, (N, H, V, K), 0.5) if h0 else None, cu=cu)
    x["do"] = rng.standard_normal((B, T, H, V))
    x["dht"] = rng.standard_normal((N, H, V, K)) if dht else None
    return x


def _grads(x, l2norm=False):
    return bw.kda_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], h0=x["h0"], dht=x["dht"],
                           cu_seqlens=x["cu"], l2norm=l2norm)


def _loss_c(x, l2norm):
    o, ht = oracle.kda_recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], cu_seqlens=x["cu"],
                                 l2norm=l2norm)
    L = float(np.sum(o * x["do"]))
    return L if x["dht"] is None else L + float(np.sum(ht * x["dht"]))


def _fd(x, name, l2norm):
    """Richardson-extrapolated central differences of the C recurrence's
    objective with respect to every element of x[name]."""
    base = x[name]
    out = np.zeros(base.shape)
    for i in np.ndindex(base.shape):
        d = []
        for h in (H_FD, H_FD / 2):
            vals = []
            for s in (1, -1):
                y = dict(x)
                y[name] = base.copy()
                y[name][i] += s * h
                vals.append(_loss_c(y, l2norm))
            d.append((vals[0] - vals[1]) / (2 * h))
        out[i] = (4 * d[1] - d[0]) / 3
    return out


def _close(a, b, tol):
    return bool(np.all(np.abs(a - b) <= tol * (1 + np.abs(b))))


# ---------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------

def pin_forward_is_the_recurrence():
    ok = True
    for l2 in (False, True):
        for x in (_problem(1), _problem(2, lens=5, B=2)):
            o, ht = bw.kda_forward_fp64(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"],
                                        cu_seqlens=x["cu"], l2norm=l2)
            o_c, ht_c = oracle.kda_recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"],
                                             cu_seqlens=x["cu"], l2norm=l2)
            ok &= _close(o, o_c, 1e-12) and _close(ht, ht_c, 1e-12)
    return bool(ok)


def pin_finite_differences():
    """All six gradients against central differences of the C recurrence."""
    ok = True
    for l2, x in ((False, _problem(3)), (True, _problem(4)), (False, _problem(5, lens=3, B=2, dht=False))):
        grads = _grads(x, l2)
        for name, gr in zip(("q", "k", "v", "g", "beta", "h0"), grads):
            if x[name] is None:
                continue
            ok &= _close(gr, _fd(x, name, l2), 1e-8)
    return bool(ok)


def pin_single_token_closed_form():
    """One token from h0 (hand-derived chain rule).  With A = D S0 (D =
    diag(exp g), S0 = h0^T), r = v - A^T k, S1 = A + beta k r^T,
    o = scale S1^T q and G = dL/dS1 = scale q do^T + dht^T:
    dq = scale S1 do, dv = beta G^T k, dbeta = k^T G r,
    dk = beta G r - beta A G^T k, dA = (I - beta k k^T) G,
    dg = rowsum(dA * A), dh0 = (D dA)^T."""
    x = _problem(6, lens=(1,), H=1, K=4, V=3)
    dq, dk, dv, dg, db, dh0 = _grads(x)
    q, k, v, g, b = x["q"][0, 0, 0], x["k"][0, 0, 0], x["v"][0, 0, 0], x["g"][0, 0, 0], x["beta"][0, 0, 0]
    sc = 4 ** -0.5
    S0 = x["h0"][0, 0].T
    A = np.exp(g)[:, None] * S0
    r = v - A.T @ k
    S1 = A + b * np.outer(k, r)
    G = sc * np.outer(q, x["do"][0, 0, 0]) + x["dht"][0, 0].T
    dA = (np.eye(4) - b * np.outer(k, k)) @ G
    return all([
        _close(dq[0, 0, 0], sc * S1 @ x["do"][0, 0, 0], 1e-12),
        _close(dv[0, 0, 0], b * G.T @ k, 1e-12),
        _close(db[0, 0, 0], k @ G @ r, 1e-12),
        _close(dk[0, 0, 0], b * G @ r - b * A @ G.T @ k, 1e-12),
        _close(dg[0, 0, 0], np.sum(dA * A, axis=1), 1e-12),
        _close(dh0[0, 0], (np.exp(g)[:, None] * dA).T, 1e-12),
    ])


def pin_frozen_state_closed_form():
    """beta = 0, g = 0: S stays S0 = h0^T.  Then dq_t = scale S0 do_t,
    dk = dv = 0, dh0 = (sum_s scale q_s do_s^T + dht^T)^T,
    dg_t = rowsum(S0 * R_t) and dbeta_t = k_t^T R_t (v_t - S0^T k_t) with
    R_t = sum_{s >= t} scale q_s do_s^T + dht^T."""
    x = _problem(7, lens=(5,), H=1, K=3, V=2)
    x["beta"] = np.zeros_like(x["beta"])
    x["g"] = np.zeros_like(x["g"])
    dq, dk, dv, dg, db, dh0 = _grads(x)
    sc = 3 ** -0.5
    S0 = x["h0"][0, 0].T
    q, k, v, do = (x[n][0, :, 0] for n in ("q", "k", "v", "do"))
    ok = _close(dk, 0 * dk, 0) and _close(dv, 0 * dv, 0)
    R = x["dht"][0, 0].T.copy()
    for t in range(4, -1, -1):
        R = R + sc * np.outer(q[t], do[t])
        ok &= _close(dq[0, t, 0], sc * S0 @ do[t], 1e-12)
        ok &= _close(dg[0, t, 0], np.sum(S0 * R, axis=1), 1e-12)
        ok &= _close(db[0, t, 0], k[t] @ R @ (v[t] - S0.T @ k[t]), 1e-12)
    ok &= _close(dh0[0, 0], R.T, 1e-12)
    return bool(ok)


def pin_state_gradient_chains():
    """Split one sequence at token m: the tail's dh0 (from the forward state
    at m) is the head's dht, and the two pieces' gradients are the whole's."""
    x = _problem(8, lens=(7,), H=2)
    m = 3
    full = _grads(x)
    head = {key: (val[:, :m] if key in ("q", "k", "v", "g", "beta", "do") else val) for key, val in x.items()}
    head["cu"] = np.array([0, m])
    tail = {key: (val[:, m:] if key in ("q", "k", "v", "g", "beta", "do") else val) for key, val in x.items()}
    tail["cu"] = np.array([0, 7 - m])
    _, S_m = bw.kda_forward_fp64(head["q"], head["k"], head["v"], head["g"], head["beta"], h0=x["h0"],
                                 cu_seqlens=head["cu"])
    tail["h0"] = S_m
    g_tail = _grads(tail)
    head["dht"] = g_tail[5]
    g_head = _grads(head)
    ok = True
    for i in range(5):
        ok &= _close(np.concatenate([g_head[i], g_tail[i]], axis=1), full[i], 1e-12)
    return bool(ok and _close(g_head[5], full[5], 1e-12))


def pin_sequences_independent():
    """Packed sequences have the gradients they have alone."""
    x = _problem(9, lens=(3, 0, 4), H=2)
    full = _grads(x)
    ok = True
    cu = x["cu"]
    for n in range(3):
        a, b = int(cu[n]), int(cu[n + 1])
        y = {key: (val[:, a:b] if key in ("q", "k", "v", "g", "beta", "do") else val) for key, val in x.items()}
        y["cu"] = np.array([0, b - a])
        y["h0"] = x["h0"][n:n + 1]
        y["dht"] = x["dht"][n:n + 1]
        one = _grads(y)
        for i in range(5):
            ok &= _close(full[i][:, a:b], one[i], 1e-12)
        ok &= _close(full[5][n:n + 1], one[5], 1e-12)
    return bool(ok)


def pin_normalised_gradients_are_tangent():
    """With q/k normalisation o depends on q_t only through q_t / |q_t| (up
    to the 1e-6 in the root), so <dq_t, q_t> ~ 0; the same for k."""
    x = _problem(10, lens=(6,), H=2, K=4, V=3)
    dq, dk = _grads(x, True)[:2]
    ok = True
    for d, a in ((dq, x["q"]), (dk, x["k"])):
        dot = np.abs(np.sum(d * a, -1))
        ok &= bool(np.all(dot <= 1e-5 * np.linalg.norm(d, axis=-1) * np.linalg.norm(a, axis=-1) + 1e-12))
        ok &= bool(np.max(np.abs(d)) > 1e-3)
    return bool(ok)


PINS = [pin_forward_is_the_recurrence, pin_finite_differences, pin_single_token_closed_form,
        pin_frozen_state_closed_form, pin_state_gradient_chains, pin_sequences_independent,
        pin_normalised_gradients_are_tangent]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_backward_oracle_pins(pin):
    assert pin()


def test_empty_and_zero_state():
    """No tokens: dh0 = dht; a zero h0 still gets its gradient."""
    x = _problem(11, lens=(0, 2))
    dq, dk, dv, dg, db, dh0 = _grads(x)
    assert _close(dh0[0], x["dht"][0], 0)
    y = dict(x, h0=None)
    assert np.max(np.abs(_grads(y)[5][1])) > 0


# ---------------------------------------------------------------------------
# Planted mistakes
# ---------------------------------------------------------------------------

def _bad_decay_after(S, qt, kt, vt, gt, bt, scale):
    pred = torch.einsum("hk,hkv->hv", kt, S)
    S = S + bt[:, None, None] * torch.einsum("hk,hv->hkv", kt, vt - pred)
    S = S * torch.exp(gt)[:, :, None]
    return S, torch.einsum("hk,hkv->hv", scale * qt, S)


def _bad_no_beta(S, qt, kt, vt, gt, bt, scale):
    S = S * torch.exp(gt)[:, :, None]
    S = S + torch.einsum("hk,hv->hkv", kt, vt - torch.einsum("hk,hkv->hv", kt, S))
    return S, torch.einsum("hk,hkv->hv", scale * qt, S)


def _bad_pred_sign(S, qt, kt, vt, gt, bt, scale):
    S = S * torch.exp(gt)[:, :, None]
    S = S + bt[:, None, None] * torch.einsum("hk,hv->hkv", kt, vt + torch.einsum("hk,hkv->hv", kt, S))
    return S, torch.einsum("hk,hkv->hv", scale * qt, S)


def _bad_pred_detached(S, qt, kt, vt, gt, bt, scale):
    S = S * torch.exp(gt)[:, :, None]
    pred = torch.einsum("hk,hkv->hv", kt, S).detach()
    S = S + bt[:, None, None] * torch.einsum("hk,hv->hkv", kt, vt - pred)
    return S, torch.einsum("hk,hkv->hv", scale * qt, S)


def _bad_readout_before(S, qt, kt, vt, gt, bt, scale):
    S = S * torch.exp(gt)[:, :, None]
    o = torch.einsum("hk,hkv->hv", scale * qt, S)
    S = S + bt[:, None, None] * torch.einsum("hk,hv->hkv", kt, vt - torch.einsum("hk,hkv->hv", kt, S))
    return S, o


def _bad_normalise_detached(x):
    return x / torch.sqrt((x * x).sum(-1, keepdim=True) + 1e-6).detach()


def _bad_normalise_eps_outside(x):
    return x / (torch.sqrt((x * x).sum(-1, keepdim=True)) + 1e-6)


def _bad_objective_no_dht(o, ht, do, dht):
    return (o * do).sum()


def _bad_objective_state_transposed(o, ht, do, dht):
    L = (o * do).sum()
    return L if dht is None else L + (ht.transpose(-1, -2) * dht.transpose(-1, -2).flip(-1)).sum()


MISTAKES = {
    "decay_after_delta": ("token_step", _bad_decay_after),
    "no_beta": ("token_step", _bad_no_beta),
    "prediction_sign": ("token_step", _bad_pred_sign),
    "prediction_detached": ("token_step", _bad_pred_detached),
    "readout_before_update": ("token_step", _bad_readout_before),
    "normaliser_detached": ("normalise", _bad_normalise_detached),
    "normaliser_eps_outside_root": ("normalise", _bad_normalise_eps_outside),
    "objective_drops_dht": ("objective", _bad_objective_no_dht),
    "objective_misindexes_dht": ("objective", _bad_objective_state_transposed),
}


def _passes(pin):
    try:
        return pin()
    except Exception:
        return False


@pytest.mark.parametrize("name", list(MISTAKES))
def test_pins_catch_planted_mistakes(name, monkeypatch):
    attr, bad = MISTAKES[name]
    monkeypatch.setattr(bw, attr, bad)
    failed = [p.__name__ for p in PINS if not _passes(p)]
    assert failed, f"no pin catches {name}"
