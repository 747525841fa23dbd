"""Pins of the decode oracle (``oracle.decode``), CPU only.

The decode oracle is pinned to the C per-token recurrence (``kda_recurrent``,
itself pinned in ``test_oracle.py``; the two share no code), to closed forms,
and to the slot semantics stated in ``oracle/decode.py`` (page
"PyPTO-Gym chunk_kda operator", section "与其他 KDA 算子的关系": in-place state
at ``ssm_state_indices``, speculative decoding via ``num_accepted_tokens``).
``test_pins_catch_planted_mistakes`` plants a mistake in each helper of the
oracle in turn and checks that at least one pin fails.
"""

import numpy as np
import pytest

import oracle
from oracle import decode as fr

TOL = 1e-10


def _f32(rng, shape, scale=1.0):
    return (scale * rng.standard_normal(shape)).astype(np.float32).astype(np.float64)


def _unit(rng, shape):
    x = rng.standard_normal(shape)
    return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32).astype(np.float64)


def _problem(seed, N=4, lens=1, H=2, K=4, V=3, P=11, stride=1, spec=False, pad=()):
    rng = np.random.default_rng(seed)
    if isinstance(lens, int):
        B, T, cu = N, lens, None
    else:
        B, T = 1, sum(lens)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q = _unit(rng, (B, T, H, K))
    k = _unit(rng, (B, T, H, K))
    v = _f32(rng, (B, T, H, V))
    g = np.log(1 / (1 + np.exp(-rng.standard_normal((B, T, H, K))))).astype(np.float32).astype(np.float64) / 4
    beta = (1 / (1 + np.exp(-rng.standard_normal((B, T, H))))).astype(np.float32).astype(np.float64)
    pool = _f32(rng, (P, H, V, K), 0.5)
    idx = rng.permutation(P)[: N * stride].reshape(N, stride)
    for n in pad:
        idx[n] = -1
    acc = rng.integers(1, stride + 1, N) if spec else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, pool=pool, idx=idx, acc=acc, cu=cu, B=B, T=T, N=N)


def _bounds(x):
    if x["cu"] is None:
        return [(n * x["T"], x["T"]) for n in range(x["N"])]
    cu = x["cu"]
    return [(int(cu[n]), int(cu[n + 1] - cu[n])) for n in range(x["N"])]


def _c_oracle_seq(x, n, h0_slot, upto, l2norm=False):
    """C recurrence over the first `upto` tokens of sequence n, from pool slot h0_slot."""
    bos, _ = _bounds(x)[n]
    sl = slice(bos, bos + upto)
    flat = lambda a: a.reshape((x["B"] * x["T"],) + a.shape[2:])[sl][None]
    o, ht = oracle.kda_recurrent(flat(x["q"]), flat(x["k"]), flat(x["v"]), flat(x["g"]), flat(x["beta"]),
                                 h0=x["pool"][h0_slot][None], l2norm=l2norm)
    return o[0], ht[0]


def _run(x, l2norm=False):
    return fr.fused_recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["pool"], x["idx"],
                              num_accepted=x["acc"], cu_seqlens=x["cu"], l2norm=l2norm)


# ---------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------

def pin_plain_decode_matches_recurrence():
    """Plain decode: sequence n reads slot idx[n][0], writes its final state
    back there; padding rows leave everything alone and output zeros."""
    ok = True
    for l2 in (False, True):
        x = _problem(1, N=5, lens=[1, 3, 0, 2, 1], pad=(3,))
        o, pool = _run(x, l2norm=l2)
        o = o.reshape(-1, *o.shape[2:])
        touched = set()
        for n, (bos, L) in enumerate(_bounds(x)):
            slot = int(x["idx"][n][0])
            if L == 0 or slot < 0:
                ok &= np.all(o[bos:bos + L] == 0)
                continue
            o_ref, ht_ref = _c_oracle_seq(x, n, slot, L, l2norm=l2)
            ok &= np.allclose(o[bos:bos + L], o_ref, atol=TOL, rtol=0)
            ok &= np.allclose(pool[slot], ht_ref, atol=TOL, rtol=0)
            touched.add(slot)
        for s in range(pool.shape[0]):
            if s not in touched:
                ok &= np.array_equal(pool[s], x["pool"][s])
    return bool(ok)


def pin_spec_checkpoints():
    """Speculative mode: start from slot idx[n][acc-1]; after token t the
    state of the first t+1 tokens is stored at idx[n][t]."""
    ok = True
    for seed in (2, 3):
        x = _problem(seed, N=4, lens=[3, 1, 4, 2], stride=4, spec=True, P=19)
        o, pool = _run(x)
        o = o.reshape(-1, *o.shape[2:])
        for n, (bos, L) in enumerate(_bounds(x)):
            src = int(x["idx"][n][x["acc"][n] - 1])
            for t in range(L):
                o_ref, ht_ref = _c_oracle_seq(x, n, src, t + 1)
                ok &= np.allclose(pool[x["idx"][n][t]], ht_ref, atol=TOL, rtol=0)
                ok &= np.allclose(o[bos + t], o_ref[t], atol=TOL, rtol=0)
            for t in range(L, 4):      # slots past the sequence keep their state
                ok &= np.array_equal(pool[x["idx"][n][t]], x["pool"][x["idx"][n][t]])
    return bool(ok)


def pin_chained_single_tokens():
    """T tokens in one call equal T calls of one token chained through the pool."""
    x = _problem(4, N=2, lens=5)
    o_all, pool_all = _run(x)
    pool = x["pool"].copy()
    outs = []
    for t in range(5):
        y = dict(x)
        for key in ("q", "k", "v", "g", "beta"):
            y[key] = x[key][:, t:t + 1]
        y["T"] = 1
        y["pool"] = pool
        o_t, pool = _run(y)
        outs.append(o_t)
    return bool(np.allclose(np.concatenate(outs, axis=1), o_all, atol=TOL, rtol=0)
                and np.allclose(pool, pool_all, atol=TOL, rtol=0))


def pin_frozen_readout():
    """beta = 0 and g = 0: the state is unchanged and o = scale * S^T q."""
    x = _problem(5, N=3, lens=2)
    x["beta"] = np.zeros_like(x["beta"])
    x["g"] = np.zeros_like(x["g"])
    o, pool = _run(x)
    K = x["q"].shape[-1]
    ok = np.array_equal(pool, x["pool"])
    for n in range(3):
        S_vk = x["pool"][x["idx"][n][0]]                    # [H, V, K]
        expect = np.einsum("thk,hvk->thv", x["q"][n] * K ** -0.5, S_vk)
        ok &= np.allclose(o[n], expect, atol=TOL, rtol=0)
    return bool(ok)


PINS = [pin_plain_decode_matches_recurrence, pin_spec_checkpoints, pin_chained_single_tokens,
        pin_frozen_readout]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_decode_oracle_pins(pin):
    assert pin()


def test_out_of_range_rejected():
    x = _problem(6, N=2, lens=1)
    x["idx"][1][0] = x["pool"].shape[0]
    with pytest.raises(ValueError):
        _run(x)
    y = _problem(7, N=2, lens=[1, 2], stride=2, spec=True)
    y["acc"][0] = 3
    with pytest.raises(ValueError):
        _run(y)


# ---------------------------------------------------------------------------
# Planted mistakes
# ---------------------------------------------------------------------------

def _bad_step_decay_after(S, q, k, v, g, beta):
    pred = k @ S
    S += beta * np.outer(k, v - pred)
    S *= np.exp(g)[:, None]
    return q @ S


def _bad_step_readout_first(S, q, k, v, g, beta):
    o = q @ (S * np.exp(g)[:, None])
    S *= np.exp(g)[:, None]
    S += beta * np.outer(k, v - k @ S)
    return o


def _bad_step_no_beta(S, q, k, v, g, beta):
    S *= np.exp(g)[:, None]
    S += np.outer(k, v - k @ S)
    return q @ S


def _bad_read_off_by_one(row, acc):
    return int(row[0]) if acc is None else int(row[min(acc, len(row) - 1)])


def _bad_read_ignores_accepted(row, acc):
    return int(row[0])


def _bad_write_final_only(row, acc, L):
    return [(L - 1, int(row[0] if acc is None else row[L - 1]))]


def _bad_write_shifted(row, acc, L):
    if acc is None:
        return [(L - 1, int(row[0]))]
    return [(t, int(row[min(t + 1, len(row) - 1)])) for t in range(L)]


MISTAKES = {
    "decay_after_delta": ("token_step", _bad_step_decay_after),
    "readout_before_update": ("token_step", _bad_step_readout_first),
    "no_beta": ("token_step", _bad_step_no_beta),
    "read_slot_off_by_one": ("read_slot", _bad_read_off_by_one),
    "read_slot_ignores_accepted": ("read_slot", _bad_read_ignores_accepted),
    "spec_writes_final_only": ("write_slots", _bad_write_final_only),
    "spec_writes_shifted": ("write_slots", _bad_write_shifted),
}


def _passes(pin):
    try:
        return pin()
    except Exception:
        return False


@pytest.mark.parametrize("name", list(MISTAKES))
def test_pins_catch_planted_mistakes(name, monkeypatch):
    assert all(_passes(p) for p in PINS)
    attr, bad = MISTAKES[name]
    monkeypatch.setattr(fr, attr, bad)
    failed = [p.__name__ for p in PINS if not _passes(p)]
    assert failed, f"no pin catches {name}"
