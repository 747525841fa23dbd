"""Pins of the KCP oracle (``oracle.kcp``), CPU only.

The KCP forward must reproduce the plain per-token recurrence on the whole
packed input (page "flash-linear-attention KCP precision-debugging guide":
per-token tensors are the ones that stay comparable across a KCP split), for
cuts inside sequences, sequences spanning several ranks, empty ranks and
empty sequences.  The rank split is pinned to the guide's worked example, and
planted mistakes in the merge are caught.
"""

import json
import os

import numpy as np
import pytest

import oracle
from oracle import kcp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(seed, lens, H=2, K=4, V=4, with_h0=True):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    q = rng.standard_normal((1, T, H, K))
    k = rng.standard_normal((1, T, H, K))
    q = f32(q / np.linalg.norm(q, axis=-1, keepdims=True))
    k = f32(k / np.linalg.norm(k, axis=-1, keepdims=True))
    v = f32(rng.standard_normal((1, T, H, V)))
    g = f32(np.log(1 / (1 + np.exp(-rng.standard_normal((1, T, H, K))))) / 4)
    beta = f32(1 / (1 + np.exp(-rng.standard_normal((1, T, H)))))
    h0 = f32(0.3 * rng.standard_normal((len(lens), H, V, K))) if with_h0 else None
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(int).tolist()
    return q, k, v, g, beta, cu, h0


CASES = [
    ([37, 50], 2, True),           # cut inside the second sequence
    ([90], 3, True),               # one sequence across three ranks
    ([20, 0, 33, 11], 4, True),    # an empty sequence
    ([5, 2], 9, True),             # more ranks than tokens: empty ranks
    ([40, 41, 7], 3, False),       # zero initial states
]


def _kcp_matches_recurrence(l2norm=False):
    ok = True
    for i, (lens, W, with_h0) in enumerate(CASES):
        q, k, v, g, beta, cu, h0 = _problem(10 + i, lens, with_h0=with_h0)
        o, ht = kcp.kcp_forward(q, k, v, g, beta, cu, W, h0=h0, l2norm=l2norm)
        o_ref, ht_ref = oracle.kda_recurrent(q, k, v, g, beta, h0=h0, cu_seqlens=cu, l2norm=l2norm)
        ok &= np.allclose(o, o_ref, atol=1e-6, rtol=0) and np.allclose(ht, ht_ref, atol=1e-6, rtol=0)
    return bool(ok)


def test_kcp_equals_recurrence():
    assert _kcp_matches_recurrence()


def test_kcp_equals_recurrence_l2norm():
    assert _kcp_matches_recurrence(l2norm=True)


def test_one_rank_is_the_recurrence_exactly():
    q, k, v, g, beta, cu, h0 = _problem(3, [30, 12, 25])
    o, ht = kcp.kcp_forward(q, k, v, g, beta, cu, 1, h0=h0)
    o_ref, ht_ref = oracle.kda_recurrent(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    assert np.array_equal(o, o_ref) and np.array_equal(ht, ht_ref)


def test_rank_split_worked_example():
    """Guide's worked example: lengths [400, 624], world size 2 -> rank 1
    starts at global token 512 (inside sequence 1)."""
    with open(os.path.join(GOLDEN, "kcp_chunk_boundaries.json")) as f:
        gold = json.load(f)
    cu = np.cumsum([0] + gold["lengths"]).tolist()
    bounds = kcp.rank_bounds(cu[-1], 2)
    assert bounds[1] == gold["rank1_global_start"]
    pc = kcp.pieces(cu, cu[-1], 2)
    assert pc[0] == [(0, 0, 400), (1, 400, 512)] and pc[1] == [(1, 512, 1024)]


def _merge_no_ext(start, mt, ext):
    return np.zeros_like(ext) if start is None else np.einsum("hvj,hjk->hvk", start, mt)


def _merge_transposed(start, mt, ext):
    return ext.copy() if start is None else np.einsum("hvj,hkj->hvk", start, mt) + ext


def _initial_ignores_merge(n, a, cu, h0, incoming):
    return None if h0 is None else h0[n]


@pytest.mark.parametrize("attr,bad", [("merge", _merge_no_ext), ("merge", _merge_transposed),
                                      ("piece_initial", _initial_ignores_merge)],
                         ids=["merge_drops_S_ext", "merge_transposes_M", "continuation_uses_h0"])
def test_pins_catch_planted_mistakes(attr, bad, monkeypatch):
    monkeypatch.setattr(kcp, attr, bad)
    assert not _kcp_matches_recurrence()
