"""Adversarial inputs for the chunked forward on the GPU.

  * cancellation stress (operator page "PyPTO-Gym chunk_kda operator",
    section "测试与验证体系": a 64-draw search for cancellation in
    v_new = u - w S; see tests/adversarial.py for the construction);
  * a 131072-token sequence at H = 32 (the page's long-sequence stress case,
    T = 131072, outside its default list), compared on sampled units;
  * gate decay beyond the range in which the factored products are exact
    (section "数值稳定性": factors capped at e^80): the (sequence, head) units
    concerned are recomputed token by token, so the result stays exact;
    just inside the range (unscaled log-sigmoid gates) the chunked path
    alone is exact.
"""

import numpy as np
import pytest
import torch

from adversarial import cancellation_stress
from chunked_gated_delta_kda_gb300.inputs import Workload, custom, make_inputs
from kda_cases import assert_within, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_cancellation_stress(seed):
    x, info = cancellation_stress(seed=seed)
    assert info["ratio"] < 0.01                   # the search found strong cancellation
    o, ht = run_gpu(x)
    stats = compare(o, ht, *run_oracle(x))
    print(info, stats)
    assert_within(stats)


def test_long_sequence_t131072_h32():
    w = Workload("t131072_h32", B=1, T=131072, H=32, seed=8)
    x = make_inputs(w)
    o, ht = run_gpu(x)
    units = [(0, 0), (0, 31)]
    stats = compare(o, ht, *run_oracle(x, units=units), units=units)
    print(stats)
    assert_within(stats)
    assert torch.isfinite(o.float()).all() and torch.isfinite(ht).all()


def _status_run(x):
    from chunked_gated_delta_kda_gb300 import binding
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    B, T, H, _ = d["q"].shape
    N = x["N"]
    o = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
    ht = torch.empty((N, H, 128, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.workspace_bytes(B, T, H, N), dtype=torch.uint8, device="cuda")
    binding.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["h0"], d["cu_seqlens"], o, ht, N, 0, ws)
    return o, ht, binding.get_status(ws)


@pytest.mark.parametrize("gate_div", [0.75, 0.5, 0.1])
def test_decay_beyond_factoring_range_is_exact(gate_div):
    """Gates strong enough that some chunk's decay from its middle row passes
    the factor cap (80 nats): those (sequence, head) units are recomputed
    token by token, so the result still matches the oracle."""
    x = make_inputs(custom("far", B=1, T=512, H=2, with_h0=True, seed=5, gate_div=gate_div))
    o, ht, st = _status_run(x)
    assert st == 0
    assert_within(compare(o, ht, *run_oracle(x)))


def test_strong_decay_in_one_sequence_of_a_varlen_batch():
    """Varlen: only the middle sequence carries extreme gates; it is
    recomputed exactly, the others keep the chunked result."""
    lens = [300, 400, 200]
    x = make_inputs(custom("farv", B=1, T=900, H=2, seqlens=lens, with_h0=True, seed=6))
    x["g"][:, 300:700] = x["g"][:, 300:700] * 40.0
    o, ht, st = _status_run(x)
    assert st == 0
    assert_within(compare(o, ht, *run_oracle(x)))


def test_unscaled_gates_exact_and_unflagged():
    x = make_inputs(custom("edge", B=1, T=512, H=2, with_h0=True, seed=5, gate_div=1.0))
    o, ht, st = _status_run(x)
    assert st == 0
    assert_within(compare(o, ht, *run_oracle(x)))
