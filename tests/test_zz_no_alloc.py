"""GPU test of kda_fwd_noalloc, the entry point for callers that cannot
allocate device memory (code inside an allocator's own callback, plug-ins
whose host owns every allocation, fixed memory budgets).  It must give bit for bit the result of kda_fwd
with a caller-provided workspace (it runs the same kernels), call after call, and refuse problems that do not
fit its static scratch.  This file is collected last on purpose."""

import pytest
import torch

from chunked_gated_delta_kda_gb300.inputs import custom, make_inputs

pytestmark = pytest.mark.gpu


def _device_inputs(w):
    x = make_inputs(w)
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _run_both(x):
    from chunked_gated_delta_kda_gb300 import binding
    q, k, v, g, beta, h0, cu = (x[n] for n in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    B, T, H, K = q.shape
    N = x["N"]
    o_ref, ht_ref = binding.fwd(q, k, v, g, beta, initial_state=h0, output_final_state=True, cu_seqlens=cu)
    o = torch.empty_like(o_ref)
    ht = torch.empty_like(ht_ref)
    binding.kda_fwd_noalloc(q, k, v, g, beta, None, h0, cu, o, ht, N, 0)
    torch.cuda.synchronize()
    return o, ht, o_ref, ht_ref


@pytest.mark.parametrize("w", [
    custom("noalloc_fixed", B=2, T=1024, H=4, with_h0=True, seed=61),
    custom("noalloc_varlen", B=1, T=612, H=3, seqlens=[100, 300, 0, 212], with_h0=True, seed=62),
    # unscaled gates: every chunk through the wide prep kernel's queue, which
    # lives in the shared scratch too
    custom("noalloc_wide", B=1, T=1024, H=3, with_h0=True, seed=65, gate_div=1.0),
], ids=lambda w: w.name)
def test_noalloc_matches_kda_fwd_on_consecutive_calls(w):
    for call in range(2):
        x = _device_inputs(custom(w.name, B=w.B, T=w.T, H=w.H, seqlens=w.seqlens, with_h0=w.with_h0,
                                  seed=w.seed + 100 * call, gate_div=w.gate_div))
        o, ht, o_ref, ht_ref = _run_both(x)
        assert torch.isfinite(o.float()).all() and torch.isfinite(ht).all()
        # the same kernels on the same inputs: bit-identical, not just close
        assert torch.equal(o, o_ref)
        assert torch.equal(ht, ht_ref)


def test_noalloc_guarded_outputs():
    """Outputs inside canary guards: the no-alloc call writes nothing outside
    o and ht and gives kda_fwd's bits (two calls in a row: the second finds
    the first one's leftovers in the shared scratch)."""
    from kda_cases import run_gpu_guarded
    for call in range(2):
        w = custom("noalloc_guard", B=1, T=700, H=2, seqlens=[1, 128, 0, 571], with_h0=True, seed=64 + call)
        x = make_inputs(w)
        o, ht, ok = run_gpu_guarded(x, noalloc=True)
        assert ok
        o_ref, ht_ref, _ = run_gpu_guarded(x)
        assert torch.equal(o, o_ref) and torch.equal(ht, ht_ref)


def test_noalloc_rejects_problem_larger_than_scratch():
    from chunked_gated_delta_kda_gb300 import binding
    lib = binding.load_library()
    limit = 64 * 1024 * 1024
    B, T, H = 1, 8192, 32
    assert lib.kda_fwd_workspace_bytes(B, T, H, 128, 128, 1) > limit
    x = _device_inputs(custom("noalloc_big", B=B, T=T, H=H, seed=63))
    o = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.KdaError) as e:
        binding.kda_fwd_noalloc(x["q"], x["k"], x["v"], x["g"], x["beta"], None, None, None, o, None, 1, 0)
    assert e.value.code == 6
