"""GPU parity of the token-by-token entry point (kda_fused_recurrent, through
the C ABI) against the fp64 decode oracle (``oracle.decode``).

Same tolerances as the chunked forward (operator page "PyPTO-Gym chunk_kda
operator", section "支持的 dtype 与形状约束"): |o - o_ref| <= 1e-2 + 1e-2 |o_ref|
on the bf16 output and |S - S_ref| <= 1e-3 + 1e-3 |S_ref| on every state slot
(written or not).  Inputs: chunked_gated_delta_kda_gb300.inputs.make_decode_inputs.
"""

import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_kda_gb300.inputs import custom, make_decode_inputs, make_inputs
from kda_cases import O_ATOL, O_RTOL, S_ATOL, S_RTOL, to_np

pytestmark = pytest.mark.gpu


def run_gpu(x, l2norm=False):
    from chunked_gated_delta_kda_gb300 import binding
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    pool = d["pool"].clone()
    o = binding.fused_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, d["indices"],
                                num_accepted_tokens=d["num_accepted"], cu_seqlens=d["cu_seqlens"],
                                use_qk_l2norm_in_kernel=l2norm)
    torch.cuda.synchronize()
    return o, pool


def run_ref(x, l2norm=False):
    acc = None if x["num_accepted"] is None else x["num_accepted"].numpy()
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].numpy()
    return oracle.fused_recurrent(to_np(x["q"]), to_np(x["k"]), to_np(x["v"]), to_np(x["g"]), to_np(x["beta"]),
                                  to_np(x["pool"]), x["indices"].numpy(), num_accepted=acc, cu_seqlens=cu,
                                  l2norm=l2norm)


def check(o, pool, o_ref, pool_ref):
    o = to_np(o).astype(np.float64)
    p = to_np(pool).astype(np.float64)
    assert np.isfinite(o).all() and np.isfinite(p).all()
    ro = (np.abs(o - o_ref) / (O_ATOL + O_RTOL * np.abs(o_ref))).max() if o.size else 0.0
    rs = (np.abs(p - pool_ref) / (S_ATOL + S_RTOL * np.abs(pool_ref))).max()
    assert ro <= 1.0 and rs <= 1.0, (ro, rs)
    return ro, rs


@pytest.mark.parametrize("N,H,T,pad", [(64, 8, 1, (5, 17)), (3, 4, 37, ()), (1, 32, 1, ())])
def test_plain_decode(N, H, T, pad):
    x = make_decode_inputs(N, H, T, pool_slots=2 * N + 3, pad=pad, seed=N + T)
    o, pool = run_gpu(x)
    print(check(o, pool, *run_ref(x)))
    for n in pad:
        assert torch.count_nonzero(o[n]) == 0


def test_varlen_decode_with_l2norm():
    x = make_decode_inputs(6, 4, [1, 5, 0, 2, 130, 1], pool_slots=9, seed=5)
    gen = torch.Generator().manual_seed(3)
    for n in ("q", "k"):   # unnormalised rows so that the flag matters
        x[n] = (x[n].float() * (0.5 + 2 * torch.rand(x[n].shape[:3] + (1,), generator=gen))).bfloat16()
    o, pool = run_gpu(x, l2norm=True)
    check(o, pool, *run_ref(x, l2norm=True))
    o2, _ = run_gpu(x, l2norm=False)
    assert (o.float() - o2.float()).abs().max().item() > 1e-4


@pytest.mark.parametrize("stride", [1, 4])
def test_spec_decode(stride):
    lens = [1 + (3 * n) % stride for n in range(16)]
    x = make_decode_inputs(16, 8, lens, pool_slots=16 * stride + 5, stride=stride, spec=True, seed=60 + stride)
    x["indices"][3, -1] = -1                 # a skipped checkpoint slot
    o, pool = run_gpu(x)
    check(o, pool, *run_ref(x))


def test_decode_continues_chunked_prefill():
    """Prefill 384 tokens with the chunked forward, put its final state in a
    pool slot, decode 5 more tokens one call at a time; outputs and state
    match the oracle's recurrence over all 389 tokens."""
    from chunked_gated_delta_kda_gb300 import binding
    w = custom("pd", B=1, T=389, H=4, seqlens=[389], with_h0=True, seed=71)
    x = make_inputs(w)
    o_ref, ht_ref = oracle.kda_recurrent(*[to_np(x[n]) for n in ("q", "k", "v", "g", "beta")], h0=to_np(x["h0"]),
                                         cu_seqlens=[0, 389])
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    pre = {n: d[n][:, :384].contiguous() for n in ("q", "k", "v", "g", "beta")}
    o_pre, ht = binding.fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], initial_state=d["h0"],
                            output_final_state=True)
    pool = torch.zeros((3, 4, 128, 128), dtype=torch.float32, device="cuda")
    pool[2] = ht[0]
    idx = torch.tensor([[2]], dtype=torch.int32, device="cuda")
    outs = []
    for t in range(384, 389):
        sl = {n: d[n][:, t:t + 1].contiguous() for n in ("q", "k", "v", "g", "beta")}
        outs.append(binding.fused_recurrent(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], pool, idx))
    o = torch.cat([o_pre] + outs, dim=1)
    torch.cuda.synchronize()
    o_np, s_np = to_np(o).astype(np.float64), to_np(pool[2]).astype(np.float64)
    assert (np.abs(o_np - o_ref) / (O_ATOL + O_RTOL * np.abs(o_ref))).max() <= 1.0
    assert (np.abs(s_np - ht_ref[0]) / (S_ATOL + S_RTOL * np.abs(ht_ref[0]))).max() <= 1.0
    assert torch.count_nonzero(pool[:2]) == 0


def test_decode_deterministic():
    x = make_decode_inputs(8, 4, 3, pool_slots=8, seed=80)
    o1, p1 = run_gpu(x)
    o2, p2 = run_gpu(x)
    assert torch.equal(o1, o2) and torch.equal(p1, p2)


def test_bad_slot_reported_and_isolated():
    """A slot >= pool size: status 7, that sequence's output is zero and the
    pool is untouched for it; the other sequences still match the oracle."""
    from chunked_gated_delta_kda_gb300 import binding
    x = make_decode_inputs(4, 2, 1, pool_slots=9, seed=90)
    good = dict(x)
    good["indices"] = x["indices"].clone()
    good["indices"][1] = -1                  # the oracle's view: sequence 1 does nothing
    o_ref, pool_ref = run_ref(good)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    d["indices"][1, 0] = 9
    pool = d["pool"].clone()
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    o = torch.empty((4, 1, 2, 128), dtype=torch.bfloat16, device="cuda")
    binding.kda_fused_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], None, pool, d["indices"], None, None,
                                o, 4, 0, ws)
    assert binding.get_status(ws) == 7
    check(o, pool, o_ref, pool_ref)
    assert torch.count_nonzero(o[1]) == 0
    # accepted count out of range
    y = make_decode_inputs(2, 2, [1, 2], pool_slots=6, stride=2, spec=True, seed=91)
    dy = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in y.items()}
    dy["num_accepted"][0] = 3
    o = torch.empty((1, 3, 2, 128), dtype=torch.bfloat16, device="cuda")
    binding.kda_fused_recurrent(dy["q"], dy["k"], dy["v"], dy["g"], dy["beta"], None, dy["pool"].clone(),
                                dy["indices"], dy["num_accepted"], dy["cu_seqlens"], o, 2, 0, ws)
    assert binding.get_status(ws) == 7
    # a valid call afterwards reports ok
    binding.kda_fused_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["pool"].clone(),
                                x["indices"].cuda(), None, None,
                                torch.empty((4, 1, 2, 128), dtype=torch.bfloat16, device="cuda"), 4, 0, ws)
    assert binding.get_status(ws) == 0


def test_bad_cu_reported():
    from chunked_gated_delta_kda_gb300 import binding
    x = make_decode_inputs(3, 2, [1, 2, 1], pool_slots=5, seed=93)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    bad = torch.tensor([0, 3, 2, 4], dtype=torch.int32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    o = torch.empty((1, 4, 2, 128), dtype=torch.bfloat16, device="cuda")
    binding.kda_fused_recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["pool"].clone(), d["indices"],
                                None, bad, o, 3, 0, ws)
    assert binding.get_status(ws) == 4
