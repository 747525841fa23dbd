"""GPU checks of the single-device KCP forward (kda_kcp_fwd through the C ABI).

Ground truth is the fp64 per-token recurrence on the whole packed input; per
the KCP debugging guide (page "flash-linear-attention KCP precision-debugging
guide", section on why per-chunk comparison misleads under varlen KCP) the
comparison is per token, with the operator page's tolerances.  Where the rank
cuts fall on the chunk grid of every sequence, the first rank's outputs must
equal the unsplit forward's bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_kda_gb300.inputs import WORKLOADS, custom, make_inputs
from kda_cases import assert_within, compare, to_np

pytestmark = pytest.mark.gpu


def _kcp(x, W, l2norm=False):
    from chunked_gated_delta_kda_gb300 import binding
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    cu = x["cu_seqlens"].tolist()
    o, ht = binding.kcp_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, W, initial_state=d["h0"],
                            output_final_state=True, use_qk_l2norm_in_kernel=l2norm)
    torch.cuda.synchronize()
    return o, ht


def _ref(x, units=None, l2norm=False):
    return oracle.kda_recurrent(*[to_np(x[n]) for n in ("q", "k", "v", "g", "beta")], h0=to_np(x["h0"]),
                                cu_seqlens=x["cu_seqlens"].tolist(), units=units, l2norm=l2norm)


@pytest.mark.parametrize("lens,H,W", [([400, 624], 4, 2), ([1000], 2, 3), ([300, 0, 129, 700, 5], 3, 4),
                                      ([3, 4], 2, 16)])
def test_kcp_matches_recurrence(lens, H, W):
    x = make_inputs(custom("kcp", B=1, T=sum(lens), H=H, seqlens=lens, with_h0=True, seed=sum(lens) + W))
    o, ht = _kcp(x, W)
    o_ref, ht_ref = _ref(x)
    stats = compare(o, ht, o_ref, ht_ref)
    print(lens, W, stats)
    assert_within(stats)


def test_kcp_varlen_workload_sampled():
    w = WORKLOADS["varlen6_t9192_h32"]
    x = make_inputs(w)
    o, ht = _kcp(x, 4)
    units = [(n, h) for n in range(w.N) for h in (0, 31)]
    o_ref, ht_ref = _ref(x, units=units)
    assert_within(compare(o, ht, o_ref, ht_ref, units=units, cu=w.cu_seqlens))


def test_kcp_l2norm():
    x = make_inputs(custom("kl2", B=1, T=700, H=2, seqlens=[250, 450], with_h0=True, seed=9))
    gen = torch.Generator().manual_seed(5)
    for n in ("q", "k"):
        x[n] = (x[n].float() * (0.5 + 2 * torch.rand(x[n].shape[:3] + (1,), generator=gen))).bfloat16()
    o, ht = _kcp(x, 3, l2norm=True)
    assert_within(compare(o, ht, *_ref(x, l2norm=True)))


def test_one_rank_equals_forward_bitwise():
    from chunked_gated_delta_kda_gb300 import binding
    x = make_inputs(custom("k1", B=1, T=777, H=2, seqlens=[300, 477], with_h0=True, seed=4))
    o, ht = _kcp(x, 1)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o2, ht2 = binding.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"],
                          output_final_state=True, cu_seqlens=d["cu_seqlens"])
    assert torch.equal(o, o2) and torch.equal(ht, ht2)


def test_first_rank_bitwise_on_the_chunk_grid():
    """One 1024-token sequence on 2 ranks: the cut (512) is on the chunk grid,
    rank 0 has no incoming state, so its outputs equal the unsplit run's."""
    from chunked_gated_delta_kda_gb300 import binding
    x = make_inputs(custom("kg", B=1, T=1024, H=2, seqlens=[1024], with_h0=True, seed=6))
    o, _ = _kcp(x, 2)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o2, _ = binding.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"],
                        cu_seqlens=d["cu_seqlens"])
    assert torch.equal(o[:, :512], o2[:, :512])


def test_kcp_bad_host_offsets():
    from chunked_gated_delta_kda_gb300 import binding
    x = make_inputs(custom("kb", B=1, T=256, H=1, seqlens=[100, 156], seed=7))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    with pytest.raises(binding.KdaError) as e:
        binding.kcp_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], [0, 200, 100], 2)
    assert e.value.code == 4
