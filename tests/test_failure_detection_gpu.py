"""Failure detection of the bounded device waits, on the GPU, without a fault.

Every wait of one CTA role on another (a tile landed, a product done, a
stage freed) polls a bounded number of times.  The test shortens that bound
through the library's test hook and makes one wait run out for real: the
sequential scan's stage load of chunk 1 is never issued for unit (sequence 0,
head 0), value tile 0, so the waits on it can only run out.  The kernels must
then report KDA_ERR_TIMEOUT through the workspace status word within a short
time, leave every other unit's results intact, and leave the CUDA context
healthy for the next call.  Nothing here traps, faults or spins without a
bound.
"""

import time

import pytest
import torch

from chunked_gated_delta_kda_gb300.inputs import custom, make_inputs
from kda_cases import assert_within, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

KDA_ERR_TIMEOUT = 5


def test_scan_wait_timeout_reported_and_contained():
    from chunked_gated_delta_kda_gb300 import binding
    w = custom("timeout", B=1, T=512, H=2, with_h0=True, seed=71)
    x = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o = torch.zeros((1, 512, 2, 128), dtype=torch.bfloat16, device="cuda")
    ht = torch.zeros((1, 2, 128, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.workspace_bytes(1, 512, 2, 1), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    try:
        binding.debug_set(binding.KDA_DEBUG_WAIT_LIMIT, 1 << 14)
        binding.debug_set(binding.KDA_DEBUG_DROP_SCAN_LOAD, 1)
        t0 = time.perf_counter()
        binding.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["h0"], None, o, ht, 1, 0, ws)
        status = binding.get_status(ws)
        elapsed = time.perf_counter() - t0
    finally:
        binding.debug_set(binding.KDA_DEBUG_WAIT_LIMIT, 0)
        binding.debug_set(binding.KDA_DEBUG_DROP_SCAN_LOAD, 0)
    assert status == KDA_ERR_TIMEOUT, status
    assert elapsed < 5.0, elapsed

    # the other head was computed by CTAs whose waits all completed
    o_ref, ht_ref = run_oracle(x, units=[(0, 1)])
    assert_within(compare(o, ht, o_ref, ht_ref, units=[(0, 1)]))

    # the context is healthy and the hook has reset itself: the same call is
    # now correct on every unit and reports no error
    o2, ht2 = run_gpu(x)
    o_ref, ht_ref = run_oracle(x)
    assert_within(compare(o2, ht2, o_ref, ht_ref))
    ws2 = torch.empty_like(ws)
    binding.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["h0"], None, o, ht, 1, 0, ws2)
    assert binding.get_status(ws2) == 0
