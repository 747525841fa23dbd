"""Shared helpers for the GPU parity tests: run the CUDA path through the
binding (which calls the C ABI) and the fp64 oracle on the same seeded inputs,
and compare with the tolerances of the operator page (section "支持的 dtype 与
形状约束": o atol = rtol = 1e-2, final state 1e-3)."""

from __future__ import annotations

import numpy as np
import torch

import oracle

O_ATOL = O_RTOL = 1e-2
S_ATOL = S_RTOL = 1e-3
# Diagnostic bound on the relative L2 error of o: |o| is ~0.01 at these input
# distributions, so the absolute term of the elementwise bound is loose.
O_RELNORM = 1e-2


def to_np(t):
    return None if t is None else t.detach().float().cpu().numpy()


def run_gpu(x, output_final_state=True, l2norm=False, device="cuda", token_exact=False):
    from chunked_gated_delta_kda_gb300 import binding
    d = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, ht = binding.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d.get("scale"),
                        initial_state=d["h0"], output_final_state=output_final_state,
                        use_qk_l2norm_in_kernel=l2norm, cu_seqlens=d["cu_seqlens"], token_exact=token_exact)
    torch.cuda.synchronize()
    return o, ht


def run_oracle(x, units=None, l2norm=False):
    args = [to_np(x[n]) for n in ("q", "k", "v", "g", "beta")]
    h0 = to_np(x["h0"])
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].cpu().numpy()
    return oracle.kda_recurrent(*args, scale=x.get("scale"), h0=h0, cu_seqlens=cu, l2norm=l2norm,
                                units=units)


def compare(o_gpu, ht_gpu, o_ref, ht_ref, units=None, cu=None, T=None, H=None):
    """Elementwise tolerance check on o (bf16 output) and the final state,
    restricted to the selected units when given.  Returns a stats dict."""
    o = to_np(o_gpu).astype(np.float64)
    if units is not None:
        B = o.shape[0]
        mask = np.zeros(o.shape[:3], dtype=bool)
        for n, h in units:
            if cu is None:
                mask[n, :, h] = True
            else:
                mask[0, int(cu[n]):int(cu[n + 1]), h] = True
        o_sel, r_sel = o[mask], o_ref[mask]
    else:
        o_sel, r_sel = o.reshape(-1, o.shape[-1]), o_ref.reshape(-1, o_ref.shape[-1])
    assert np.isfinite(o_sel).all(), "non-finite output"
    err = np.abs(o_sel - r_sel)
    ratio_o = (err / (O_ATOL + O_RTOL * np.abs(r_sel))).max() if err.size else 0.0
    relnorm = float(np.linalg.norm(o_sel - r_sel) / max(np.linalg.norm(r_sel), 1e-30)) if err.size else 0.0
    stats = {"o_tol_ratio": float(ratio_o), "o_relnorm": relnorm, "o_maxabs": float(err.max()) if err.size else 0.0}
    if ht_ref is not None and ht_gpu is not None:
        s = to_np(ht_gpu).astype(np.float64)
        if units is not None:
            s_sel = np.stack([s[n, h] for n, h in units])
            r_s = np.stack([ht_ref[n, h] for n, h in units])
        else:
            s_sel, r_s = s, ht_ref
        assert np.isfinite(s_sel).all(), "non-finite state"
        es = np.abs(s_sel - r_s)
        stats["S_tol_ratio"] = float((es / (S_ATOL + S_RTOL * np.abs(r_s))).max())
        stats["S_maxabs"] = float(es.max())
    return stats


def assert_within(stats):
    assert stats["o_tol_ratio"] <= 1.0, stats
    assert stats["o_relnorm"] <= O_RELNORM, stats
    if "S_tol_ratio" in stats:
        assert stats["S_tol_ratio"] <= 1.0, stats


# ---------------------------------------------------------------------------
# Stand-ins for a memory checker (the GPU sanitizer is closed on this machine):
# outputs allocated inside guard regions holding canary bit patterns that no
# kernel writes, and a workspace poisoned with 0xFF bytes (NaN as fp16 and
# fp32) before the call.  A write past a tail shows up as a changed canary;
# a read of a workspace byte that was never written shows up as a NaN in the
# outputs (or as a difference from an unpoisoned run).
# ---------------------------------------------------------------------------

CANARY16 = 0x7FA1          # a bf16 NaN payload
CANARY32 = 0x7FC0DEAD      # an fp32 NaN payload
GUARD = 4096               # elements on each side (16-byte aligned views)


def guarded(shape, dtype, device="cuda"):
    """(buffer, view): a view of `shape` with GUARD canary elements on both
    sides inside one allocation."""
    n = 1
    for s in shape:
        n *= int(s)
    if dtype == torch.bfloat16:
        buf = torch.full((n + 2 * GUARD,), CANARY16, dtype=torch.int16, device=device)
        view = buf[GUARD:GUARD + n].view(torch.bfloat16).view(*shape)
    else:
        assert dtype == torch.float32
        buf = torch.full((n + 2 * GUARD,), CANARY32 - (1 << 32) if CANARY32 >= (1 << 31) else CANARY32,
                         dtype=torch.int32, device=device)
        view = buf[GUARD:GUARD + n].view(torch.float32).view(*shape)
    return buf, view


def canaries_intact(buf):
    want = CANARY16 if buf.dtype == torch.int16 else CANARY32
    lo, hi = buf[:GUARD].cpu().numpy(), buf[-GUARD:].cpu().numpy()
    mask = 0xFFFF if buf.dtype == torch.int16 else 0xFFFFFFFF
    return bool(((lo.astype(np.int64) & mask) == want).all() and ((hi.astype(np.int64) & mask) == want).all())


def run_gpu_guarded(x, l2norm=False, noalloc=False):
    """The forward through the C ABI with guarded outputs and (unless
    ``noalloc``) a poisoned workspace.  Returns (o, ht, canaries_ok)."""
    from chunked_gated_delta_kda_gb300 import binding
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    B, T, H, K = d["q"].shape
    V = d["v"].shape[-1]
    N = x["N"]
    ob, o = guarded((B, T, H, V), torch.bfloat16)
    hb, ht = guarded((N, H, V, K), torch.float32)
    flags = binding.KDA_FLAG_QK_L2NORM if l2norm else 0
    if noalloc:
        binding.kda_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("scale"), d["h0"],
                                d["cu_seqlens"], o, ht, N, flags)
    else:
        ws = torch.full((binding.workspace_bytes(B, T, H, N),), 0xFF, dtype=torch.uint8, device="cuda")
        binding.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("scale"), d["h0"], d["cu_seqlens"],
                        o, ht, N, flags, ws)
        assert binding.get_status(ws) == 0
    torch.cuda.synchronize()
    return o, ht, canaries_intact(ob) and canaries_intact(hb)
