"""Seeded synthetic KDA forward inputs (the workload recipe, no method arithmetic).

This module is the one piece shared by the oracle-side tests and the CUDA
path's tests and benchmark: it only draws random tensors.  It imports nothing
else from this package, so importing it never loads the CUDA library.

Recipe (for every named workload): a torch CPU ``Generator`` seeded with the
workload's seed draws, in this order and in fp32,
  q ~ N(0,1) [B,T,H,K], L2-normalised over K per (token, head), cast to bf16;
  k ~ N(0,1) [B,T,H,K], L2-normalised the same way, cast to bf16;
  v ~ N(0,1) [B,T,H,V], cast to bf16;
  g = logsigmoid(N(0,1)) / 16 per dimension [B,T,H,K], fp32 (so g <= 0);
  beta = sigmoid(N(0,1)) [B,T,H], fp32;
  h0 = 0.1 * N(0,1) [N,H,V,K], fp32, for the workloads that carry one.
The backward's upstream gradients (``make_grad_inputs``) come from a second
generator seeded with seed + 7919: do ~ N(0,1) [B,T,H,V] cast to bf16, then
dht = 0.1 * N(0,1) [N,H,V,K] fp32 (the scale of h0).
This follows the operator page's "stable inputs" convention (log-sigmoid
gates, sigmoid beta) with the scalings that the five named workloads fix.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int = 128
    V: int = 128
    seqlens: Optional[Sequence[int]] = None   # varlen packing (B == 1)
    with_h0: bool = False
    seed: int = 0
    gate_div: float = 16.0
    extra: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return len(self.seqlens) if self.seqlens is not None else self.B

    @property
    def cu_seqlens(self) -> Optional[list]:
        if self.seqlens is None:
            return None
        cu = [0]
        for s in self.seqlens:
            cu.append(cu[-1] + int(s))
        return cu

    @property
    def token_heads(self) -> int:
        return self.B * self.T * self.H


# The five named workloads.
WORKLOADS = {
    "tiny": Workload("tiny", B=1, T=256, H=1, seed=0),
    "b2_t2048_h8": Workload("b2_t2048_h8", B=2, T=2048, H=8, with_h0=True, seed=1),
    "b4_t8192_h16": Workload("b4_t8192_h16", B=4, T=8192, H=16, seed=2),
    "varlen6_t9192_h32": Workload("varlen6_t9192_h32", B=1, T=9192, H=32,
                                  seqlens=(400, 624, 1000, 3000, 129, 4039),
                                  with_h0=True, seed=3),
    "t65536_h32": Workload("t65536_h32", B=1, T=65536, H=32, seed=4),
}


def make_inputs(w: Workload, device: str = "cpu", draw_on_device: bool = False, seed_offset: int = 0):
    """Draw the workload's tensors.  Returns a dict with q, k, v (bf16), g, beta,
    h0 (fp32 or None), cu_seqlens (int32 tensor or None), scale (None), N.

    By default the draws come from a CPU generator (the values the oracle
    tests use) and are then moved to ``device``.  ``draw_on_device=True``
    draws the same distributions with a generator on ``device`` instead (a
    different, equally seeded stream of numbers; used where only timing
    matters and the workload is too large to draw quickly on the host)."""
    gdev = device if draw_on_device else "cpu"
    gen = torch.Generator(device=gdev)
    gen.manual_seed(int(w.seed) + int(seed_offset))
    B, T, H, K, V = w.B, w.T, w.H, w.K, w.V

    def randn(shape):
        return torch.randn(shape, generator=gen, dtype=torch.float32, device=gdev)

    def unit_rows(shape):
        x = randn(shape)
        x = x / x.norm(dim=-1, keepdim=True)
        return x.to(torch.bfloat16)

    q = unit_rows((B, T, H, K))
    k = unit_rows((B, T, H, K))
    v = randn((B, T, H, V)).to(torch.bfloat16)
    g = F.logsigmoid(randn((B, T, H, K))) / w.gate_div
    beta = torch.sigmoid(randn((B, T, H)))
    h0 = None
    if w.with_h0:
        h0 = 0.1 * randn((w.N, H, V, K))
    cu = None
    if w.seqlens is not None:
        assert B == 1 and sum(w.seqlens) == T
        cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=gdev)
    out = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, cu_seqlens=cu, scale=None, N=w.N)
    if device != gdev:
        out = {kk: (vv.to(device) if isinstance(vv, torch.Tensor) else vv) for kk, vv in out.items()}
    return out


def make_grad_inputs(w: Workload, device: str = "cpu", draw_on_device: bool = False, seed_offset: int = 0,
                     with_dht: bool = True):
    """Upstream gradients for the backward of ``make_inputs(w)``: a dict with
    do (bf16 [B,T,H,V]) and dht (fp32 [N,H,V,K] or None)."""
    gdev = device if draw_on_device else "cpu"
    gen = torch.Generator(device=gdev)
    gen.manual_seed(int(w.seed) + 7919 + int(seed_offset))
    do = torch.randn((w.B, w.T, w.H, w.V), generator=gen, dtype=torch.float32, device=gdev).to(torch.bfloat16)
    dht = None
    if with_dht:
        dht = 0.1 * torch.randn((w.N, w.H, w.V, w.K), generator=gen, dtype=torch.float32, device=gdev)
    out = dict(do=do, dht=dht)
    if device != gdev:
        out = {kk: (vv.to(device) if isinstance(vv, torch.Tensor) else vv) for kk, vv in out.items()}
    return out


def custom(name: str, B: int, T: int, H: int, seqlens=None, with_h0=False, seed=0,
           gate_div=16.0) -> Workload:
    """A workload with the same distributions and other sizes (tests use these)."""
    return Workload(name, B=B, T=T, H=H, seqlens=tuple(seqlens) if seqlens else None,
                    with_h0=with_h0, seed=seed, gate_div=gate_div)


def make_decode_inputs(N: int, H: int, lens, pool_slots: int, stride: int = 1, spec: bool = False,
                       pad: Sequence[int] = (), seed: int = 0, gate_div: float = 16.0, K: int = 128,
                       V: int = 128, device: str = "cpu", draw_on_device: bool = False):
    """Inputs of the token-by-token (decode) entry point, with the same
    distributions as the forward recipe.

    ``lens`` is an int (fixed length: B = N sequences of that many tokens) or
    a list of N lengths (varlen: B = 1, packed, with cu_seqlens).  The state
    pool is 0.1 * N(0,1) [pool_slots, H, V, K]; each sequence gets ``stride``
    distinct slots drawn without replacement (so no two sequences share one);
    sequences listed in ``pad`` get slot -1 in every column (padding
    entries).  With ``spec`` the accepted-token counts are drawn uniformly
    from [1, stride].  Returns a dict with q, k, v, g, beta, pool, indices
    (int32 [N, stride]), num_accepted (int32 [N] or None), cu_seqlens (int32
    or None), B, T, N."""
    gdev = device if draw_on_device else "cpu"
    gen = torch.Generator(device=gdev)
    gen.manual_seed(int(seed))
    if isinstance(lens, int):
        B, T, seqlens = N, lens, None
    else:
        seqlens = [int(x) for x in lens]
        assert len(seqlens) == N
        B, T = 1, sum(seqlens)
    assert N * stride <= pool_slots

    def randn(shape):
        return torch.randn(shape, generator=gen, dtype=torch.float32, device=gdev)

    def unit_rows(shape):
        x = randn(shape)
        x = x / x.norm(dim=-1, keepdim=True)
        return x.to(torch.bfloat16)

    q = unit_rows((B, T, H, K))
    k = unit_rows((B, T, H, K))
    v = randn((B, T, H, V)).to(torch.bfloat16)
    g = F.logsigmoid(randn((B, T, H, K))) / gate_div
    beta = torch.sigmoid(randn((B, T, H)))
    pool = 0.1 * randn((pool_slots, H, V, K))
    perm = torch.randperm(pool_slots, generator=torch.Generator().manual_seed(int(seed) + 7919))
    indices = perm[: N * stride].reshape(N, stride).to(torch.int32)
    for n in pad:
        indices[n] = -1
    num_accepted = None
    if spec:
        num_accepted = torch.randint(1, stride + 1, (N,), generator=torch.Generator().manual_seed(int(seed) + 31),
                                     dtype=torch.int32)
    cu = None
    if seqlens is not None:
        c = [0]
        for s in seqlens:
            c.append(c[-1] + s)
        cu = torch.tensor(c, dtype=torch.int32)
    out = dict(q=q, k=k, v=v, g=g, beta=beta, pool=pool, indices=indices, num_accepted=num_accepted,
               cu_seqlens=cu, B=B, T=T, N=N)
    if device != "cpu":
        out = {kk: (vv.to(device) if isinstance(vv, torch.Tensor) else vv) for kk, vv in out.items()}
    return out
