"""Adversarial inputs for the chunked forward (test helpers; uses the oracle).

cancellation_stress: the operator page (section "测试与验证体系") describes an
input generator mode that searches 64 random scalings for cancellation in
M4's subtraction v_new = u - w S.  Reading used here: start from a named-recipe
input with an initial state; on the first chunk set the values to the state's
own decayed prediction plus a small perturbation, v_t = s (exp(G_t) k_t)^T S0
+ eps eta_t (then bf16), with the state scaled by s; draw (s, eps) 64 times
(log-uniform s in [0.1, 10], eps in [1e-4, 1]) and keep the draw with the
smallest cancellation ratio ||u - w S|| / max(||u||, ||w S||) over the heads.
"""

from __future__ import annotations

import numpy as np
import torch

from chunked_gated_delta_kda_gb300.inputs import custom, make_inputs
from oracle.chunked import cancellation_ratio


def cancellation_stress(T=384, H=2, seed=0, trials=64):
    x = make_inputs(custom("cancel", B=1, T=T, H=H, seqlens=[T], with_h0=True, seed=seed))
    rng = np.random.default_rng(seed + 1000)
    k = x["k"].double().numpy()[0]
    g = x["g"].double().numpy()[0]
    beta = x["beta"].double().numpy()[0]
    v0 = x["v"].double().numpy()[0]
    h0 = x["h0"].double().numpy()[0]
    L = min(T, 128)
    G = np.cumsum(g[:L], axis=0)                                   # (L, H, K)
    best = None
    for _ in range(trials):
        s = float(np.exp(rng.uniform(np.log(0.1), np.log(10.0))))
        eps = float(np.exp(rng.uniform(np.log(1e-4), np.log(1.0))))
        v = v0.copy()
        ratios = []
        for h in range(H):
            S0 = s * h0[h].T                                       # (K, V)
            pred = (np.exp(G[:, h]) * k[:L, h]) @ S0               # (L, V)
            v[:L, h] = pred + eps * v0[:L, h]
        vb = torch.from_numpy(v).float().bfloat16().double().numpy()
        for h in range(H):
            ratios.append(cancellation_ratio(s * h0[h].T, k[:L, h], vb[:L, h], g[:L, h], beta[:L, h]))
        r = max(ratios)
        if best is None or r < best[0]:
            best = (r, s, eps, vb)
    r, s, eps, vb = best
    y = dict(x)
    y["v"] = torch.from_numpy(vb).float().bfloat16()[None]
    y["h0"] = (s * x["h0"].double()).float()
    return y, {"ratio": r, "state_scale": s, "eps": eps}
