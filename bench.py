#!/usr/bin/env python
"""Benchmark of the chunked KDA forward on GB300.

One step = one full forward (every stage of the hot path) over the workload's
synthetic inputs, already resident in HBM.  Default workload: B=1, T=65536,
H=32, K=V=128 (the large named workload), whose 2.7 GB of inputs per step
exceed the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 oracle
on the host cores instead (the reference arm; no public implementation of
this method exists to run).
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from chunked_gated_delta_kda_gb300.inputs import WORKLOADS, custom, make_inputs  # noqa: E402

METRIC = "KDA fwd tokens*heads/s and TFLOP/s, % of roofline, at T=64K H=32 K=V=128"
UNIT = "token*heads/s"
N128 = 128
# Algorithmic work per token-head (n = 128, triangular products at their
# triangular size): 11 1/3 n^2 flop; dense-tile count 16 1/3 n^2.
ALG_FLOP_PER_TH = (34.0 / 3.0) * N128 * N128
DENSE_FLOP_PER_TH = (49.0 / 3.0) * N128 * N128
# Algorithmic HBM bytes per token-head: q, k, v bf16 (3 x 256) + g fp32 512
# + beta 4 + o bf16 256.  The chunk-parallel kernel's share is the inputs
# (1284 B), the scan kernel's share the output (256 B) plus state I/O.
BYTES_PER_TH = 1540
PREP_BYTES_PER_TH = 1284
SCAN_BYTES_PER_TH = 256
STATE_BYTES = N128 * N128 * 4


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def load_traffic():
    """Per-kernel DRAM traffic (bytes per token-head) from the committed ncu
    summary, keyed by the source hash it was captured on; a kernel whose
    source changed since reads as None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.md")
    out = {}
    if not os.path.exists(path):
        return out
    src_dir = os.path.join(ROOT, "chunked_gated_delta_kda_gb300", "csrc")
    with open(path) as f:
        for line in f:
            parts = [p.strip() for p in line.strip().strip("|").split("|")]
            if len(parts) >= 4 and parts[0].startswith("kda_"):
                kernel, fname, sha, per_th = parts[0], parts[1], parts[2], parts[3]
                fp = os.path.join(src_dir, fname)
                if not os.path.exists(fp):
                    continue
                cur = hashlib.sha256(open(fp, "rb").read()).hexdigest()[:12]
                try:
                    out[kernel] = float(per_th) if cur == sha else None
                except ValueError:
                    out[kernel] = None
    return out


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start, t_end):
        rows = []
        for ts, line in self.lines:
            if t_start <= ts <= t_end + 0.05:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 7:
                    rows.append(parts)
        if not rows:
            rows = [[p.strip() for p in l.split(",")] for _, l in self.lines[-3:] if l.count(",") >= 6]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def algorithmic(w, N):
    th = w.B * w.T * w.H
    state_io = (STATE_BYTES * N * w.H) * (2 if w.with_h0 else 1)
    return th, th * BYTES_PER_TH + state_io, th * ALG_FLOP_PER_TH, th * DENSE_FLOP_PER_TH


# ---------------------------------------------------------------------------
# Ranks: one process per GPU; the (sequence, head) units of a step are
# independent, so every rank runs its own full copy of the workload (weak
# scaling) and the only collectives are the barrier around the timed region
# and the max of the elapsed times.
# ---------------------------------------------------------------------------

def rank_env():
    """(world, rank, local_rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, device, world: int) -> float:
    """Max of a per-rank number over all ranks (all_reduce MAX; the identity
    at world 1)."""
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: int, world: int, slowest_ms_per_step: float) -> float:
    """Whole-job throughput: the units every rank processed, over the slowest
    rank's time."""
    return world * units_per_rank / (slowest_ms_per_step * 1e-3)


# ---------------------------------------------------------------------------
# CPU baseline / reference arm: the fp64 oracle on a bounded sample
# ---------------------------------------------------------------------------

def oracle_rate(w, target_s=10.0, max_tokens=None):
    """Time the oracle (as it stands) on the first T_s tokens of the workload,
    all heads; T_s sized so the run takes about ``target_s`` seconds."""
    import oracle
    threads = oracle.max_threads()
    H = w.H

    def run(Ts):
        x = make_inputs(custom("sample", B=1, T=Ts, H=H, seed=w.seed))
        args = [x[n].float().numpy() for n in ("q", "k", "v", "g", "beta")]
        t0 = time.perf_counter()
        oracle.kda_recurrent(*args)
        return time.perf_counter() - t0

    Ts = 128
    dt = run(Ts)
    while dt < target_s / 8 and Ts < (max_tokens or w.T):
        Ts = min(Ts * 4, max_tokens or w.T)
        dt = run(Ts)
    if dt < target_s / 2 and Ts < (max_tokens or w.T):
        Ts = min(int(Ts * target_s / max(dt, 1e-3)), max_tokens or w.T)
        dt = run(Ts)
    return {"value": Ts * H / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"fp64 per-token recurrence (C, OpenMP over heads) on the first {Ts} tokens x {H} heads "
                      f"of the {w.name} workload ({Ts * H} token-heads, {dt:.1f} s)",
            "seconds": dt, "tokens": Ts}


def run_reference(args, w, rank, world):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cal = oracle_rate(w, target_s=2.0)
    per_step_s = max(0.05, min(1.0, 120.0 / max(1, args.steps + args.warmup)))
    Ts = max(8, min(w.T, int(cal["tokens"] * per_step_s / max(cal["seconds"], 1e-3))))
    x = make_inputs(custom("ref", B=1, T=Ts, H=w.H, seed=w.seed))
    a = [x[n].float().numpy() for n in ("q", "k", "v", "g", "beta")]
    for _ in range(args.warmup):
        oracle.kda_recurrent(*a)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.kda_recurrent(*a)
    dt = (time.perf_counter() - t0) / args.steps
    value = Ts * w.H / dt
    th, _, _, _ = algorithmic(w, w.N)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "runs_on": "host cores (the fp64 oracle; no GPU work)",
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V,
                       "step": f"bounded sample: first {Ts} tokens x {w.H} heads of the workload"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cal["cores"], "kind": "oracle",
                             "sample": f"first {Ts} tokens x {w.H} heads per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Decode (token-by-token entry point)
# ---------------------------------------------------------------------------

DECODE_METRIC = "KDA decode (token-by-token, in-place state pool) token*heads/s"
DECODE_N, DECODE_H, DECODE_POOL = 256, 32, 512
# Per (sequence, head) and token: the fp32 state read and written once
# (2 x 64 KiB) plus q, k, v, o bf16 (4 x 256 B), g fp32 512 B, beta 4 B.
DECODE_BYTES_PER_UNIT = 2 * STATE_BYTES + 4 * 256 + 512 + 4


def decode_oracle_rate(x, target_s):
    import oracle
    n = 1
    while True:
        sl = {k: x[k][:n].float().cpu().numpy() for k in ("q", "k", "v", "g", "beta")}
        # the slots the sample touches, renumbered 0..n-1 (the oracle copies its pool)
        sub = x["pool"][x["indices"][:n, 0].long()].cpu().numpy()
        t0 = time.perf_counter()
        oracle.fused_recurrent(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], sub, np.arange(n))
        dt = time.perf_counter() - t0
        if dt > target_s / 4 or n >= DECODE_N:
            break
        n = min(DECODE_N, n * 4)
    return {"value": n * DECODE_H / dt, "unit": UNIT, "cores": 1, "kind": "oracle", "seconds": dt,
            "sample": f"fp64 numpy decode oracle, {n} sequences x {DECODE_H} heads x 1 token ({dt:.1f} s)"}


def run_decode(args, rank, world, local):
    from chunked_gated_delta_kda_gb300 import binding
    from chunked_gated_delta_kda_gb300.inputs import make_decode_inputs
    name = f"decode_n{DECODE_N}_h{DECODE_H}_pool{DECODE_POOL}"
    if args.impl == "reference":
        if rank != 0:
            return 0
        x = make_decode_inputs(DECODE_N, DECODE_H, 1, pool_slots=DECODE_POOL, seed=5)
        cb = decode_oracle_rate(x, target_s=max(1.0, 60.0 / max(1, args.steps + args.warmup)))
        line = {"impl": "reference", "metric": DECODE_METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": world,
                "runs_on": "host cores (the fp64 oracle; no GPU work)",
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["seconds"] * 1e3,
                "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": {"workload": name},
                "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load_library()
    x = make_decode_inputs(DECODE_N, DECODE_H, 1, pool_slots=DECODE_POOL, seed=5 + rank, device=str(dev))
    q, k, v, g, beta, pool = (x[n] for n in ("q", "k", "v", "g", "beta", "pool"))
    # two disjoint slot sets, alternated between steps: the 1 GiB touched per
    # pair of steps is far larger than L2, so no step reads a cached state
    perm = torch.randperm(DECODE_POOL, generator=torch.Generator().manual_seed(11)).to(torch.int32)
    idx = [perm[:DECODE_N].reshape(-1, 1).to(dev), perm[DECODE_N:].reshape(-1, 1).to(dev)]
    o = torch.empty((DECODE_N, 1, DECODE_H, 128), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        binding.kda_fused_recurrent(q, k, v, g, beta, None, pool, idx[i & 1], None, None, o, DECODE_N, 0, ws)

    for i in range(args.warmup):
        step(i)
    assert binding.get_status(ws) == 0
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_start = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    clocks.stop()
    assert binding.get_status(ws) == 0
    ms = max_over_ranks(e0.elapsed_time(e1), dev, world) / args.steps
    units = DECODE_N * DECODE_H
    peaks = load_peaks()
    achieved = units * DECODE_BYTES_PER_UNIT / (ms * 1e-3) / 1e9
    tr = load_traffic().get("kda_recurrent_kernel")
    line = {"metric": DECODE_METRIC, "value": job_rate(units, world, ms), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": name, "sequences": DECODE_N, "H": DECODE_H, "tokens_per_sequence": 1,
                       "pool_slots": DECODE_POOL,
                       "l2_between_steps": "alternating disjoint slot sets, 1 GiB of state per step pair; no flush"},
            "roofline": {"kernel": "kda_recurrent_kernel", "bound": "hbm", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": (tr * units if tr is not None else None),
                         "alg_bytes_per_launch": units * DECODE_BYTES_PER_UNIT, "ms_per_launch": ms},
            "gpu_launches": args.steps}
    if args.e2e_steps > 0:
        host = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta")}
        dbuf = {n: torch.empty_like(x[n]) for n in host}
        o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(args.e2e_steps):
            for n, tt in host.items():
                dbuf[n].copy_(tt, non_blocking=True)
            binding.kda_fused_recurrent(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["g"], dbuf["beta"], None, pool,
                                        idx[i & 1], None, None, o, DECODE_N, 0, ws)
            o_host.copy_(o, non_blocking=True)
        f1.record(stream)
        torch.cuda.synchronize(dev)
        te = max_over_ranks(f0.elapsed_time(f1) / args.e2e_steps, dev, world)
        line["e2e"] = {"value": job_rate(units, world, te), "unit": UNIT,
                       "h2d_bytes_per_step": sum(tt.numel() * tt.element_size() for tt in host.values()),
                       "d2h_bytes_per_step": o_host.numel() * o_host.element_size(), "ms_per_step": te}
    line["clocks"] = clocks.summary(t_start, t_end)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = decode_oracle_rate({kk: (vv.cpu() if isinstance(vv, torch.Tensor) else vv)
                                                   for kk, vv in x.items()}, target_s=min(args.cpu_seconds, 10.0))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# KCP forward with the ranks simulated on one GPU
# ---------------------------------------------------------------------------

KCP_METRIC = "KDA KCP forward (ranks simulated on one GPU) token*heads/s at T=64K H=32 K=V=128"


def run_kcp(args, rank, world, local, w):
    """The KCP forward of the workload packed as one batch of sequences, with
    --kcp-world ranks simulated on this GPU (per rank: the pre-process of its
    last piece, the merge, its local forward; all on one stream, so the
    ranks run one after another), beside the unsplit forward of the same
    inputs.  The C entry point is called with preallocated buffers."""
    import ctypes
    from chunked_gated_delta_kda_gb300 import binding
    W = args.kcp_world
    name = f"{w.name}_kcp{W}"
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the forward "
                              "(bench.py --impl reference); the KCP simulator has no separate one"}), flush=True)
        return 0
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = binding.load_library()
    x = make_inputs(w, device=str(dev), draw_on_device=True, seed_offset=rank)
    q, k, v, g, beta, h0 = (x[nn] for nn in ("q", "k", "v", "g", "beta", "h0"))
    B, T, H = w.B, w.T, w.H
    # packed: B fixed-length sequences become one batch of B sequences (a
    # varlen workload is packed already)
    q, k, v, g, beta = (t.reshape((1, B * T) + tuple(t.shape[2:])) for t in (q, k, v, g, beta))
    N = w.N
    cu_host = torch.tensor([i * T for i in range(N + 1)], dtype=torch.int32) if w.seqlens is None else \
        torch.tensor([0] + list(np.cumsum(w.seqlens)), dtype=torch.int32)
    Tp = int(cu_host[-1])
    o = torch.empty((1, Tp, H, w.V), dtype=torch.bfloat16, device=dev)
    ht = torch.empty((N, H, w.V, w.K), dtype=torch.float32, device=dev)
    nbytes = int(lib.kda_kcp_workspace_bytes(Tp, H, w.K, w.V, N, W))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None

    def step():
        rc = lib.kda_kcp_fwd(ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), -1.0, ptr(h0), ctypes.c_void_p(cu_host.data_ptr()),
                             ptr(o), ptr(ht), Tp, H, w.K, w.V, N, W, 0, ptr(ws), nbytes,
                             ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, f"kda_kcp_fwd: {rc}"

    cu_dev = cu_host.to(dev)
    fws = torch.empty(binding.workspace_bytes(1, Tp, H, N), dtype=torch.uint8, device=dev)

    def unsplit():
        binding.kda_fwd(q, k, v, g, beta, None, h0, cu_dev, o, ht, N, 0, fws)

    def timed(fn, steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps

    for _ in range(args.warmup):
        step()
        unsplit()
    assert binding.get_status(ws) == 0
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_start = time.time()
    ms = max_over_ranks(timed(step, args.steps), dev, world)
    t_end = time.time()
    clocks.stop()
    ms_unsplit = timed(unsplit, args.steps)
    th, alg_bytes, _, _ = algorithmic(w, N)
    peaks = load_peaks()
    # the simulated ranks run in series: local forwards over every token, plus
    # for every rank whose last piece continues two forwards of that piece
    n_carry = sum(1 for r in range(W - 1) if (r + 1) * Tp // W not in set(cu_host.tolist()))
    line = {"metric": KCP_METRIC, "value": job_rate(th, world, ms), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in/out; fp16 MMA operands, fp32 accumulate, fp32 state",
            "data": "synthetic",
            "config": {"workload": name, "T": Tp, "H": H, "sequences": N, "world_size_simulated": W,
                       "ranks_carrying_state": n_carry,
                       "l2_between_steps": "inputs (2.7 GB per step at T=64K H=32) larger than L2; no flush"},
            "unsplit_forward_ms": ms_unsplit,
            "path_roofline": {"bound": "hbm", "alg_bytes": alg_bytes, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "achieved": alg_bytes / (ms * 1e-3) / 1e9,
                              "frac": alg_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                              "note": "the simulator replays each carrying rank's last piece twice (pre-process) "
                                      "and runs the ranks in series"},
            # per forward: fast prep, wide prep, scan, exact recompute; plus the
            # identity kernel and one merge per carrying rank
            "gpu_launches": args.steps * (4 * (W + 2 * n_carry) + (1 + n_carry if n_carry else 0)),
            "clocks": clocks.summary(t_start, t_end)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# Backward (gradients of <do, o> + <dht, ht>)
# ---------------------------------------------------------------------------

BWD_METRIC = "KDA bwd (dq, dk, dv, dg, dbeta, dh0) token*heads/s at T=64K H=32 K=V=128"
# The per-chunk kernel (chunked chain rule, kda_bwd_tc_kernel): algorithmic HBM
# bytes per token-head = q, k, v, do bf16 (4 x 256) + g fp32 512 + beta 4 + the
# chunk's entering state and exit state gradient (2 x 64 KiB per 128 tokens:
# 1024) + dq, dk, dg fp32 (3 x 512) + dv fp32 512 + dbeta 4; algorithmic flop
# per token-head = its sixteen 128 x 128 x 128 products at their triangular
# sizes (5 dense + 11 triangular: 10.5 x 2 n^3 per chunk) plus the triangular
# inverse (2/3 n^3), over n = 128 tokens.
BWD_TC_BYTES_PER_TH = 4 * 256 + 512 + 4 + 1024 + 3 * 512 + 512 + 4
BWD_TC_FLOP_PER_TH = (21.0 + 2.0 / 3.0) * N128 * N128
# TF32 dense peak: the measured bf16 peak x the nominal TF32 / bf16 ratio (1.1 / 2.25).
TF32_OVER_BF16 = 1.1 / 2.25


def bwd_oracle_rate(w, target_s):
    """The gradient oracle (torch fp64 autograd, as it stands) on the first
    Ts tokens of the workload, all heads."""
    from oracle import backward as obw
    from chunked_gated_delta_kda_gb300.inputs import make_grad_inputs
    Ts, dt = 4, 0.0
    while True:
        x = make_inputs(custom("sample", B=1, T=Ts, H=w.H, seed=w.seed))
        gr = make_grad_inputs(custom("sample", B=1, T=Ts, H=w.H, seed=w.seed))
        a = [x[n].float().numpy() for n in ("q", "k", "v", "g", "beta")]
        t0 = time.perf_counter()
        obw.kda_backward(*a, gr["do"].float().numpy(), dht=gr["dht"].numpy())
        dt = time.perf_counter() - t0
        # the autograd graph grows with T, so the cost is superlinear: double
        # only while the next run is predicted to stay within the target
        if dt * 4 > target_s or Ts >= w.T:
            break
        Ts = min(w.T, Ts * 2)
    return {"value": Ts * w.H / dt, "unit": UNIT, "cores": torch.get_num_threads(), "kind": "oracle", "seconds": dt,
            "sample": f"fp64 torch autograd through the per-token recurrence on the first {Ts} tokens x {w.H} heads "
                      f"of the {w.name} workload ({dt:.1f} s)"}


def run_bwd(args, rank, world, local, w):
    from chunked_gated_delta_kda_gb300 import binding
    from chunked_gated_delta_kda_gb300.inputs import make_grad_inputs
    if args.impl == "reference":
        if rank != 0:
            return 0
        cb = bwd_oracle_rate(w, target_s=max(2.0, 60.0 / max(1, args.steps + args.warmup)))
        line = {"impl": "reference", "metric": BWD_METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": world,
                "runs_on": "host cores (the fp64 oracle; no GPU work)",
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["seconds"] * 1e3,
                "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": {"workload": w.name},
                "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load_library()
    x = make_inputs(w, device=str(dev), draw_on_device=True, seed_offset=rank)
    gr = make_grad_inputs(w, device=str(dev), draw_on_device=True, seed_offset=rank)
    B, T, H, N = w.B, w.T, w.H, w.N
    q, k, v, g, beta, h0, cu = (x[n] for n in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    do, dht = gr["do"], gr["dht"]
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk, dg = (torch.empty((B, T, H, 128), **f32) for _ in range(3))
    dv = torch.empty((B, T, H, 128), **f32)
    dbeta = torch.empty((B, T, H), **f32)
    dh0 = torch.empty((N, H, 128, 128), **f32)
    ws = torch.empty(binding.bwd_workspace_bytes(B, T, H, N), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for six in ev:             # torch creates the CUDA event on first record
        for e in six:
            e.record(stream)

    def step(i, timed):
        args_ = (q, k, v, g, beta, None, h0, cu, do, dht, dq, dk, dv, dg, dbeta, dh0, N, 0, ws)
        if timed:
            binding.kda_bwd_timed(*args_, ev[i])
        else:
            binding.kda_bwd(*args_)

    for i in range(args.warmup):
        step(i, False)
    assert binding.get_status(ws) == 0
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_start = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i, True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    clocks.stop()
    assert binding.get_status(ws) == 0
    ms = max_over_ranks(e0.elapsed_time(e1), dev, world) / args.steps
    stages = ["forward_replay", "transposed_tiles", "reverse_state_pass", "chunk_chain_rule", "rest"]
    # chunk_chain_rule = the tensor-core per-chunk kernel and the per-token kernel for the chunks it left
    stage_ms = {nm: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev) for j, nm in enumerate(stages)}
    # training path: one forward that saves its chunk states, then backwards that reuse them
    o_tmp = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=dev)
    binding.kda_fwd(q, k, v, g, beta, None, h0, cu, o_tmp, None, N, binding.KDA_FLAG_SAVE_FOR_BWD, ws)
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for i in range(args.steps):
        binding.kda_bwd(q, k, v, g, beta, None, h0, cu, do, dht, dq, dk, dv, dg, dbeta, dh0, N,
                        binding.KDA_FLAG_BWD_REUSE_FWD, ws)
    r1.record(stream)
    torch.cuda.synchronize(dev)
    assert binding.get_status(ws) == 0
    ms_reuse = max_over_ranks(r0.elapsed_time(r1), dev, world) / args.steps
    del o_tmp
    th = B * T * H
    ck = clocks.summary(t_start, t_end)
    peaks = load_peaks()
    k_ms = stage_ms["chunk_chain_rule"]
    tf32_peak = peaks["bf16_tflops"] * TF32_OVER_BF16
    t_hbm = th * BWD_TC_BYTES_PER_TH / (peaks["hbm_gbs"] * 1e9) * 1e3
    t_tc = th * BWD_TC_FLOP_PER_TH / (tf32_peak * 1e12) * 1e3
    gbs = th * BWD_TC_BYTES_PER_TH / (k_ms * 1e-3) / 1e9
    tfl = th * BWD_TC_FLOP_PER_TH / (k_ms * 1e-3) / 1e12
    tr = load_traffic().get("kda_bwd_tc_kernel")
    if t_hbm >= t_tc:
        roof = {"kernel": "kda_bwd_tc_kernel", "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"]}
    else:
        roof = {"kernel": "kda_bwd_tc_kernel", "bound": "tensor", "achieved": tfl, "peak": tf32_peak,
                "unit": "TFLOP/s", "frac": tfl / tf32_peak}
    roof.update({"traffic": (tr * th if tr is not None else None),
                 "alg_bytes_per_launch": th * BWD_TC_BYTES_PER_TH, "alg_flop_per_launch": th * BWD_TC_FLOP_PER_TH,
                 "ms_per_launch": k_ms, "tensor_tflops": tfl, "tensor_peak_tf32": tf32_peak,
                 "peak_source": f"{peaks['source']} (HBM copy; TF32 = bf16 x 1.1/2.25)",
                 "t_hbm_ms": t_hbm, "t_tensor_ms": t_tc})
    line = {"metric": BWD_METRIC, "value": job_rate(th, world, ms), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": B, "T": T, "H": H, "K": 128, "V": 128,
                       "l2_between_steps": "inputs and workspace (several GB) exceed L2; no flush"},
            "stage_ms": stage_ms,
            "ms_per_step_reusing_saved_forward": ms_reuse,
            "roofline": roof,
            "gpu_launches": 8 * args.steps}
    if args.e2e_steps > 0:
        host_in = {n: t.cpu().pin_memory() for n, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta),
                                                        ("do", do), ("dht", dht))}
        outs = (dq, dk, dv, dg, dbeta, dh0)
        sets = []
        for _ in range(2):   # double-buffered: the copies of one step overlap the backward of the other
            sets.append({
                "in": {n: torch.empty_like(t, device=dev) for n, t in host_in.items()},
                "out": [torch.empty_like(t) for t in outs], "ws": torch.empty_like(ws),
                "host_out": [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs],
                "in_done": torch.cuda.Event(), "bwd_done": torch.cuda.Event(), "out_done": torch.cuda.Event(),
            })
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_run(steps):
            for i in range(steps):
                b = sets[i % 2]
                with torch.cuda.stream(s_in):          # inputs of step i
                    s_in.wait_event(b["bwd_done"])     # the backward of step i-2 has read this set
                    for n, t in host_in.items():
                        b["in"][n].copy_(t, non_blocking=True)
                    b["in_done"].record(s_in)
                stream.wait_event(b["in_done"])
                stream.wait_event(b["out_done"])       # the gradient copies of step i-2 are done
                d, o_ = b["in"], b["out"]
                binding.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, h0, cu, d["do"], d["dht"],
                                o_[0], o_[1], o_[2], o_[3], o_[4], o_[5], N, 0, b["ws"])
                b["bwd_done"].record(stream)
                with torch.cuda.stream(s_out):         # gradients of step i
                    s_out.wait_event(b["bwd_done"])
                    for ho, t in zip(b["host_out"], o_):
                        ho.copy_(t, non_blocking=True)
                    b["out_done"].record(s_out)

        e2e_run(2)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e2e_run(args.e2e_steps)
        torch.cuda.synchronize(dev)
        te = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.e2e_steps, dev, world)
        line["e2e"] = {"value": job_rate(th, world, te), "unit": UNIT,
                       "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in.values()),
                       "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outs), "ms_per_step": te,
                       "timing": "host wall clock around the whole run, synchronised on both sides",
                       "pipelining": "input copy of step i+1 and gradient copy of step i-1 overlap the backward of step i"}
    line["clocks"] = ck
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = bwd_oracle_rate(w, target_s=min(args.cpu_seconds, 10.0))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="t65536_h32", choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--gate-div", type=float, default=None,
                    help="forward: divide logsigmoid(N(0,1)) by this for g instead of the workload's 16 "
                         "(1 = the pages' unscaled stable-input gates, whose chunks take the wide prep kernel)")
    ap.add_argument("--op", choices=["fwd", "decode", "bwd", "kcp"], default="fwd",
                    help="fwd: the chunked forward (default); decode: the token-by-token entry point; "
                         "bwd: the chunked backward; kcp: the KCP forward with --kcp-world ranks simulated "
                         "on this GPU")
    ap.add_argument("--kcp-world", type=int, default=4, help="simulated ranks for --op kcp")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"

    world, rank, local = rank_env()
    w = WORKLOADS[args.workload]
    if args.gate_div is not None:
        assert args.op == "fwd", "--gate-div applies to the forward"
        w = dataclasses.replace(w, gate_div=args.gate_div)

    if args.op == "decode":
        return run_decode(args, rank, world, local)
    if args.op == "bwd":
        return run_bwd(args, rank, world, local, w)
    if args.op == "kcp":
        return run_kcp(args, rank, world, local, w)
    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    import torch.distributed as dist
    from chunked_gated_delta_kda_gb300 import binding
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load_library()

    # Weak scaling: every rank runs the full workload on its own GPU (the
    # (sequence, head) units are independent; no data-path collective).
    x = make_inputs(w, device=str(dev), draw_on_device=True, seed_offset=rank)
    q, k, v, g, beta, h0, cu = (x[n] for n in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    N, H, B, T = w.N, w.H, w.B, w.T
    o = torch.empty((B, T, H, w.V), dtype=torch.bfloat16, device=dev)
    ht = torch.empty((N, H, w.V, w.K), dtype=torch.float32, device=dev)
    ws = torch.empty(binding.workspace_bytes(B, T, H, N), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.kda_fwd(q, k, v, g, beta, None, h0, cu, o, ht, N, 0, ws)

    for _ in range(args.warmup):
        step()
    st = binding.get_status(ws)
    assert st == 0, f"device status {st}"

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for trio in ev:            # torch creates the CUDA event on first record
        for e in trio:
            e.record(stream)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_start = time.time()
    e0.record(stream)
    for i in range(args.steps):
        binding.kda_fwd_timed(q, k, v, g, beta, None, h0, cu, o, ht, N, 0, ws, ev[i])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    if world > 1:
        dist.barrier()
    clocks.stop()
    total_ms = e0.elapsed_time(e1)
    prep_ms = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)) / args.steps
    scan_ms = sum(ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)) / args.steps
    st = binding.get_status(ws)
    assert st == 0, f"device status {st}"
    # chunks the last step queued for the wide (bf16) prep kernel: word 1 of
    # the workspace header
    wide_chunks = int(ws[4:8].view(torch.int32).item())

    ms_per_step = max_over_ranks(total_ms, dev, world) / args.steps

    th, alg_bytes, alg_flop, dense_flop = algorithmic(w, N)
    value = job_rate(th, world, ms_per_step)
    peaks = load_peaks()
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg_flop / (peaks["bf16_tflops_sustained"] * 1e12)
    t_roof = max(t_hbm, t_tc)
    traffic = load_traffic()

    stages = {
        "kda_prep_kernel": {"ms": prep_ms, "alg_bytes": th * PREP_BYTES_PER_TH},
        "kda_scan_kernel": {"ms": scan_ms, "alg_bytes": th * SCAN_BYTES_PER_TH + STATE_BYTES * N * H * (2 if h0 is not None else 1)},
    }
    dom = max(stages, key=lambda s: stages[s]["ms"])
    d = stages[dom]
    achieved = d["alg_bytes"] / (d["ms"] * 1e-3) / 1e9
    # the committed traffic row is the fast prep kernel's: it does not
    # describe a step whose chunks went to the wide kernel
    tr = traffic.get(dom) if (dom != "kda_prep_kernel" or wide_chunks == 0) else None
    roofline = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "traffic": (tr * th if tr is not None else None),
                "peak_source": f"{peaks['source']} (hbm_gbs, MEASURED_PEAKS.json)" if peaks["source"] == "measured"
                else "fallback 6.8 TB/s",
                "alg_bytes_per_launch": d["alg_bytes"], "ms_per_launch": d["ms"]}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in/out; fp16 MMA operands, fp32 accumulate, fp32 state", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "T": T, "H": H, "K": w.K, "V": w.V, "chunk": 128,
                   "h0": h0 is not None, "output_final_state": True, "gate_div": w.gate_div,
                   "wide_chunks": wide_chunks,
                   "l2_between_steps": "inputs (2.7 GB per step) larger than L2 (129 MB); no flush",
                   "inputs": "seeded synthetic, drawn on device with the workload's recipe"},
        "tflops_alg": alg_flop / (ms_per_step * 1e-3) / 1e12,
        "tflops_dense": dense_flop / (ms_per_step * 1e-3) / 1e12,
        "gbs_alg": alg_bytes / (ms_per_step * 1e-3) / 1e9,
        "path_roofline": {"bound": "hbm" if t_hbm >= t_tc else "tensor", "t_roof_us": t_roof * 1e6,
                          "t_hbm_us": t_hbm * 1e6, "t_tensor_us": t_tc * 1e6,
                          "frac": t_roof / (ms_per_step * 1e-3)},
        "stages_ms": {"kda_prep_kernel": prep_ms, "kda_scan_kernel": scan_ms},
        "roofline": roofline,
        "gpu_launches": 4 * args.steps,   # fast prep, wide prep and exact recompute (both exit at once when unused), scan
    }

    # End to end through the public API: pinned host inputs -> device, forward,
    # output and final state -> pinned host, all inside the timed region.  The
    # steps are independent batches, so they are pipelined the way a caller
    # would: the input copy of step i+1 (copy-in stream) and the output copy
    # of step i-1 (copy-out stream) overlap the forward of step i; inputs,
    # outputs and workspaces are double-buffered.
    if args.e2e_steps > 0:
        names = [n for n in ("q", "k", "v", "g", "beta") if x[n] is not None]
        host = {n: x[n].cpu().pin_memory() for n in names}
        if h0 is not None:
            host["h0"] = h0.cpu().pin_memory()
        sets = []
        for _ in range(2):
            sets.append({
                "in": {n: torch.empty_like(x[n] if n != "h0" else h0) for n in host},
                "o": torch.empty_like(o), "ht": torch.empty_like(ht), "ws": torch.empty_like(ws),
                "o_host": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                "ht_host": torch.empty(ht.shape, dtype=ht.dtype).pin_memory(),
                "in_done": torch.cuda.Event(), "fwd_done": torch.cuda.Event(), "out_done": torch.cuda.Event(),
            })
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = o.numel() * o.element_size() + ht.numel() * ht.element_size()
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_run(steps):
            for i in range(steps):
                b = sets[i % 2]
                with torch.cuda.stream(s_in):          # inputs of step i
                    s_in.wait_event(b["fwd_done"])     # the forward of step i-2 has read this set
                    for n, t in host.items():
                        b["in"][n].copy_(t, non_blocking=True)
                    b["in_done"].record(s_in)
                stream.wait_event(b["in_done"])
                stream.wait_event(b["out_done"])       # the output copy of step i-2 has read o / ht
                d = b["in"]
                binding.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d.get("h0"), cu, b["o"], b["ht"],
                                N, 0, b["ws"])
                b["fwd_done"].record(stream)
                with torch.cuda.stream(s_out):         # results of step i
                    s_out.wait_event(b["fwd_done"])
                    b["o_host"].copy_(b["o"], non_blocking=True)
                    b["ht_host"].copy_(b["ht"], non_blocking=True)
                    b["out_done"].record(s_out)

        e2e_run(2)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e2e_run(args.e2e_steps)
        torch.cuda.synchronize(dev)
        te = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.e2e_steps, dev, world)
        line["e2e"] = {"value": job_rate(th, world, te), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": te,
                       "timing": "host wall clock around the whole run, synchronised on both sides",
                       "pipelining": "input copy of step i+1 and output copy of step i-1 overlap the forward of step i"}
        line["gpu_launches_e2e"] = 4 * args.e2e_steps

    line["clocks"] = clocks.summary(t_start, t_end)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_rate(w, target_s=args.cpu_seconds)
        for kk in ("seconds", "tokens"):
            line["cpu_baseline"].pop(kk, None)

    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
