"""CPU-side checks of the C-ABI library: it builds, loads, exports every
function include/kda.h declares, sizes the workspace, and rejects invalid
arguments on the host before any CUDA call.  No compute runs here."""

import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    from chunked_gated_delta_kda_gb300 import binding
    lib = binding.load_library()
    names = _declared_functions()
    assert {"kda_fwd", "kda_fwd_workspace_bytes", "kda_get_status", "kda_status_str"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libkda.so does not export {n}"


def test_flag_constants_match_the_header():
    """Every KDA_FLAG_* of include/kda.h has the same value in the Python
    binding, and the flags are distinct single bits."""
    from chunked_gated_delta_kda_gb300 import binding
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    flags = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(KDA_FLAG_[A-Z0-9_]+)\s+(\d+)u", text)}
    assert len(flags) >= 6, flags
    for name, value in flags.items():
        assert getattr(binding, name) == value, name
        assert value > 0 and value & (value - 1) == 0, name
    assert len(set(flags.values())) == len(flags)


def test_debug_constants_match_the_header():
    """The KDA_DEBUG_* selectors of include/kda.h have the binding's values,
    and kda_debug_set rejects an unknown selector without touching a GPU."""
    import re
    from chunked_gated_delta_kda_gb300 import binding
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    sel = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(KDA_DEBUG_[A-Z0-9_]+)\s+(\d+)\b", text)}
    assert sel == {"KDA_DEBUG_WAIT_LIMIT": 1, "KDA_DEBUG_DROP_SCAN_LOAD": 2}
    for name, value in sel.items():
        assert getattr(binding, name) == value
    lib = binding.load_library()
    assert lib.kda_debug_set(99, 0) == 1
    assert lib.kda_debug_set(binding.KDA_DEBUG_WAIT_LIMIT, 0) == 0


def test_workspace_bytes():
    from chunked_gated_delta_kda_gb300 import binding
    lib = binding.load_library()
    tile = 131584
    r256 = lambda b: (b + 255) // 256 * 256
    # header, wide queue, tiles (fixed length: B * T/128 slots; varlen bound:
    # T/128 + N + 1), then one flag word per (sequence, head)
    assert lib.kda_fwd_workspace_bytes(1, 65536, 32, 128, 128, 1) == 256 + r256(514 * 32 * 4) + 514 * 32 * tile + r256(32 * 4)
    assert lib.kda_fwd_workspace_bytes(4, 8192, 16, 128, 128, 4) == 256 + r256(256 * 16 * 4) + 256 * 16 * tile + r256(64 * 4)
    assert lib.kda_fwd_workspace_bytes(1, 9192, 32, 128, 128, 6) == 256 + r256(78 * 32 * 4) + 78 * 32 * tile + r256(192 * 4)
    assert lib.kda_fwd_workspace_bytes(1, 256, 1, 64, 128, 1) == 0


def test_status_strings():
    from chunked_gated_delta_kda_gb300 import binding
    lib = binding.load_library()
    for code in range(8):
        assert lib.kda_status_str(code)
    assert b"unknown" in lib.kda_status_str(99)


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-pointer validation cases run on CPU-only hosts")
def test_host_validation_rejects_before_any_cuda_call():
    """Every case below fails a host check, so no pointer is ever used."""
    from chunked_gated_delta_kda_gb300 import binding
    lib = binding.load_library()
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 256), ctypes.c_void_p)
    ws = lib.kda_fwd_workspace_bytes(1, 256, 1, 128, 128, 1)

    def call(**kw):
        a = dict(q=p, k=p, v=p, g=p, beta=p, scale=0.0, h0=None, cu=None, o=p, ht=None, B=1, T=256,
                 H=1, K=128, V=128, N=1, flags=0, ws=p, wsb=ws)
        a.update(kw)
        return lib.kda_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["h0"], a["cu"], a["o"],
                           a["ht"], a["B"], a["T"], a["H"], a["K"], a["V"], a["N"], a["flags"], a["ws"],
                           a["wsb"], None)

    assert call(K=64) == 2                  # unsupported head size
    assert call(V=256) == 2
    assert call(q=None) == 1                # null tensor
    assert call(ws=None) == 1
    assert call(T=200) == 1                 # fixed length needs T % 128 == 0
    assert call(N=2) == 1                   # fixed length needs N == B
    assert call(B=2, N=2, cu=p) == 1        # varlen needs B == 1
    assert call(wsb=ws - 1) == 1            # workspace too small
    assert call(flags=4) == 1               # unknown flag (a backward-only flag)
    assert call(flags=8) == 1               # save for the backward: workspace below kda_bwd_workspace_bytes
    assert lib.kda_fwd_noalloc(p, p, p, p, p, 0.0, None, None, p, None, 1, 256, 1, 128, 128, 1, 8, None) == 1
    assert call(H=0) == 1
    misaligned = ctypes.c_void_p(p.value + 8)
    assert call(o=misaligned) == 1          # 16-byte alignment
    assert call(ws=misaligned) == 1         # 256-byte workspace alignment


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-pointer validation cases run on CPU-only hosts")
def test_fused_recurrent_host_validation():
    """kda_fused_recurrent's host checks fail before any CUDA call."""
    from chunked_gated_delta_kda_gb300 import binding
    lib = binding.load_library()
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 256), ctypes.c_void_p)

    def call(**kw):
        a = dict(q=p, k=p, v=p, g=p, beta=p, scale=0.0, pool=p, P=4, idx=p, stride=1, acc=None, cu=None, o=p,
                 B=2, T=1, H=1, K=128, V=128, N=2, flags=0, ws=p)
        a.update(kw)
        return lib.kda_fused_recurrent(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["pool"], a["P"],
                                       a["idx"], a["stride"], a["acc"], a["cu"], a["o"], a["B"], a["T"], a["H"],
                                       a["K"], a["V"], a["N"], a["flags"], a["ws"], None)

    assert call(K=64) == 2
    assert call(V=64) == 2
    assert call(pool=None) == 1
    assert call(idx=None) == 1
    assert call(ws=None) == 1
    assert call(q=None) == 1
    assert call(P=0) == 1
    assert call(stride=0) == 1
    assert call(N=3) == 1                   # fixed length needs N == B
    assert call(cu=p) == 1                  # varlen needs B == 1
    assert call(flags=2) == 1
    misaligned = ctypes.c_void_p(p.value + 8)
    assert call(pool=misaligned) == 1
    assert call(ws=misaligned) == 1


def test_decode_status_string():
    from chunked_gated_delta_kda_gb300 import binding
    lib = binding.load_library()
    assert b"slot" in lib.kda_status_str(7)


def test_kcp_workspace_and_host_checks():
    """kda_kcp_fwd's size function and its host-side checks (which run before
    any CUDA call: unsupported sizes and invalid host offsets)."""
    from chunked_gated_delta_kda_gb300 import binding
    lib = binding.load_library()
    assert lib.kda_kcp_workspace_bytes(1024, 4, 128, 128, 2, 2) > 0
    assert lib.kda_kcp_workspace_bytes(1024, 4, 64, 128, 2, 2) == 0
    assert lib.kda_kcp_workspace_bytes(1024, 4, 128, 128, 2, 0) == 0
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 256), ctypes.c_void_p)
    cu_bad = (ctypes.c_int32 * 3)(0, 200, 100)
    big = 1 << 40
    args = [p, p, p, p, p, 0.0, None, cu_bad, p, None, 100, 1, 128, 128, 2, 2, 0, p, big, None]
    assert lib.kda_kcp_fwd(*args) == 4          # offsets not non-decreasing
    args[12] = 64
    assert lib.kda_kcp_fwd(*args) == 2          # K != 128


def test_bwd_workspace_and_host_checks():
    """kda_bwd's workspace formula and its host-side checks (all fail before
    any CUDA call)."""
    from chunked_gated_delta_kda_gb300 import binding
    lib = binding.load_library()
    state = 128 * 128 * 4
    tile = 131584
    r256 = lambda b: (b + 255) // 256 * 256

    def expect(slots, H, N):
        # header + wide queue, forward tiles, exact flags, reversed tiles,
        # three state checkpoints per (slot, head), one skip word per item, then
        # min(max(items, N H), 152) scratch buffers of 128 states
        items = slots * H
        ctas = min(max(items, N * H), 152)
        return 256 + r256(items * 4) + items * tile + r256(N * H * 4) + items * tile + 3 * items * state + \
            r256(items * 4) + ctas * 128 * state

    assert lib.kda_bwd_workspace_bytes(1, 65536, 32, 128, 128, 1) == expect(514, 32, 1)
    assert lib.kda_bwd_workspace_bytes(4, 8192, 16, 128, 128, 4) == expect(256, 16, 4)
    assert lib.kda_bwd_workspace_bytes(1, 9192, 32, 128, 128, 6) == expect(78, 32, 6)
    assert lib.kda_bwd_workspace_bytes(1, 128, 1, 128, 128, 1) == expect(3, 1, 1)   # varlen bound T/128 + N + 1
    assert lib.kda_bwd_workspace_bytes(1, 256, 1, 64, 128, 1) == 0
    if torch.cuda.is_available():
        return
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 256), ctypes.c_void_p)
    ws = lib.kda_bwd_workspace_bytes(1, 256, 1, 128, 128, 1)

    def call(**kw):
        a = dict(q=p, k=p, v=p, g=p, beta=p, scale=0.0, h0=None, cu=None, do=p, dht=None, dq=p, dk=p, dv=p,
                 dg=p, db=p, dh0=None, B=1, T=256, H=1, K=128, V=128, N=1, flags=0, ws=p, wsb=ws)
        a.update(kw)
        return lib.kda_bwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["h0"], a["cu"], a["do"],
                           a["dht"], a["dq"], a["dk"], a["dv"], a["dg"], a["db"], a["dh0"], a["B"], a["T"], a["H"],
                           a["K"], a["V"], a["N"], a["flags"], a["ws"], a["wsb"], None)

    assert call(K=64) == 2
    assert call(do=None) == 1
    assert call(dg=None) == 1
    assert call(db=None) == 1
    assert call(T=200) == 1
    assert call(N=2) == 1
    assert call(B=2, N=2, cu=p) == 1
    assert call(wsb=ws - 1) == 1
    assert call(flags=8) == 1                # the forward's save flag
    assert call(flags=64) == 1
    assert call(flags=16 | 2) == 1           # reusing a saved forward is not for the token path
    misaligned = ctypes.c_void_p(p.value + 8)
    assert call(dq=misaligned) == 1
    assert call(dh0=misaligned) == 1
    assert call(ws=misaligned) == 1
