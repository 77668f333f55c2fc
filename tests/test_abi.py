"""The C ABI: the library builds, loads and exports what include/gdr.h declares.

These tests need no GPU: they call only entry points that do host work
(workspace sizing, status strings) and argument validation that rejects a call
before anything is enqueued.
"""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr.h")


@pytest.fixture(scope="session")
def lib():
    from gated_delta_rule_03_gb300 import build, ops
    if not os.path.exists(ops.library_path()):
        build.build()
    return ops._load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdr_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("gdr_chunk_fwd", "gdr_decode_step", "gdr_chunk_fwd_workspace_size",
                 "gdr_status_string", "gdr_read_device_status"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in gdr.h but not exported"


def test_status_strings(lib):
    assert lib.gdr_status_string(0) == b"GDR_OK"
    for code in range(-7, 0):
        assert lib.gdr_status_string(code).startswith(b"GDR_ERR_")
    assert lib.gdr_status_string(-99) == b"GDR_ERR_UNKNOWN"


def test_workspace_size(lib):
    from gated_delta_rule_03_gb300 import chunk_fwd_workspace_size
    import torch
    n1 = chunk_fwd_workspace_size(4, 4 * 4096, 16, 128, 128, 64, torch.bfloat16)
    assert n1 > 0 and n1 % 256 == 0
    n0 = chunk_fwd_workspace_size(1, 256, 2, 64, 64, 64, torch.float32)
    assert n0 > 0
    # unsupported shapes report 0
    assert chunk_fwd_workspace_size(1, 256, 2, 96, 64, 64, torch.float32) == 0
    assert chunk_fwd_workspace_size(1, 256, 2, 64, 64, 32, torch.float32) == 0
    assert chunk_fwd_workspace_size(0, 256, 2, 64, 64, 64, torch.float32) == 0


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_invalid_arguments_rejected_on_the_host(lib):
    A = 0x10000  # 16-byte aligned fake device addresses; never dereferenced on rejection
    p = [_fake(A + i * 0x1000000) for i in range(12)]
    ws_bytes = lib.gdr_chunk_fwd_workspace_size(1, 128, 2, 64, 64, 64, 0)
    base = dict(q=p[0], k=p[1], v=p[2], la=p[3], b=p[4], S0=None, cu=None, n=1, T=128, H=2,
                dk=64, dv=64, C=64, dt=0, o=p[5], Sf=p[6], ws=p[7], wsb=ws_bytes, st=None)

    def call(**kw):
        a = dict(base, **kw)
        return lib.gdr_chunk_fwd(a["q"], a["k"], a["v"], a["la"], a["b"], a["S0"], a["cu"],
                                 a["n"], a["T"], a["H"], a["dk"], a["dv"], a["C"], a["dt"],
                                 a["o"], a["Sf"], a["ws"], a["wsb"], a["st"])

    assert call(q=None) == -1
    assert call(H=0) == -1
    assert call(n=0) == -1
    assert call(n=3) == -1            # 128 tokens do not split into 3 equal sequences
    assert call(dk=96) == -2
    assert call(dv=48) == -2
    assert call(C=32) == -2
    assert call(dt=7) == -2
    assert call(q=_fake(A + 8)) == -3
    assert call(la=_fake(A + 0x3000002)) == -3
    # gates need only 4-byte alignment: this call gets past the alignment check and is
    # rejected by the next one (workspace too small), so nothing is ever launched
    assert call(la=_fake(A + 0x3000004), wsb=ws_bytes - 1) == -4
    assert call(wsb=ws_bytes - 1) == -4
    assert call(ws=None) == -4
    assert call(Sf=p[5]) == -1        # S_final overlapping o

    def dcall(**kw):
        a = dict(q=p[0], k=p[1], v=p[2], la=p[3], b=p[4], S=p[5], o=p[6], N=4, H=2, dk=128,
                 dv=128, dt=1, st=None)
        a.update(kw)
        return lib.gdr_decode_step(a["q"], a["k"], a["v"], a["la"], a["b"], a["S"], a["o"],
                                   a["N"], a["H"], a["dk"], a["dv"], a["dt"], a["st"])

    assert dcall(N=-1) == -1
    assert dcall(dk=32) == -2
    assert dcall(dv=96) == -2
    assert dcall(o=None) == -1
    assert dcall(S=_fake(A + 4)) == -3
    assert dcall(o=p[5]) == -1        # o overlapping S
    assert dcall(N=0) == 0            # nothing to do, nothing enqueued


def test_options_validated_on_the_host(lib):
    # gdr_options: an unknown rule is unsupported, an unknown decay granularity is invalid;
    # both are rejected before any other check, so fake pointers are never touched
    from gated_delta_rule_03_gb300.ops import GdrOptions
    A = 0x10000
    p = [_fake(A + i * 0x1000000) for i in range(12)]
    ws_bytes = lib.gdr_chunk_fwd_workspace_size(1, 128, 2, 64, 64, 64, 0)

    def call(opt):
        return lib.gdr_chunk_fwd_ex(p[0], p[1], p[2], p[3], p[4], None, None, 1, 128, 2, 64, 64,
                                    64, 0, p[5], p[6], p[7], ws_bytes, opt, None)

    def dcall(opt):
        return lib.gdr_decode_step_ex(p[0], p[1], p[2], p[3], p[4], p[5], p[6], 4, 2, 128, 128,
                                      1, opt, None)

    bad_rule = GdrOptions(2)
    bad_decay = GdrOptions(1)
    bad_decay.decay = 2
    for f in (call, dcall):
        assert f(ctypes.byref(bad_rule)) == -2
        assert f(ctypes.byref(bad_decay)) == -1
    # the output-step fields: a weight or an eps without a gate, a negative eps, an
    # unaligned gate
    fake = lambda a: ctypes.c_void_p(a)
    o1 = GdrOptions(0, 0.0, None, A + 0x9000000)
    o2 = GdrOptions(0, 1e-5, None, None)
    o3 = GdrOptions(0, -1.0, A + 0x8000000, None)
    o4 = GdrOptions(0, 0.0, A + 0x8000008, None)
    for f in (call, dcall):
        assert f(ctypes.byref(o1)) == -1
        assert f(ctypes.byref(o2)) == -1
        assert f(ctypes.byref(o3)) == -1
        assert f(ctypes.byref(o4)) == -3
    # the prologue: an unknown kind, a rate without it, an unaligned rate
    p1 = GdrOptions(0, 0.0, None, None, 2, 0, None)
    p2 = GdrOptions(0, 0.0, None, None, 0, 0, A + 0x8000000)
    p3 = GdrOptions(0, 0.0, None, None, 1, 0, A + 0x8000002)
    for f in (call, dcall):
        assert f(ctypes.byref(p1)) == -2
        assert f(ctypes.byref(p2)) == -1
        assert f(ctypes.byref(p3)) == -3
    # a valid options block gets as far as the argument checks of the plain entry points
    ok = GdrOptions(1)
    assert lib.gdr_chunk_fwd_ex(None, p[1], p[2], p[3], p[4], None, None, 1, 128, 2, 64, 64, 64,
                                0, p[5], p[6], p[7], ws_bytes, ctypes.byref(ok), None) == -1
    assert lib.gdr_decode_step_ex(p[0], p[1], p[2], p[3], p[4], p[5], p[6], 0, 2, 128, 128, 1,
                                  ctypes.byref(ok), None) == 0


def test_per_channel_workspace_follows_the_path(lib):
    # per-channel rates: bf16 with d_k = d_v = 128 takes the per-channel tensor-core path,
    # whose workspace holds every unit's operands; other sizes take the exact path, whose
    # layout adds one fp32 [C][d_k] block of cumulative log decay per unit. The plain query
    # (head rates) is unchanged; bad options size nothing.
    from gated_delta_rule_03_gb300.ops import GdrOptions
    head = lib.gdr_chunk_fwd_workspace_size(4, 4 * 4096, 16, 128, 128, 64, 1)
    pc = GdrOptions(0)
    pc.decay = 1
    chan = lib.gdr_chunk_fwd_workspace_size_ex(4, 4 * 4096, 16, 128, 128, 64, 1, ctypes.byref(pc))
    assert lib.gdr_chunk_fwd_workspace_size_ex(4, 4 * 4096, 16, 128, 128, 64, 1, None) == head
    units = (4 * 4096 // 64 + 4) * 16
    # per unit: A^T and T' (2 x 64 x 64 bf16), 384 decay factors, [e^g Q | -W] (64 x 256
    # bf16), decayed K (64 x 128 bf16), U~^T (128 x 64 bf16)
    per_unit = 2 * 64 * 64 * 2 + 384 * 4 + 64 * 256 * 2 + 64 * 128 * 2 + 128 * 64 * 2
    assert units * per_unit <= chan <= units * per_unit + (1 << 20)
    pc.prologue = 1  # (the prologue keeps the tensor-core layout)
    assert lib.gdr_chunk_fwd_workspace_size_ex(4, 4 * 4096, 16, 128, 128, 64, 1,
                                               ctypes.byref(pc)) == chan
    pc.prologue = 0
    exact_chan = lib.gdr_chunk_fwd_workspace_size_ex(4, 4 * 4096, 16, 128, 128, 64, 0,
                                                     ctypes.byref(pc))
    exact_f32 = lib.gdr_chunk_fwd_workspace_size(4, 4 * 4096, 16, 128, 128, 64, 0)
    assert exact_chan >= exact_f32 + units * 64 * 128 * 4
    bad = GdrOptions(0)
    bad.decay = 7
    assert lib.gdr_chunk_fwd_workspace_size_ex(1, 128, 2, 64, 64, 64, 0, ctypes.byref(bad)) == 0


def test_path_query_with_options(lib):
    from gated_delta_rule_03_gb300.ops import GdrOptions
    fn = lib.gdr_chunk_fwd_path_ex
    fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    EXACT, TENSOR, CHANNEL = 0, 1, 2
    opt = lambda decay=0, prologue=0: ctypes.byref(GdrOptions(0, 0.0, None, None, prologue,
                                                              decay, None))
    for dk, dv, dt in [(128, 128, 1), (128, 256, 1), (64, 64, 1), (128, 128, 0)]:
        assert fn(dk, dv, dt, None) == lib.gdr_chunk_fwd_path(dk, dv, dt)
        assert fn(dk, dv, dt, opt()) == lib.gdr_chunk_fwd_path(dk, dv, dt)
    assert fn(128, 128, 1, None) == TENSOR
    assert fn(128, 128, 1, opt(decay=1)) == CHANNEL
    assert fn(128, 128, 1, opt(decay=1, prologue=1)) == CHANNEL
    assert fn(128, 256, 1, opt(decay=1)) == EXACT
    assert fn(128, 128, 0, opt(decay=1)) == EXACT
    assert fn(64, 64, 1, opt(decay=1)) == EXACT
    assert fn(128, 128, 1, opt(decay=7)) == -1  # GDR_ERR_INVALID_ARG
    assert fn(100, 128, 1, opt(decay=1)) < 0


@pytest.mark.parametrize("env", ["GDR_PREFILL_PHASES", "GDR_PREFILL_SEGMENTS"])
def test_schedule_model_on_a_152_sm_device(env, monkeypatch):
    # the schedule selection is host logic: checked here for the workloads' sizes on a
    # device like the target's, without one
    from gated_delta_rule_03_gb300 import ops
    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    monkeypatch.delenv("GDR_PREFILL_SEGMENTS", raising=False)
    bf = torch.bfloat16
    m = lambda *a, **k: ops.chunk_fwd_schedule_model(*a, **k)
    seg = ops.SCHEDULE_SEGMENTED
    assert m(4, 4 * 4096, 16, 128, 128, bf, 152) == 0                     # fused
    assert m(4, 4 * 4096, 16, 128, 128, bf, 152, cooperative=False) == 2   # phased instead
    assert m(8, 34816, 16, 128, 128, bf, 152, varlen=True) == 0            # packed: fused,
    # its solve claiming units (the chains leave at least 16 SMs)
    assert m(8, 34816, 16, 128, 128, bf, 152, varlen=True, cooperative=False) == 1
    assert m(9, 34816, 16, 128, 128, bf, 152, varlen=True) == 1            # 144 chains: phased
    assert m(128, 128 * 2048, 1, 128, 128, bf, 152, varlen=True) == 0      # most sequences
    assert m(129, 129 * 2048, 1, 128, 128, bf, 152, varlen=True) == 1
    assert m(8, 8 * 2047, 16, 128, 128, bf, 152, varlen=True) == 1         # short: phased
    assert m(2, 70000, 16, 128, 256, bf, 152, varlen=True) == 0            # 64 two-slice chains
    assert m(1, 65536, 8, 128, 256, bf, 152) == seg + 7                    # long: 7 segments
    assert m(1, 65536, 8, 128, 256, bf, 40) < seg                          # too few SMs
    assert m(4, 4 * 4096, 16, 128, 128, torch.float32, 152) == 1           # exact path
    assert m(1, 0, 2, 128, 128, bf, 152) == 1                              # nothing to do
    with pytest.raises(Exception):
        m(1, 64, 2, 128, 128, bf, 0)
    # the forcing knobs
    monkeypatch.setenv(env, "3")
    forced = m(1, 65536, 8, 128, 256, bf, 152)
    assert forced == (3 if env == "GDR_PREFILL_PHASES" else seg + 3)


def test_workspace_holds_the_segment_sets_only_when_segmenting_is_possible(lib):
    # few chains over sequences of 64 chunks or more: 29 fp32 state sets of
    # num_seqs * H * d_k * d_v floats (7 each of P, R, discard; 8 starts) are added
    sets = 29 * 1 * 2 * 128 * 128 * 4
    seg = lib.gdr_chunk_fwd_workspace_size(1, 64 * 64, 2, 128, 128, 64, 1)
    plain = lib.gdr_chunk_fwd_workspace_size(1, 63 * 64, 2, 128, 128, 64, 1)
    assert sets <= seg - plain < sets + (1 << 20)
    # many chains: no sets
    many = lib.gdr_chunk_fwd_workspace_size(20, 20 * 64 * 64, 2, 128, 128, 64, 1)
    per_chunk = (lib.gdr_chunk_fwd_workspace_size(20, 20 * 64 * 64 + 20 * 64, 2, 128, 128, 64, 1)
                 - many)
    assert per_chunk < 80 * 1024 * 20  # grows by the per-unit buffers, not by state sets


def test_a_missing_library_fails_loudly(monkeypatch):
    # without the built library every call raises GdrError naming the missing file (no
    # fallback path, and no recursion through the status-text lookup)
    from gated_delta_rule_03_gb300 import ops
    monkeypatch.setattr(ops, "_lib", None)
    monkeypatch.setattr(ops, "_LIB_PATH", "/nonexistent/libgdr.so")
    with pytest.raises(ops.GdrError, match="not found") as e:
        ops.chunk_fwd_workspace_size(1, 64, 2, 64, 64)
    assert e.value.status == -5
    with pytest.raises(ops.GdrError, match="not built"):
        ops.status_string(0)
