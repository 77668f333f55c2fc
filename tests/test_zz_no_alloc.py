"""gdr_chunk_fwd_noalloc: the prefill entry point for callers that cannot allocate.

Callers such as a plugin inside a runtime that owns the device allocator, or a
serving loop that forbids device allocations after start-up, cannot pass
gdr_chunk_fwd a workspace; gdr_chunk_fwd_noalloc uses a fixed scratch array
inside the library instead. These tests call it through the C ABI and check it
against gdr_chunk_fwd (with a torch-allocated workspace) and against the float64
oracle, each case twice in a row: the second call finds the first call's
contents in the shared array and must still be right. The cases cover the
schedules that keep per-call state in the array: the fused one over packed
sequences (a claim counter, the claim order and per-unit ready flags), the
phased one (forced, packed sequences), the fused one over equal lengths
(per-unit ready flags) and the segmented one (few long chains: segment state
sets). The device status word
is read back through gdr_noalloc_read_device_status. The file is collected
last, so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from gated_delta_rule_03_gb300 import chunk_fwd_workspace_size, inputs, ops
from tests.helpers import TOL, chunk_fwd, f64, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20  # GDR_NOALLOC_SCRATCH_BYTES in include/gdr.h
GDR_ERR_BAD_SEQLENS = -7


def noalloc_fn():
    fn = ops._load().gdr_chunk_fwd_noalloc
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, ci, ci, ci, ci, ci, vp, vp, vp]
    fn.restype = ci
    return fn


def read_status(stream):
    fn = ops._load().gdr_noalloc_read_device_status
    fn.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    out = ctypes.c_int(12345)
    st = fn(ctypes.byref(out), ctypes.c_void_p(stream.cuda_stream))
    assert st == 0, ops.status_string(st)
    return out.value


def ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def run_noalloc(fn, dev, q, k, v, la, b, S0, cu, num_seqs, inp):
    o = torch.full((inp.total_tokens, inp.H, inp.dv), float("nan"), dtype=q.dtype, device=dev)
    S = torch.full((num_seqs, inp.H, inp.dk, inp.dv), float("nan"), device=dev)
    stream = torch.cuda.current_stream(dev)
    st = fn(ptr(q), ptr(k), ptr(v), ptr(la), ptr(b), ptr(S0), ptr(cu), num_seqs,
            inp.total_tokens, inp.H, inp.dk, inp.dv, inp.chunk,
            0 if inp.dtype == "f32" else 1, ptr(o), ptr(S), ctypes.c_void_p(stream.cuda_stream))
    assert st == 0, ops.status_string(st)
    assert read_status(stream) == 0
    return f64(o), f64(S)


CASES = {
    # packed sequences: the fused schedule with the solve claiming units (bf16), the
    # phased schedule (bf16, forced below) and the exact path (fp32)
    "packed_bf16": lambda: inputs.prefill_inputs([150, 4000], H=2, dk=128, dv=128, dtype="bf16",
                                                 seed=31, s0_std=0.2, gate="slow"),
    "packed_bf16_phased": lambda: inputs.prefill_inputs([150, 77], H=2, dk=128, dv=128,
                                                        dtype="bf16", seed=35, s0_std=0.2,
                                                        gate="slow"),
    "packed_f32": lambda: inputs.prefill_inputs([64, 3, 200], H=3, dk=64, dv=96, dtype="f32",
                                                seed=32, s0_std=0.5, gate="slow"),
    # equal lengths, no cu_seqlens: the fused cooperative schedule
    "fused_bf16": lambda: inputs.prefill_inputs([512, 512], H=4, dk=128, dv=128, dtype="bf16",
                                                seed=33, s0_std=0.2, gate="slow"),
    # one long sequence, segmented into 4 (forced below)
    "segmented_bf16": lambda: inputs.prefill_inputs([4096], H=2, dk=128, dv=128, dtype="bf16",
                                                    seed=34, s0_std=0.2, gate="slow"),
}


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_chunk_fwd_and_the_oracle_on_two_calls_in_a_row(case, monkeypatch):
    if case == "segmented_bf16":
        monkeypatch.setenv("GDR_PREFILL_SEGMENTS", "4")
    if case == "packed_bf16_phased":
        monkeypatch.setenv("GDR_PREFILL_PHASES", "2")
    dev = torch.device("cuda", 0)
    fn = noalloc_fn()
    inp = CASES[case]()
    n = inp.num_seqs
    varlen = inp.cu_seqlens is not None
    assert chunk_fwd_workspace_size(n, inp.total_tokens, inp.H, inp.dk, inp.dv, 64,
                                    torch.float32 if inp.dtype == "f32" else torch.bfloat16) \
        <= SCRATCH_BYTES
    if inp.dtype == "bf16":
        sched = ops.chunk_fwd_schedule(n, inp.total_tokens, inp.H, inp.dk, inp.dv,
                                       torch.bfloat16, varlen=varlen)
        if case in ("fused_bf16", "packed_bf16"):
            assert sched == 0
        elif case == "packed_bf16_phased":
            assert sched == 2
        elif case == "segmented_bf16":
            assert sched == ops.SCHEDULE_SEGMENTED + 4
    d = lambda t: None if t is None else t.to(dev)
    q, k, v, la, b = d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta)
    S0, cu = d(inp.S0), d(inp.cu_seqlens)
    ref_o, ref_S = chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=n)
    ref_o, ref_S = f64(ref_o), f64(ref_S)
    orc_o, orc_S = oracle_prefill(inp)
    tol = TOL[inp.dtype]
    for call in range(2):
        o, S = run_noalloc(fn, dev, q, k, v, la, b, S0, cu, n, inp)
        assert rel_err(o, ref_o) <= tol, (case, call)
        assert rel_err(S, ref_S) <= tol, (case, call)
        assert rel_err(o, orc_o) <= tol, (case, call)
        assert rel_err(S, orc_S) <= tol, (case, call)


def test_noalloc_reports_a_rejected_cu_seqlens_through_its_status_word():
    dev = torch.device("cuda", 0)
    fn = noalloc_fn()
    inp = CASES["packed_bf16"]()
    d = lambda t: t.to(dev)
    q, k, v, la, b, S0 = d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), d(inp.S0)
    stream = torch.cuda.current_stream(dev)
    bad = torch.tensor([0, 200, 150, inp.total_tokens], dtype=torch.int32, device=dev)  # decreasing
    o = torch.full((inp.total_tokens, inp.H, inp.dv), float("nan"), dtype=q.dtype, device=dev)
    S = torch.full((3, inp.H, inp.dk, inp.dv), float("nan"), device=dev)
    S0_3 = torch.zeros((3, inp.H, inp.dk, inp.dv), device=dev)
    st = fn(ptr(q), ptr(k), ptr(v), ptr(la), ptr(b), ptr(S0_3), ptr(bad), 3, inp.total_tokens,
            inp.H, inp.dk, inp.dv, 64, 1, ptr(o), ptr(S), ctypes.c_void_p(stream.cuda_stream))
    assert st == 0, ops.status_string(st)  # the check is on the device
    assert read_status(stream) == GDR_ERR_BAD_SEQLENS
    assert bool(torch.isnan(o).all()) and bool(torch.isnan(S).all())  # nothing was written
    # the next good call clears it
    o2, S2 = run_noalloc(fn, dev, q, k, v, la, b, S0, d(inp.cu_seqlens), inp.num_seqs, inp)
    orc_o, orc_S = oracle_prefill(inp)
    assert rel_err(o2, orc_o) <= TOL["bf16"] and rel_err(S2, orc_S) <= TOL["bf16"]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fn = noalloc_fn()
    # far more chunks than 32 MiB of scratch can hold on the exact path
    T, H = 1 << 20, 16
    assert chunk_fwd_workspace_size(1, T, H, 128, 128, 64, torch.float32) > SCRATCH_BYTES
    # null data pointers: were the size check missing, the call would still be rejected
    # by argument validation and never launch anything
    st = fn(None, None, None, None, None, None, None, 1, T, H, 128, 128, 64, 0, None, None, None)
    assert st == -4, ops.status_string(st)


def test_noalloc_status_reader_rejects_a_null_pointer():
    fn = ops._load().gdr_noalloc_read_device_status
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    assert fn(None, None) == -1
