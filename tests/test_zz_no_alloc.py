"""gdr_chunk_fwd_noalloc: the prefill entry point for callers that cannot allocate.

Callers such as a plugin inside a runtime that owns the device allocator, or a
serving loop that forbids device allocations after start-up, cannot pass
gdr_chunk_fwd a workspace; gdr_chunk_fwd_noalloc uses a fixed scratch array
inside the library instead. This test calls it through the C ABI and checks it
against gdr_chunk_fwd (with a torch-allocated workspace) on two calls in a row:
the second call finds the first call's contents in the shared array and must
still be right. It lives in a file of its own that pytest collects last.
"""
import ctypes

import pytest
import torch

from gated_delta_rule_03_gb300 import chunk_fwd, chunk_fwd_workspace_size, inputs, ops
from tests.helpers import TOL, f64, rel_err

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20  # GDR_NOALLOC_SCRATCH_BYTES in include/gdr.h


def noalloc_fn():
    fn = ops._load().gdr_chunk_fwd_noalloc
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, ci, ci, ci, ci, ci, vp, vp, vp]
    fn.restype = ci
    return fn


def ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(fn, inp, dev):
    d = lambda t: None if t is None else t.to(dev)
    q, k, v, la, b = d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta)
    S0, cu = d(inp.S0), d(inp.cu_seqlens)
    o = torch.full((inp.total_tokens, inp.H, inp.dv), float("nan"), dtype=q.dtype, device=dev)
    S = torch.full((inp.num_seqs, inp.H, inp.dk, inp.dv), float("nan"), device=dev)
    stream = torch.cuda.current_stream(dev)
    st = fn(ptr(q), ptr(k), ptr(v), ptr(la), ptr(b), ptr(S0), ptr(cu), inp.num_seqs,
            inp.total_tokens, inp.H, inp.dk, inp.dv, inp.chunk,
            0 if inp.dtype == "f32" else 1, ptr(o), ptr(S), ctypes.c_void_p(stream.cuda_stream))
    assert st == 0, ops.status_string(st)
    ref_o, ref_S = chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=inp.num_seqs)
    torch.cuda.synchronize(dev)
    return (f64(o), f64(S)), (f64(ref_o), f64(ref_S))


def test_noalloc_matches_chunk_fwd_on_two_calls_in_a_row():
    dev = torch.device("cuda", 0)
    fn = noalloc_fn()
    cases = [
        inputs.prefill_inputs([150, 77], H=2, dk=128, dv=128, dtype="bf16", seed=31,
                              s0_std=0.2, gate="slow"),
        inputs.prefill_inputs([64, 3, 200], H=3, dk=64, dv=96, dtype="f32", seed=32,
                              s0_std=0.5, gate="slow"),
    ]
    for inp in cases:
        (o, S), (ref_o, ref_S) = call_noalloc(fn, inp, dev)
        tol = TOL[inp.dtype]
        assert rel_err(o, ref_o) <= tol
        assert rel_err(S, ref_S) <= tol


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fn = noalloc_fn()
    # far more chunks than 32 MiB of scratch can hold on the exact path
    T, H = 1 << 20, 16
    assert chunk_fwd_workspace_size(1, T, H, 128, 128, 64, torch.float32) > SCRATCH_BYTES
    # null data pointers: were the size check missing, the call would still be rejected
    # by argument validation and never launch anything
    st = fn(None, None, None, None, None, None, None, 1, T, H, 128, 128, 64, 0, None, None, None)
    assert st == -4, ops.status_string(st)
