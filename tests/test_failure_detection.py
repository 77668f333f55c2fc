"""The tensor-core chain's bounded device waits give up cleanly.

Every wait in the chain kernel is bounded. A role that gives up marks the call
GDR_ERR_DEVICE_TIMEOUT in the status word, the other roles give up in turn, the
loads already issued land, issued MMAs complete, TMEM is freed and the kernel
returns: nothing faults, traps or hangs, and the context stays usable. The
failure is made on purpose by the library's test knob GDR_DEBUG_CHAIN_FAULT=<chunk>:
the producer of one chain CTA skips that chunk's K-slot load (a barrier phase
that nothing completes), and every wait's bound drops to about 10 ms. The test
checks that the call returns, that the status word reads the timeout, and that
the next ordinary call on the same workspace matches the float64 oracle.
"""
import time

import pytest
import torch

from gated_delta_rule_03_gb300 import inputs, ops
from tests.helpers import TOL, chunk_fwd, f64, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu

GDR_ERR_DEVICE_TIMEOUT = -6


@pytest.mark.parametrize("schedule", ["phased", "fused", "fused_packed"])
@pytest.mark.parametrize("fault_chunk", [0, 2, 7])
def test_chain_gives_up_on_a_missing_load_then_the_next_call_is_clean(schedule, fault_chunk,
                                                                     monkeypatch):
    # (fused_packed: packed sequences, the solve claiming units and the chain CTAs of the
    # shorter sequence solving before their chains start)
    if schedule == "phased":
        monkeypatch.setenv("GDR_PREFILL_PHASES", "1")
    lens = [4000, 300] if schedule == "fused_packed" else [512, 512]
    inp = inputs.prefill_inputs(lens, H=2, dk=128, dv=128, dtype="bf16", seed=41,
                                s0_std=0.2, gate="slow")
    n, T = inp.num_seqs, inp.total_tokens
    varlen = inp.cu_seqlens is not None
    assert varlen == (schedule == "fused_packed")
    assert ops.chunk_fwd_schedule(n, T, inp.H, 128, 128, torch.bfloat16, varlen=varlen) == \
        (1 if schedule == "phased" else 0)
    dev = torch.device("cuda", 0)
    d = lambda t: None if t is None else t.to(dev)
    q, k, v, la, b, S0 = d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), d(inp.S0)
    cu = d(inp.cu_seqlens)
    ws = torch.empty(ops.chunk_fwd_workspace_size(n, T, inp.H, 128, 128), dtype=torch.uint8,
                     device=dev)

    monkeypatch.setenv("GDR_DEBUG_CHAIN_FAULT", str(fault_chunk))
    t0 = time.perf_counter()
    ops.chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=n, workspace=ws)
    status = ops.read_device_status(ws)  # synchronises
    elapsed = time.perf_counter() - t0
    assert status == GDR_ERR_DEVICE_TIMEOUT, ops.status_string(status)
    assert elapsed < 10.0

    monkeypatch.delenv("GDR_DEBUG_CHAIN_FAULT")
    o, S = chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=n, workspace=ws)
    assert ops.read_device_status(ws) == 0
    ref_o, ref_S = oracle_prefill(inp)
    assert rel_err(f64(o), ref_o) <= TOL["bf16"]
    assert rel_err(f64(S), ref_S) <= TOL["bf16"]


@pytest.mark.parametrize("fault_chunk", [0, 3])
def test_per_channel_chain_gives_up_on_a_missing_load_then_the_next_call_is_clean(fault_chunk,
                                                                                 monkeypatch):
    # the per-channel tensor-core path: its chain takes the same knob, so that its
    # producer skips one K-slot load (e^{g_C - g} . K, A^T, exp(g_C))
    inp = inputs.prefill_inputs([300, 200], H=2, dk=128, dv=128, dtype="bf16", seed=42,
                                s0_std=0.2, gate="slow", decay="channel")
    assert ops.chunk_fwd_path(128, 128, torch.bfloat16, "channel") == ops.PATH_CHANNEL_TENSOR
    n, T = inp.num_seqs, inp.total_tokens
    dev = torch.device("cuda", 0)
    d = lambda t: None if t is None else t.to(dev)
    q, k, v, la, b, S0 = d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), d(inp.S0)
    cu = d(inp.cu_seqlens)
    ws = torch.empty(ops.chunk_fwd_workspace_size(n, T, inp.H, 128, 128, decay="channel"),
                     dtype=torch.uint8, device=dev)

    monkeypatch.setenv("GDR_DEBUG_CHAIN_FAULT", str(fault_chunk))
    t0 = time.perf_counter()
    ops.chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=n, workspace=ws)
    status = ops.read_device_status(ws)  # synchronises
    elapsed = time.perf_counter() - t0
    assert status == GDR_ERR_DEVICE_TIMEOUT, ops.status_string(status)
    assert elapsed < 10.0

    monkeypatch.delenv("GDR_DEBUG_CHAIN_FAULT")
    o, S = chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=n, workspace=ws)
    assert ops.read_device_status(ws) == 0
    ref_o, ref_S = oracle_prefill(inp)
    assert rel_err(f64(o), ref_o) <= TOL["bf16"]
    assert rel_err(f64(S), ref_S) <= TOL["bf16"]


@pytest.mark.parametrize("fault_chunk,lens,H", [(0, [300, 200], 2), (6, [300, 200], 2),
                                                (70, [4096, 4096], 16)])
def test_per_channel_operands_kernel_gives_up_then_the_next_call_is_clean(fault_chunk, lens, H,
                                                                         monkeypatch):
    # GDR_DEBUG_PREP_FAULT=<chunk>: head 0's unit of that chunk in the kernel that builds the
    # per-channel operands gets no key and query loads; its wait runs out, its CTA marks
    # the status word and drains, and the chain after it writes nothing. With 2,048 units
    # (more than the kernel's resident CTAs) the dropped unit, 70 * 16 = 1,120, is its
    # CTA's second: the copies were to be issued while the first unit's outputs were stored.
    inp = inputs.prefill_inputs(lens, H=H, dk=128, dv=128, dtype="bf16", seed=43,
                                s0_std=0.2, gate="slow", decay="channel")
    n, T = inp.num_seqs, inp.total_tokens
    dev = torch.device("cuda", 0)
    d = lambda t: None if t is None else t.to(dev)
    q, k, v, la, b, S0 = d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), d(inp.S0)
    cu = d(inp.cu_seqlens)
    ws = torch.empty(ops.chunk_fwd_workspace_size(n, T, inp.H, 128, 128, decay="channel"),
                     dtype=torch.uint8, device=dev)
    o = torch.full((T, inp.H, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    S = torch.full((n, inp.H, 128, 128), float("nan"), device=dev)
    if H == 16:  # the dropped unit is the second of its CTA on a 152-SM device
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        assert fault_chunk * H >= 4 * sms

    monkeypatch.setenv("GDR_DEBUG_PREP_FAULT", str(fault_chunk))
    t0 = time.perf_counter()
    ops.chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=n, o=o, S_final=S, workspace=ws)
    status = ops.read_device_status(ws)  # synchronises
    elapsed = time.perf_counter() - t0
    assert status == GDR_ERR_DEVICE_TIMEOUT, ops.status_string(status)
    assert elapsed < 10.0
    assert bool(torch.isnan(o).all()) and bool(torch.isnan(S).all())  # the chain wrote nothing

    monkeypatch.delenv("GDR_DEBUG_PREP_FAULT")
    o, S = chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=n, workspace=ws)
    assert ops.read_device_status(ws) == 0
    ref_o, ref_S = oracle_prefill(inp)
    assert rel_err(f64(o), ref_o) <= TOL["bf16"]
    assert rel_err(f64(S), ref_S) <= TOL["bf16"]
