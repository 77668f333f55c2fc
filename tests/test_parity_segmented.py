"""GPU parity of the segmented schedule of the tensor-core prefill against the oracle.

For a few long chains (sequences x heads x 128-column value slices) the call cuts each
sequence into n segments. The state after a run of chunks is affine in the state before
it (S_end = P S + R): a first chain kernel summarises every segment but the last (P from
the identity with zero values, R from zero), a scan chains the segments' start states in
fp32, and a second chain kernel runs every segment from its start state with output.
The result differs from the other schedules only by rounding. Tolerances as for every
prefill: max |gpu - oracle| / max |oracle| <= 2e-2 for bf16 inputs, per output tensor.
The "none" gate (alpha = 1) and "slow" gate carry the state across the whole sequence,
so a wrong start state shows.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_03_gb300 import inputs, ops
from tests.helpers import TOL, chunk_fwd, f64, gpu_prefill, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu

SEG = ops.SCHEDULE_SEGMENTED


@functools.lru_cache(maxsize=None)
def case(lens, H, dv, gate, seed):
    inp = inputs.prefill_inputs(list(lens), H=H, dk=128, dv=dv, dtype="bf16", seed=seed,
                                s0_std=0.5, gate=gate)
    return inp, oracle_prefill(inp)


def schedule_of(inp):
    return ops.chunk_fwd_schedule(inp.num_seqs, inp.total_tokens, inp.H, 128, inp.dv,
                                  torch.bfloat16, varlen=inp.cu_seqlens is not None)


def assert_close(o, S, ref, per_sequence_of=None):
    o_ref, S_ref = ref
    o_g, S_g = f64(o), f64(S)
    assert np.isfinite(o_g).all() and np.isfinite(S_g).all()
    eo, es = rel_err(o_g, o_ref), rel_err(S_g, S_ref)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (eo, es)
    if per_sequence_of is not None and per_sequence_of.cu_seqlens is not None:
        cu = per_sequence_of.cu_seqlens.numpy()
        for n in range(per_sequence_of.num_seqs):
            if cu[n + 1] > cu[n]:
                assert rel_err(o_g[cu[n]:cu[n + 1]], o_ref[cu[n]:cu[n + 1]]) <= TOL["bf16"], n
            assert rel_err(S_g[n], S_ref[n]) <= TOL["bf16"], n


def test_long_context_workload_takes_the_segmented_schedule(monkeypatch):
    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    monkeypatch.delenv("GDR_PREFILL_SEGMENTS", raising=False)
    w = inputs.WORKLOADS["long_bf16"]
    N, T = w["num_seqs"], w["num_seqs"] * w["seq_len"]
    sched = ops.chunk_fwd_schedule(N, T, w["H"], w["dk"], w["dv"], torch.bfloat16)
    assert SEG + 3 <= sched <= SEG + 8
    assert ops.chunk_fwd_kernel_launches(N, T, w["H"], w["dk"], w["dv"], torch.bfloat16) == 5
    # many chains keep the other schedules
    assert ops.chunk_fwd_schedule(4, 4 * 4096, 16, 128, 128, torch.bfloat16) < SEG


@pytest.mark.parametrize("gate", ["none", "slow", "default"])
@pytest.mark.parametrize("dv", [128, 256])
@pytest.mark.parametrize("segs", [2, 3, 8, None])
def test_one_long_sequence(segs, dv, gate, monkeypatch):
    # one ragged sequence of 128 chunks and a 37-token tail, nonzero S0
    inp, ref = case((8229,), 2, dv, gate, 300 + dv)
    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    if segs is None:
        monkeypatch.delenv("GDR_PREFILL_SEGMENTS", raising=False)
    else:
        monkeypatch.setenv("GDR_PREFILL_SEGMENTS", str(segs))
    sched = schedule_of(inp)
    assert sched > SEG and (segs is None or sched == SEG + segs)
    o, S = gpu_prefill(inp)
    assert_close(o, S, ref)


@pytest.mark.parametrize("segs", [3, 5, 8])
def test_packed_sequences_with_empty_and_short_ones(segs, monkeypatch):
    # sequences shorter than the segment count leave segments empty (their transition is
    # the identity, their summary zero); one sequence is empty
    inp, ref = case((9000, 64, 1, 0, 12000), 1, 256, "slow", 310)
    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    monkeypatch.setenv("GDR_PREFILL_SEGMENTS", str(segs))
    assert schedule_of(inp) == SEG + segs
    o, S = gpu_prefill(inp)
    assert_close(o, S, ref, per_sequence_of=inp)


def test_segmented_close_to_phased(monkeypatch):
    # the two schedules round differently but agree to well inside the tolerance
    inp, ref = case((8229,), 2, 256, "none", 556)
    monkeypatch.setenv("GDR_PREFILL_SEGMENTS", "6")
    o_s, S_s = gpu_prefill(inp)
    monkeypatch.delenv("GDR_PREFILL_SEGMENTS")
    monkeypatch.setenv("GDR_PREFILL_PHASES", "1")
    o_p, S_p = gpu_prefill(inp)
    assert rel_err(f64(o_s), f64(o_p)) <= TOL["bf16"] / 2
    assert rel_err(f64(S_s), f64(S_p)) <= TOL["bf16"] / 2


def test_in_place_state(monkeypatch):
    # S_final may be S0: the first segment starts from the scan's copy of S0
    inp, ref = case((8229,), 2, 128, "none", 128)
    monkeypatch.setenv("GDR_PREFILL_SEGMENTS", "8")
    S = inp.S0.cuda()
    o, S_out = chunk_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.log_alpha.cuda(),
                         inp.beta.cuda(), S0=S, S_final=S)
    torch.cuda.synchronize()
    assert S_out.data_ptr() == S.data_ptr()
    assert_close(o, S, ref)


def test_graph_capture_and_repeated_calls(monkeypatch):
    # one stream, no side resources: the call captures into a graph, and calls on one
    # workspace give identical bits
    inp, _ = case((8229,), 2, 128, "slow", 128)
    monkeypatch.setenv("GDR_PREFILL_SEGMENTS", "4")
    dev = lambda t: t.cuda()
    q, k, v, la, b, S0 = map(dev, (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0))
    ws = torch.empty(ops.chunk_fwd_workspace_size(1, inp.total_tokens, 2, 128, 128),
                     dtype=torch.uint8, device="cuda")
    o_e, S_e = chunk_fwd(q, k, v, la, b, S0=S0, workspace=ws)
    o_e2, S_e2 = chunk_fwd(q, k, v, la, b, S0=S0, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o_e, o_e2) and torch.equal(S_e, S_e2)
    o, S = torch.empty_like(o_e), torch.empty_like(S_e)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chunk_fwd(q, k, v, la, b, S0=S0, o=o, S_final=S, workspace=ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_e) and torch.equal(S, S_e)
    assert ops.read_device_status(ws) == 0


@pytest.mark.parametrize("dv", [128, 256])
def test_additive_rule(dv, monkeypatch):
    # the additive rule's transition is gamma_C I: P_f is a decayed identity
    inp, _ = case((8229,), 2, dv, "slow", 560 + dv)
    monkeypatch.setenv("GDR_PREFILL_SEGMENTS", "5")
    d = lambda t: None if t is None else t.cuda()
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), S0=d(inp.S0),
                     rule="additive")
    torch.cuda.synchronize()
    ref = oracle.forward(f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.log_alpha),
                         f64(inp.beta), S0=f64(inp.S0), num_seqs=1, additive=True)
    assert_close(o, S, ref)


@pytest.mark.parametrize("dv", [128, 256])
def test_output_step(dv, monkeypatch):
    # the output step: fused into the second chain's epilogue (d_v = 128), else its own
    # kernel after the chains; the summary chain writes no output
    inp, (o_ref, S_ref) = case((8229,), 2, dv, "slow", 300 + dv)
    monkeypatch.setenv("GDR_PREFILL_SEGMENTS", "7")
    rng = np.random.default_rng(570 + dv)
    z = torch.from_numpy((2.0 * rng.standard_normal((inp.total_tokens, 2, dv))).astype(
        np.float32)).to(torch.bfloat16)
    w = torch.from_numpy(rng.uniform(0.5, 1.5, dv).astype(np.float32))
    d = lambda t: None if t is None else t.cuda()
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), S0=d(inp.S0),
                     out_gate=d(z), out_norm_weight=d(w), out_norm_eps=1e-5)
    torch.cuda.synchronize()
    assert_close(o, S, (oracle.out_norm_gate(o_ref, f64(z), f64(w), eps=1e-5), S_ref))


def test_layer_prologue(monkeypatch):
    # raw q, k and gate pre-activations: the summaries use the same unit-length keys
    rng = np.random.default_rng(580)
    T, H, dv = 8229, 2, 256
    st = lambda x: torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    q, k = st(rng.standard_normal((T, H, 128))), st(rng.standard_normal((T, H, 128)))
    v = st(rng.standard_normal((T, H, dv)))
    a = torch.from_numpy((rng.standard_normal((T, H)) - 4.0).astype(np.float32))
    b = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32))
    A = torch.from_numpy(rng.uniform(0.2, 2.0, H).astype(np.float32))
    S0 = torch.from_numpy((0.3 * rng.standard_normal((1, H, 128, dv))).astype(np.float32))
    monkeypatch.setenv("GDR_PREFILL_SEGMENTS", "8")
    c = lambda t: t.cuda()
    o, S = chunk_fwd(c(q), c(k), c(v), c(a), c(b), S0=c(S0), prologue=True, gate_A=c(A))
    torch.cuda.synchronize()
    qn, kn, la, beta = oracle.layer_prologue(f64(q), f64(k), f64(a), f64(b), f64(A))
    assert_close(o, S, oracle.forward(qn, kn, f64(v), la, beta, S0=f64(S0), num_seqs=1))
