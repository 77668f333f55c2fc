"""GPU parity of the fused schedule over packed sequences, where the solve claims its units.

Packed sequences (cu_seqlens) whose chains leave at least 16 SMs free run as one
cooperative launch: every chain CTA, plus solve CTAs that claim (chunk, head) units from a
counter in an order the planning kernel lists, so that each sequence's chunks are solved
by the time its chain reaches them. A chain CTA whose sequence is shorter than the longest
first solves units too and starts its chain when the claims reach the trigger the plan gives
it, so that all chains end about together. After it the host launches the phased
schedule's solve and chain kernels (one phase): when the lengths leave little of the solve
to overlap the chains, the plan hands the call to that pair instead and the fused kernel
returns at once (the plan's choice is read back from the workspace's control word 33).
Each case is compared with the float64 oracle (max |gpu - oracle| / max |oracle| <= 2e-2
for bf16 inputs) and, bit for bit, with the phased two-kernel schedule
(GDR_PREFILL_PHASES=1), which solves the same units with the same arithmetic in separate
launches. The cases cover the workload's mix of lengths, equal and nearly equal lengths
packed (handed to the pair), empty and single-token sequences, many short sequences, the
most sequences the schedule takes, two 128-column value slices, and the options that
change what the solve and chain compute.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_03_gb300 import inputs, ops
from tests.helpers import TOL, chunk_fwd, f64, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu


def lens_of(seed, n, lo, hi):
    return [int(x) for x in np.random.default_rng(seed).integers(lo, hi + 1, size=n)]


# pair: whether the plan is expected to hand the call to the two-kernel pair
CASES = {
    "workload_lengths": dict(lens=[6945, 2521, 1351, 2804, 3690, 6766, 3978, 1218], H=16, dv=128,
                             pair=False),
    "equal_lengths_packed": dict(lens=[2048] * 8, H=16, dv=128, pair=True),
    "nearly_equal_lengths": dict(lens=[2048, 2100, 2060, 2010, 2090, 2048, 2070, 2035], H=16,
                                 dv=128, pair=True),
    "empty_and_short": dict(lens=[0, 300, 1, 0, 64, 65, 14000], H=3, dv=128, pair=False),
    "many_sequences": dict(lens=lens_of(1, 40, 1, 4096) + [40000], H=2, dv=128, pair=False),
    "most_sequences": dict(lens=lens_of(2, 127, 0, 300) + [250000], H=1, dv=128, pair=False),
    "two_value_slices": dict(lens=[900, 130, 6000], H=4, dv=256, pair=False),
}
# (the schedule takes packed sequences of 32 chunks or more on average)
PAIR_WORD = 33  # int32 control word of the workspace: 1 when the pair ran the call


def call(inp, ws=None, **kw):
    # poisoned, guard-banded outputs (tests.helpers.chunk_fwd)
    d = lambda t: None if t is None else t.cuda()
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), S0=d(inp.S0),
                     cu_seqlens=d(inp.cu_seqlens), num_seqs=inp.num_seqs, workspace=ws, **kw)
    torch.cuda.synchronize()
    return o, S


def pair_chosen(ws):
    return int(ws[4 * PAIR_WORD:4 * PAIR_WORD + 4].view(torch.int32).item())


def run_both(inp, monkeypatch, pair=False, **kw):
    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    monkeypatch.delenv("GDR_PREFILL_SEGMENTS", raising=False)
    assert ops.chunk_fwd_schedule(inp.num_seqs, inp.total_tokens, inp.H, 128, inp.dv,
                                  torch.bfloat16, varlen=True) == 0
    assert ops.chunk_fwd_kernel_launches(inp.num_seqs, inp.total_tokens, inp.H, 128, inp.dv,
                                         torch.bfloat16, varlen=True) == 4
    ws = torch.empty(ops.chunk_fwd_workspace_size(inp.num_seqs, inp.total_tokens, inp.H, 128,
                                                  inp.dv, prologue=bool(kw.get("prologue"))),
                     dtype=torch.uint8, device="cuda")
    o_c, S_c = call(inp, ws=ws, **kw)
    assert pair_chosen(ws) == int(pair)
    monkeypatch.setenv("GDR_PREFILL_PHASES", "1")
    o_p, S_p = call(inp, **kw)
    monkeypatch.delenv("GDR_PREFILL_PHASES")
    return o_c, S_c, o_p, S_p


@pytest.mark.parametrize("case", list(CASES))
def test_claimed_solve_matches_the_oracle_and_the_phased_schedule(case, monkeypatch):
    c = CASES[case]
    inp = inputs.prefill_inputs(c["lens"], H=c["H"], dk=128, dv=c["dv"], dtype="bf16",
                                seed=100 + len(case), s0_std=0.3, gate="slow", packed=True)
    o_c, S_c, o_p, S_p = run_both(inp, monkeypatch, pair=c["pair"])
    assert torch.equal(o_c, o_p) and torch.equal(S_c, S_p)
    heads = None if inp.H <= 4 else [0, inp.H - 1]
    o_ref, S_ref = oracle_prefill(inp, heads)
    o_g, S_g = f64(o_c), f64(S_c)
    if heads is not None:
        o_g, S_g = o_g[:, heads], S_g[:, heads]
    assert np.isfinite(o_g).all() and np.isfinite(S_g).all()
    assert rel_err(o_g, o_ref) <= TOL["bf16"], rel_err(o_g, o_ref)
    assert rel_err(S_g, S_ref) <= TOL["bf16"], rel_err(S_g, S_ref)
    cu = inp.cu_seqlens.numpy()
    for n in range(inp.num_seqs):  # sequence by sequence: each chain's own result
        if cu[n + 1] > cu[n]:
            assert rel_err(o_g[cu[n]:cu[n + 1]], o_ref[cu[n]:cu[n + 1]]) <= TOL["bf16"], n
        else:  # an empty sequence keeps its initial state
            S0_n = f64(inp.S0)[n]
            np.testing.assert_array_equal(S_g[n], S0_n if heads is None else S0_n[heads])
        assert rel_err(S_g[n], S_ref[n]) <= TOL["bf16"], n


@pytest.mark.parametrize("option", ["additive", "prologue", "out_step"])
def test_claimed_solve_with_options(option, monkeypatch):
    rng = np.random.default_rng(7)
    inp = inputs.prefill_inputs([700, 0, 1500, 64, 8000], H=3, dk=128, dv=128, dtype="bf16",
                                seed=200, s0_std=0.3, gate="slow", packed=True)
    kw, z, w, A = {}, None, None, None
    if option == "additive":
        kw = dict(rule="additive")
    elif option == "prologue":
        # raw projections and gate pre-activations: the kernels apply the prologue
        T = inp.total_tokens
        q = torch.from_numpy((2.0 * rng.standard_normal((T, 3, 128))).astype(np.float32))
        k = torch.from_numpy((2.0 * rng.standard_normal((T, 3, 128))).astype(np.float32))
        inp.q, inp.k = q.to(torch.bfloat16), k.to(torch.bfloat16)
        inp.log_alpha = torch.from_numpy((rng.standard_normal((T, 3)) - 3.0).astype(np.float32))
        inp.beta = torch.from_numpy(rng.standard_normal((T, 3)).astype(np.float32))
        A = torch.from_numpy(rng.uniform(0.2, 2.0, 3).astype(np.float32))
        kw = dict(prologue=True, gate_A=A.cuda())
    else:
        z = torch.from_numpy((2.0 * rng.standard_normal((inp.total_tokens, 3, 128))).astype(
            np.float32)).to(torch.bfloat16)
        w = torch.from_numpy(rng.uniform(0.5, 1.5, 128).astype(np.float32))
        kw = dict(out_gate=z.cuda(), out_norm_weight=w.cuda(), out_norm_eps=1e-5)
    o_c, S_c, o_p, S_p = run_both(inp, monkeypatch, **kw)
    assert torch.equal(o_c, o_p) and torch.equal(S_c, S_p)
    import oracle
    qo, ko, lao, bo = f64(inp.q), f64(inp.k), f64(inp.log_alpha), f64(inp.beta)
    if option == "prologue":
        qo, ko, lao, bo = oracle.layer_prologue(qo, ko, lao, bo, f64(A))
    o_ref, S_ref = oracle.forward(qo, ko, f64(inp.v), lao, bo, S0=f64(inp.S0),
                                  cu_seqlens=inp.cu_seqlens.numpy().astype(np.int64),
                                  additive=option == "additive")
    if option == "out_step":
        o_ref = oracle.out_norm_gate(o_ref, f64(z), f64(w), eps=1e-5)
    assert rel_err(f64(o_c), o_ref) <= TOL["bf16"]
    assert rel_err(f64(S_c), S_ref) <= TOL["bf16"]


def test_claimed_solve_repeated_calls_share_a_workspace():
    # every call's plan resets the claim counter and the unit flags: back-to-back calls on
    # one workspace and stream give identical results
    inp = inputs.prefill_inputs([900, 77, 6000], H=4, dk=128, dv=128, dtype="bf16", seed=301,
                                s0_std=0.2, gate="slow")
    d = lambda t: t.cuda()
    q, k, v, la, b, S0, cu = map(d, (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0,
                                     inp.cu_seqlens))
    ws = torch.empty(ops.chunk_fwd_workspace_size(3, inp.total_tokens, 4, 128, 128),
                     dtype=torch.uint8, device="cuda")
    outs = [ops.chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, workspace=ws) for _ in range(4)]
    torch.cuda.synchronize()
    for o, S in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(S, outs[0][1])
    assert ops.read_device_status(ws) == 0


def test_bad_cu_seqlens_under_the_claimed_solve():
    # a rejected cu_seqlens: the plan reports it, no CTA solves or chains, the call returns
    inp = inputs.prefill_inputs([100, 4000], H=2, dk=128, dv=128, dtype="bf16", seed=9)
    args = [t.cuda() for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    assert ops.chunk_fwd_schedule(2, 4100, 2, 128, 128, torch.bfloat16, varlen=True) == 0
    bad = torch.tensor([0, 120, 4090], dtype=torch.int32, device="cuda")
    ops.chunk_fwd(*args, cu_seqlens=bad, workspace=ws)
    assert ops.read_device_status(ws) == -7
    good = inp.cu_seqlens.cuda()
    o, S = ops.chunk_fwd(*args, cu_seqlens=good, workspace=ws)
    assert ops.read_device_status(ws) == 0
    o_ref, S_ref = oracle_prefill(inp)
    assert rel_err(f64(o), o_ref) <= TOL["bf16"] and rel_err(f64(S), S_ref) <= TOL["bf16"]


@pytest.mark.parametrize("packed", [False, True])
def test_fused_schedules_inside_graph_capture(packed, monkeypatch):
    # both forms of the fused schedule are stream-ordered launches on the caller's stream
    # (the equal-length one a single cooperative kernel that plans itself): a captured call
    # replays to the eager bits, twice in a row on one workspace
    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    lens = [900, 77, 6000] if packed else [2048, 2048]
    inp = inputs.prefill_inputs(lens, H=4, dk=128, dv=128, dtype="bf16", seed=410 + packed,
                                s0_std=0.2, gate="slow")
    assert (inp.cu_seqlens is not None) == packed
    n, T = inp.num_seqs, inp.total_tokens
    assert ops.chunk_fwd_schedule(n, T, 4, 128, 128, torch.bfloat16, varlen=packed) == 0
    d = lambda t: None if t is None else t.cuda()
    q, k, v, la, b, S0, cu = map(d, (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0,
                                     inp.cu_seqlens))
    ws = torch.empty(ops.chunk_fwd_workspace_size(n, T, 4, 128, 128), dtype=torch.uint8,
                     device="cuda")
    o_e, S_e = chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=n, workspace=ws)
    torch.cuda.synchronize()
    o, S = torch.full_like(o_e, float("nan")), torch.full_like(S_e, float("nan"))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ops.chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=n, o=o, S_final=S,
                      workspace=ws, stream=s)
    for _ in range(2):
        o.fill_(float("nan"))
        S.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_e) and torch.equal(S, S_e)
    assert ops.read_device_status(ws) == 0


@pytest.mark.parametrize("seed", range(16))
def test_claimed_solve_seeded_sweep(seed, monkeypatch):
    # seeded packed batches the claiming form takes (32 chunks or more per sequence on
    # average, 40 to 136 chains: fewer long chains take the segmented schedule): lengths
    # from 0 to 9000 tokens, 3-8 sequences, one or two value slices, an initial state or
    # none, the additive rule at random; bit-equal to the phased schedule and within 2e-2
    # of the oracle (head 0)
    rng = np.random.default_rng(900 + seed)
    n = int(rng.integers(3, 9))
    lens = [int(x) for x in rng.integers(0, 9001, size=n)]
    lens[int(rng.integers(0, n))] = max(lens) + 2048  # at least one long sequence
    dv = 256 if rng.random() < 0.3 else 128
    per = n * (dv // 128)
    H = int(rng.integers(-(-40 // per), 136 // per + 1))
    inp = inputs.prefill_inputs(lens, H=H, dk=128, dv=dv, dtype="bf16", seed=1000 + seed,
                                s0_std=0.3 if rng.random() < 0.6 else 0.0,
                                gate="slow" if rng.random() < 0.5 else "default", packed=True)
    if sum(lens) < 32 * 64 * n:
        pytest.skip("too short on average for the claiming form")
    kw = dict(rule="additive") if rng.random() < 0.25 else {}
    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    assert ops.chunk_fwd_schedule(n, inp.total_tokens, H, 128, dv, torch.bfloat16,
                                  varlen=True) == 0
    o_c, S_c = call(inp, **kw)
    monkeypatch.setenv("GDR_PREFILL_PHASES", "1")
    o_p, S_p = call(inp, **kw)
    assert torch.equal(o_c, o_p) and torch.equal(S_c, S_p)
    import oracle
    h0 = lambda t: f64(t[:, :1])  # head 0 only
    cu = inp.cu_seqlens.numpy().astype(np.int64)
    o_ref, S_ref = oracle.forward(h0(inp.q), h0(inp.k), h0(inp.v), h0(inp.log_alpha),
                                  h0(inp.beta), S0=None if inp.S0 is None else h0(inp.S0),
                                  cu_seqlens=cu, additive=bool(kw))
    o_g, S_g = h0(o_c), h0(S_c)
    assert np.isfinite(o_g).all() and np.isfinite(S_g).all()
    assert rel_err(o_g, o_ref) <= TOL["bf16"], rel_err(o_g, o_ref)
    assert rel_err(S_g, S_ref) <= TOL["bf16"], rel_err(S_g, S_ref)
