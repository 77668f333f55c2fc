"""GPU parity of gdr_chunk_fwd against the float64 oracle, element by element.

Tolerance: max |gpu - oracle| / max |oracle| per output tensor, <= 1e-4 for fp32
inputs and <= 2e-2 for bf16 inputs. With the workloads' default gates
(alpha about 0.45) a chunk decays the state by about e^-52, so state passing
between chunks is numerically invisible there; the "none" (alpha = 1) and
"slow" (alpha about 0.9975) gate variants with a nonzero S0 exercise it.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_03_gb300 import inputs
from tests.helpers import TOL, chunk_fwd, gpu_prefill, oracle_prefill, rel_err, f64

pytestmark = pytest.mark.gpu


def check(inp, heads=None, per_sequence=False):
    o, S = gpu_prefill(inp)
    o_ref, S_ref = oracle_prefill(inp, heads)
    o_g, S_g = f64(o), f64(S)
    if heads is not None:
        o_g, S_g = o_g[:, list(heads)], S_g[:, list(heads)]
    assert np.isfinite(o_g).all() and np.isfinite(S_g).all()
    tol = TOL[inp.dtype]
    eo, es = rel_err(o_g, o_ref), rel_err(S_g, S_ref)
    assert eo <= tol and es <= tol, (eo, es)
    if per_sequence and inp.cu_seqlens is not None:
        cu = inp.cu_seqlens.numpy()
        for n in range(inp.num_seqs):
            sl = slice(cu[n], cu[n + 1])
            if cu[n + 1] > cu[n]:
                assert rel_err(o_g[sl], o_ref[sl]) <= tol, n
            assert rel_err(S_g[n], S_ref[n]) <= tol, n
    return eo, es


def test_tiny_fp32_workload():
    check(inputs.workload_prefill("tiny_fp32"))


@pytest.mark.parametrize("gate", ["default", "slow", "none", "strong"])
def test_prefill_bf16_workload(gate):
    check(inputs.workload_prefill("prefill_bf16", gate=gate))


@pytest.mark.parametrize("gate", ["default", "slow"])
def test_varlen_bf16_workload(gate):
    check(inputs.workload_prefill("varlen_bf16", gate=gate), per_sequence=True)


def test_long_bf16_workload_heads_0_1():
    check(inputs.workload_prefill("long_bf16"), heads=[0, 1])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 256), (64, 32), (128, 96)])
@pytest.mark.parametrize("gate", ["default", "slow", "none", "strong"])
def test_ragged_multi_chunk(dtype, dk, dv, gate):
    # several chunks plus a ragged tail, nonzero initial state
    inp = inputs.prefill_inputs([200, 64, 1, 130], H=3, dk=dk, dv=dv, dtype=dtype,
                                seed=dk + dv, s0_std=0.5, gate=gate)
    check(inp, per_sequence=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_empty_and_zero_length_sequences(dtype):
    inp = inputs.prefill_inputs([0, 70, 0, 5, 0], H=2, dk=128, dv=128, dtype=dtype, seed=5,
                                s0_std=1.0)
    o, S = gpu_prefill(inp)
    cu = inp.cu_seqlens.numpy()
    for n in (0, 2, 4):
        assert cu[n + 1] == cu[n]
        np.testing.assert_array_equal(f64(S[n]), f64(inp.S0[n]))
    check(inp, per_sequence=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_no_tokens_at_all(dtype):
    inp = inputs.prefill_inputs([0, 0], H=2, dk=64, dv=64, dtype=dtype, seed=6, s0_std=1.0,
                                packed=True)
    o, S = gpu_prefill(inp)
    assert o.shape[0] == 0
    np.testing.assert_array_equal(f64(S), f64(inp.S0))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("tau", [1, 63, 64, 100, 257])
def test_split_and_resume(dtype, tau):
    # prefill [0, tau) then [tau, T) passing S equals one call over [0, T), for any tau
    full = inputs.prefill_inputs([300], H=2, dk=128, dv=128, dtype=dtype, seed=7, s0_std=0.3,
                                 gate="slow")
    dev = lambda t: None if t is None else t.cuda()
    q, k, v, la, b, S0 = (dev(full.q), dev(full.k), dev(full.v), dev(full.log_alpha),
                          dev(full.beta), dev(full.S0))
    o_all, S_all = chunk_fwd(q, k, v, la, b, S0=S0)
    o1, S1 = chunk_fwd(q[:tau].contiguous(), k[:tau].contiguous(), v[:tau].contiguous(),
                       la[:tau].contiguous(), b[:tau].contiguous(), S0=S0)
    o2, S2 = chunk_fwd(q[tau:].contiguous(), k[tau:].contiguous(), v[tau:].contiguous(),
                       la[tau:].contiguous(), b[tau:].contiguous(), S0=S1)
    torch.cuda.synchronize()
    tol = TOL[dtype]
    assert rel_err(f64(torch.cat([o1, o2])), f64(o_all)) <= tol
    assert rel_err(f64(S2), f64(S_all)) <= tol
    o_ref, S_ref = oracle_prefill(full)
    assert rel_err(f64(S2), S_ref) <= tol


def test_in_place_state_update():
    inp = inputs.prefill_inputs([150, 90], H=2, dk=128, dv=128, dtype="bf16", seed=8,
                                s0_std=0.5, gate="slow")
    o_ref, S_ref = oracle_prefill(inp)
    S = inp.S0.cuda()
    o, S_out = chunk_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.log_alpha.cuda(),
                         inp.beta.cuda(), S0=S, cu_seqlens=inp.cu_seqlens.cuda(), S_final=S)
    torch.cuda.synchronize()
    assert S_out.data_ptr() == S.data_ptr()
    assert rel_err(f64(S), S_ref) <= 2e-2
    assert rel_err(f64(o), o_ref) <= 2e-2


@pytest.mark.parametrize("dv", [128, 256])
@pytest.mark.parametrize("phases", [2, 3, 5, 8])
def test_phase_split_matches_single_phase(phases, dv, monkeypatch):
    # The tensor path may split each sequence's chunks into phases (the solve of the next
    # phase overlapping the chain of this one); the state passes between phases in fp32
    # as it does between chunks, so every phase count gives the single-phase bits.
    # Sequences shorter than the phase count leave some phases empty; one is empty.
    inp = inputs.prefill_inputs([700, 64, 1, 0, 130, 2000], H=3, dk=128, dv=dv, dtype="bf16",
                                seed=11 + dv, s0_std=0.5, gate="slow")
    monkeypatch.setenv("GDR_PREFILL_PHASES", "1")
    o1, S1 = gpu_prefill(inp)
    monkeypatch.setenv("GDR_PREFILL_PHASES", str(phases))
    from gated_delta_rule_03_gb300 import ops
    assert ops.chunk_fwd_kernel_launches(inp.num_seqs, inp.total_tokens, inp.H, 128, dv,
                                         torch.bfloat16, varlen=True) == 1 + 2 * phases
    oP, SP = gpu_prefill(inp)
    assert torch.equal(o1, oP) and torch.equal(S1, SP)
    check(inp, per_sequence=True)


@pytest.mark.parametrize("phases", [1, 4])
def test_phase_split_in_place_state(phases, monkeypatch):
    # S_final may be S0: the first phase reads S0 and the last writes S_final
    monkeypatch.setenv("GDR_PREFILL_PHASES", str(phases))
    inp = inputs.prefill_inputs([640, 1000, 3], H=2, dk=128, dv=128, dtype="bf16", seed=12,
                                s0_std=0.5, gate="none")
    o_ref, S_ref = oracle_prefill(inp)
    S = inp.S0.cuda()
    o, _ = chunk_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.log_alpha.cuda(),
                     inp.beta.cuda(), S0=S, cu_seqlens=inp.cu_seqlens.cuda(), S_final=S)
    torch.cuda.synchronize()
    assert rel_err(f64(S), S_ref) <= 2e-2
    assert rel_err(f64(o), o_ref) <= 2e-2


def test_phase_split_inside_graph_capture(monkeypatch):
    # the side stream forks from and joins the captured stream; replaying the graph
    # gives the eager result
    monkeypatch.setenv("GDR_PREFILL_PHASES", "4")
    inp = inputs.prefill_inputs([1024, 960], H=4, dk=128, dv=128, dtype="bf16", seed=13,
                                s0_std=0.2, gate="slow")
    dev = lambda t: t.cuda()
    q, k, v, la, b, S0 = map(dev, (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0))
    cu = inp.cu_seqlens.cuda()
    o_eager, S_eager = chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu)
    o = torch.empty_like(o_eager)
    S = torch.empty_like(S_eager)
    from gated_delta_rule_03_gb300 import ops
    ws = torch.empty(ops.chunk_fwd_workspace_size(inp.num_seqs, inp.total_tokens, inp.H, 128, 128),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # an uncaptured call on this thread first
        chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, o=o, S_final=S, workspace=ws, stream=s)
    s.synchronize()
    o.zero_()
    S.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, o=o, S_final=S, workspace=ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_eager) and torch.equal(S, S_eager)


@pytest.mark.parametrize("S,T,H,dv", [(1, 300, 2, 128), (2, 1000, 3, 128), (3, 640, 5, 256),
                                      (4, 4096, 16, 128)])
def test_fused_schedule_matches_phased(S, T, H, dv, monkeypatch):
    # Equal-length batches take the fused cooperative launch (solve and chain CTAs in one
    # grid, chains waiting on per-unit flags). Forcing the phased two-kernel schedule must
    # give the same bits; both match the oracle.
    from gated_delta_rule_03_gb300 import ops
    inp = inputs.prefill_inputs([T] * S, H=H, dk=128, dv=dv, dtype="bf16", seed=20 + S,
                                s0_std=0.5, gate="slow")
    assert inp.cu_seqlens is None
    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    assert ops.chunk_fwd_schedule(S, S * T, H, 128, dv, torch.bfloat16) == 0
    assert ops.chunk_fwd_kernel_launches(S, S * T, H, 128, dv, torch.bfloat16) == 1
    o_f, S_f = gpu_prefill(inp)
    monkeypatch.setenv("GDR_PREFILL_PHASES", "1")
    o_p, S_p = gpu_prefill(inp)
    assert torch.equal(o_f, o_p) and torch.equal(S_f, S_p)
    if S * T <= 4000:
        check(inp)


def test_fused_schedule_repeated_calls_share_a_workspace():
    # the unit flags are cleared by every call's plan: back-to-back calls on one workspace
    # and stream give identical results
    from gated_delta_rule_03_gb300 import ops
    inp = inputs.prefill_inputs([512] * 2, H=4, dk=128, dv=128, dtype="bf16", seed=31, s0_std=0.2)
    dev = lambda t: t.cuda()
    q, k, v, la, b, S0 = map(dev, (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0))
    ws = torch.empty(ops.chunk_fwd_workspace_size(2, 1024, 4, 128, 128), dtype=torch.uint8,
                     device="cuda")
    outs = [chunk_fwd(q, k, v, la, b, S0=S0, num_seqs=2, workspace=ws) for _ in range(4)]
    torch.cuda.synchronize()
    for o, S in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(S, outs[0][1])
    assert ops.read_device_status(ws) == 0


def test_bad_cu_seqlens_reported_through_the_status_word():
    from gated_delta_rule_03_gb300 import read_device_status
    inp = inputs.prefill_inputs([100, 50], H=2, dk=128, dv=128, dtype="bf16", seed=9)
    dev = "cuda"
    bad = torch.tensor([0, 120, 100 + 50], dtype=torch.int32)      # fine
    ws = torch.empty(1 << 24, dtype=torch.uint8, device=dev)
    args = [t.to(dev) for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
    chunk_fwd(*args, cu_seqlens=bad.to(dev), workspace=ws)
    assert read_device_status(ws) == 0
    bad = torch.tensor([0, 120, 110], dtype=torch.int32)           # decreasing, wrong end
    chunk_fwd(*args, cu_seqlens=bad.to(dev), workspace=ws)
    assert read_device_status(ws) == -7
    bad = torch.tensor([5, 60, 150], dtype=torch.int32)            # does not start at 0
    chunk_fwd(*args, cu_seqlens=bad.to(dev), workspace=ws)
    assert read_device_status(ws) == -7
    good = inp.cu_seqlens.to(dev)
    o, S = chunk_fwd(*args, cu_seqlens=good, workspace=ws)
    assert read_device_status(ws) == 0
    o_ref, S_ref = oracle_prefill(inp)
    assert rel_err(f64(o), o_ref) <= 2e-2


def test_beta_zero_alpha_one_keeps_the_state():
    inp = inputs.prefill_inputs([333], H=2, dk=128, dv=128, dtype="f32", seed=10, s0_std=1.0,
                                gate="none")
    inp.beta.zero_()
    o, S = gpu_prefill(inp)
    np.testing.assert_allclose(f64(S), f64(inp.S0), rtol=0, atol=1e-6)
    # o_t = S0^T q_t
    want = np.einsum("thd,hde->the", f64(inp.q), f64(inp.S0)[0])
    assert rel_err(f64(o), want) <= 1e-5


def test_unit_key_beta_one_reads_back_value():
    # beta = 1 with keys of exactly unit length: S_t^T k_t = v_t (here checked on the last token)
    rng = np.random.default_rng(11)
    T, H, dk, dv = 97, 2, 64, 64
    k = 0.125 * rng.choice([-1.0, 1.0], size=(T, H, dk))          # 64 entries of 1/8: unit norm
    inp = inputs.prefill_inputs([T], H=H, dk=dk, dv=dv, dtype="f32", seed=12, s0_std=0.1)
    inp.k.copy_(torch.from_numpy(k.astype(np.float32)))
    inp.beta.fill_(1.0)
    o, S = gpu_prefill(inp)
    readback = np.einsum("hdv,hd->hv", f64(S)[0], k[-1])
    np.testing.assert_allclose(readback, f64(inp.v)[-1], rtol=0, atol=2e-4)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_near_zero_decay_tokens(dtype):
    # alpha = 0 written as log alpha = -1e4 on a few tokens (the state is wiped there),
    # mixed with slow decay elsewhere, so chunks of both decay regimes follow each other
    inp = inputs.prefill_inputs([333, 200], H=2, dk=128, dv=128, dtype=dtype, seed=14,
                                s0_std=0.5, gate="slow")
    rng = np.random.default_rng(15)
    idx = rng.choice(inp.total_tokens, size=12, replace=False)
    la = inp.log_alpha.clone()
    la[idx, :] = -1.0e4
    inp.log_alpha.copy_(la)
    check(inp, per_sequence=True)


@pytest.mark.parametrize("dtype,dk,lens", [("bf16", 128, [512, 512]), ("bf16", 128, [300, 77]),
                                           ("f32", 64, [300, 77])])
def test_gates_at_a_4_byte_offset(dtype, dk, lens):
    # log_alpha and beta need only 4-byte alignment (per-token slices of a larger buffer):
    # the fused, phased and exact paths read them at any such offset, same bits
    inp = inputs.prefill_inputs(lens, H=2, dk=dk, dv=dk, dtype=dtype, seed=57, s0_std=0.2,
                                gate="slow")
    d = lambda t: None if t is None else t.cuda()

    def shifted(t):
        flat = torch.empty(t.numel() + 1, dtype=torch.float32, device="cuda")
        out = flat[1:].view(t.shape)
        out.copy_(t)
        assert out.data_ptr() % 16 == 4
        return out

    args = (d(inp.q), d(inp.k), d(inp.v))
    kw = dict(S0=d(inp.S0), cu_seqlens=d(inp.cu_seqlens), num_seqs=inp.num_seqs)
    o, S = chunk_fwd(*args, shifted(inp.log_alpha), shifted(inp.beta), **kw)
    o_a, S_a = chunk_fwd(*args, d(inp.log_alpha), d(inp.beta), **kw)
    torch.cuda.synchronize()
    assert torch.equal(o, o_a) and torch.equal(S, S_a)
    ref_o, ref_S = oracle_prefill(inp)
    assert rel_err(f64(o), ref_o) <= TOL[dtype] and rel_err(f64(S), ref_S) <= TOL[dtype]
