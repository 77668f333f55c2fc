"""GPU parity of per-channel decay (gdr_options.decay = GDR_DECAY_CHANNEL) against the oracle.

One forget rate per token, head and key channel: row c of the state decays by
alpha_t[c] ("Attention as Matrix Algebra: From Softmax to the Delta Rule", section 10:
Kimi Delta Attention gives each feature channel its own rate). The oracle takes
log_alpha [T, H, d_k] and runs the same token loop. Prefill with bf16 inputs and
d_k = d_v = 128 runs on the per-channel tensor-core path (a chunk-parallel kernel folds
each channel's decay into the operands, the chain applies it per state row); other
sizes run on the exact fp32 path (the decay inside the Gram products). Decode streams the
state once with the rates applied per row. Tolerances as for every path: max |gpu -
oracle| / max |oracle| <= 1e-4 for fp32 inputs and <= 2e-2 for bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_03_gb300 import inputs, ops
from tests.helpers import TOL, chunk_fwd, decode_step, f64, gpu_prefill, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu


def check(inp, heads=None, per_sequence=False, **kw):
    d = lambda t: None if t is None else t.cuda()
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), S0=d(inp.S0),
                     cu_seqlens=d(inp.cu_seqlens), num_seqs=inp.num_seqs, **kw)
    torch.cuda.synchronize()
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
            if cu[n + 1] > cu[n]:
                assert rel_err(o_g[cu[n]:cu[n + 1]], o_ref[cu[n]:cu[n + 1]]) <= tol, n
            assert rel_err(S_g[n], S_ref[n]) <= tol, n
    return eo, es


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 256), (64, 32), (128, 96)])
@pytest.mark.parametrize("gate", ["default", "slow", "none", "strong"])
def test_ragged_packed(dtype, dk, dv, gate):
    # ragged tails, a one-token and a one-chunk sequence, a nonzero S0
    inp = inputs.prefill_inputs([200, 64, 1, 130], H=3, dk=dk, dv=dv, dtype=dtype,
                                seed=600 + dk + dv, s0_std=0.5, gate=gate, decay="channel")
    assert tuple(inp.log_alpha.shape) == (inp.total_tokens, 3, dk)
    check(inp, per_sequence=True)


def test_empty_sequences_keep_their_state():
    inp = inputs.prefill_inputs([0, 70, 0, 5], H=2, dk=64, dv=64, dtype="f32", seed=610,
                                s0_std=0.5, gate="slow", decay="channel")
    check(inp, per_sequence=True)


def test_equal_rates_match_the_head_rate():
    # the same rate in every channel is the one-rate-per-head recurrence
    inp = inputs.prefill_inputs([300, 77], H=2, dk=128, dv=128, dtype="f32", seed=611,
                                s0_std=0.3, gate="slow")
    d = lambda t: None if t is None else t.cuda()
    o_h, S_h = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta),
                         S0=d(inp.S0), cu_seqlens=d(inp.cu_seqlens))
    la_c = inp.log_alpha[:, :, None].expand(-1, -1, 128).contiguous()
    o_c, S_c = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(la_c), d(inp.beta), S0=d(inp.S0),
                         cu_seqlens=d(inp.cu_seqlens))
    torch.cuda.synchronize()
    assert rel_err(f64(o_c), f64(o_h)) <= 1e-5 and rel_err(f64(S_c), f64(S_h)) <= 1e-5


def test_prefill_workload_shape_sampled_heads():
    # the prefill_bf16 shapes (4 x 4096 tokens, 16 heads, d = 128) with per-channel rates;
    # the oracle checks heads 0 and 9
    w = inputs.WORKLOADS["prefill_bf16"]
    inp = inputs.prefill_inputs([w["seq_len"]] * w["num_seqs"], H=w["H"], dk=128, dv=128,
                                dtype="bf16", seed=w["seed"], gate="slow", decay="channel")
    assert ops.chunk_fwd_workspace_size(inp.num_seqs, inp.total_tokens, inp.H, 128, 128,
                                        decay="channel") > 0
    check(inp, heads=[0, 9])


@pytest.mark.parametrize("tau", [64, 100])
def test_split_and_resume(tau):
    inp = inputs.prefill_inputs([230], H=2, dk=64, dv=64, dtype="f32", seed=612, s0_std=0.4,
                                gate="slow", decay="channel")
    c = lambda t: t.cuda()
    q, k, v, la, b = c(inp.q), c(inp.k), c(inp.v), c(inp.log_alpha), c(inp.beta)
    o1, S1 = chunk_fwd(q[:tau].contiguous(), k[:tau].contiguous(), v[:tau].contiguous(),
                       la[:tau].contiguous(), b[:tau].contiguous(), S0=c(inp.S0))
    o2, S2 = chunk_fwd(q[tau:].contiguous(), k[tau:].contiguous(), v[tau:].contiguous(),
                       la[tau:].contiguous(), b[tau:].contiguous(), S0=S1)
    o, S = chunk_fwd(q, k, v, la, b, S0=c(inp.S0))
    torch.cuda.synchronize()
    assert rel_err(f64(torch.cat([o1, o2])), f64(o)) <= 1e-5
    assert rel_err(f64(S2), f64(S)) <= 1e-5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_additive_rule(dtype):
    inp = inputs.prefill_inputs([200, 64, 1, 130], H=3, dk=128, dv=128, dtype=dtype, seed=613,
                                s0_std=0.5, gate="slow", decay="channel")
    d = lambda t: None if t is None else t.cuda()
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), S0=d(inp.S0),
                     cu_seqlens=d(inp.cu_seqlens), rule="additive")
    torch.cuda.synchronize()
    cu = inp.cu_seqlens.numpy().astype(np.int64)
    o_ref, S_ref = oracle.forward(f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.log_alpha),
                                  f64(inp.beta), S0=f64(inp.S0), cu_seqlens=cu, additive=True)
    assert rel_err(f64(o), o_ref) <= TOL[dtype] and rel_err(f64(S), S_ref) <= TOL[dtype]


@pytest.mark.parametrize("dv", [128, 256])
def test_prologue_and_output_step(dv):
    # raw q, k and per-channel gate pre-activations, with the output step after
    rng = np.random.default_rng(614 + dv)
    lens, H, dk = [150, 64, 33], 2, 128
    T = sum(lens)
    st = lambda x: torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    q, k = st(rng.standard_normal((T, H, dk))), st(rng.standard_normal((T, H, dk)))
    v = st(rng.standard_normal((T, H, dv)))
    a = torch.from_numpy((rng.standard_normal((T, H, dk)) - 4.0).astype(np.float32))
    b = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32))
    A = torch.from_numpy(rng.uniform(0.2, 2.0, H).astype(np.float32))
    S0 = torch.from_numpy((0.3 * rng.standard_normal((3, H, dk, dv))).astype(np.float32))
    z = st(2.0 * rng.standard_normal((T, H, dv)))
    w = torch.from_numpy(rng.uniform(0.5, 1.5, dv).astype(np.float32))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    c = lambda t: t.cuda()
    o, S = chunk_fwd(c(q), c(k), c(v), c(a), c(b), S0=c(S0), cu_seqlens=c(cu), prologue=True,
                     gate_A=c(A), out_gate=c(z), out_norm_weight=c(w), out_norm_eps=1e-5)
    torch.cuda.synchronize()
    qn, kn, la, beta = oracle.layer_prologue(f64(q), f64(k), f64(a), f64(b), f64(A))
    o_ref, S_ref = oracle.forward(qn, kn, f64(v), la, beta, S0=f64(S0),
                                  cu_seqlens=cu.numpy().astype(np.int64))
    o_ref = oracle.out_norm_gate(o_ref, f64(z), f64(w), eps=1e-5)
    assert rel_err(f64(o), o_ref) <= TOL["bf16"] and rel_err(f64(S), S_ref) <= TOL["bf16"]


# ------------------------------------------------- prefill on the per-channel tensor-core path

def test_bf16_128_takes_the_channel_tensor_path():
    assert ops.chunk_fwd_path(128, 128, torch.bfloat16, "channel") == ops.PATH_CHANNEL_TENSOR
    assert ops.chunk_fwd_main_kernel(128, 128, torch.bfloat16, decay="channel") == \
        "channel_prep_kernel"
    assert ops.chunk_fwd_compute_dtype(128, 128, torch.bfloat16, "channel") == "bf16"


@pytest.mark.parametrize("lens", [[64], [63], [1], [65, 64], [2048], [130, 1, 64, 700, 0, 65]])
def test_tensor_path_lengths(lens):
    # one chunk, a short one, a single token, two chunks, a long chain, and a packed mix
    # with an empty sequence: ragged tails fall inside the chunk-parallel tiles
    inp = inputs.prefill_inputs(lens, H=3, dk=128, dv=128, dtype="bf16", seed=650 + len(lens),
                                s0_std=0.5, gate="default", decay="channel", packed=True)
    check(inp, per_sequence=True)


def test_tensor_path_mixes_factored_and_exact_chunks():
    # channels that lose e^-160 over half a chunk cannot be split into two bounded
    # factors around the chunk's middle token; those chunks build their Gram products
    # one element at a time, the others from factored operands, in the same call
    rng = np.random.default_rng(651)
    inp = inputs.prefill_inputs([300, 200], H=2, dk=128, dv=128, dtype="bf16", seed=651,
                                s0_std=0.5, gate="slow", decay="channel")
    la = inp.log_alpha.clone()
    steep = rng.choice(128, 5, replace=False)
    la[64:128, 0, steep] = -5.0  # chunk 1 of sequence 0, head 0
    la[300 + 130:300 + 200, 1, steep[:2]] = -6.0  # the tail of sequence 1, head 1
    la[200:230, :, :] = -0.02  # slow everywhere in between
    inp.log_alpha = la
    check(inp, per_sequence=True)


def test_tensor_path_output_step():
    inp = inputs.prefill_inputs([150, 64, 33], H=2, dk=128, dv=128, dtype="bf16", seed=652,
                                s0_std=0.3, gate="default", decay="channel")
    rng = np.random.default_rng(652)
    z = torch.from_numpy((2.0 * rng.standard_normal((inp.total_tokens, 2, 128))).astype(
        np.float32)).to(torch.bfloat16)
    w = torch.from_numpy(rng.uniform(0.5, 1.5, 128).astype(np.float32))
    d = lambda t: None if t is None else t.cuda()
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), S0=d(inp.S0),
                     cu_seqlens=d(inp.cu_seqlens), out_gate=d(z), out_norm_weight=d(w),
                     out_norm_eps=1e-5)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle_prefill(inp)
    o_ref = oracle.out_norm_gate(o_ref, f64(z), f64(w), eps=1e-5)
    assert rel_err(f64(o), o_ref) <= TOL["bf16"] and rel_err(f64(S), S_ref) <= TOL["bf16"]


def test_tensor_path_equal_rates_match_the_head_rate_path():
    # the same rate in every channel: the per-channel and the one-rate-per-head tensor-core
    # paths compute the same recurrence with different operand scalings
    inp = inputs.prefill_inputs([300, 77], H=2, dk=128, dv=128, dtype="bf16", seed=653,
                                s0_std=0.3, gate="default")
    d = lambda t: None if t is None else t.cuda()
    o_h, S_h = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta),
                         S0=d(inp.S0), cu_seqlens=d(inp.cu_seqlens))
    la_c = inp.log_alpha[:, :, None].expand(-1, -1, 128).contiguous()
    o_c, S_c = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(la_c), d(inp.beta), S0=d(inp.S0),
                         cu_seqlens=d(inp.cu_seqlens))
    torch.cuda.synchronize()
    assert rel_err(f64(o_c), f64(o_h)) <= TOL["bf16"] and rel_err(f64(S_c), f64(S_h)) <= TOL["bf16"]


@pytest.mark.parametrize("lens", [[0, 70, 0, 5], [0, 0]])
def test_tensor_path_empty_sequences_keep_their_state(lens):
    inp = inputs.prefill_inputs(lens, H=2, dk=128, dv=128, dtype="bf16", seed=654,
                                s0_std=0.5, gate="slow", decay="channel", packed=True)
    check(inp, per_sequence=True)


def test_tensor_path_in_place_state_graph_capture_and_repeated_calls():
    # S_final may be S0 (each chain thread reads its entries of S0 before it writes the same
    # entries of S_final); calls on one workspace give identical bits; the call captures
    # into a CUDA graph on one stream and its replay gives the same bits again
    inp = inputs.prefill_inputs([300, 77, 64], H=2, dk=128, dv=128, dtype="bf16", seed=655,
                                s0_std=0.3, gate="default", decay="channel")
    d = lambda t: None if t is None else t.cuda()
    q, k, v, la, b, S0, cu = map(d, (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0,
                                     inp.cu_seqlens))
    n, T = inp.num_seqs, inp.total_tokens
    ws = torch.empty(ops.chunk_fwd_workspace_size(n, T, 2, 128, 128, decay="channel"),
                     dtype=torch.uint8, device="cuda")
    o_e, S_e = chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, workspace=ws)
    o_e2, S_e2 = chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, workspace=ws)
    S_io = S0.clone()
    o_io, _ = chunk_fwd(q, k, v, la, b, S0=S_io, cu_seqlens=cu, S_final=S_io, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o_e, o_e2) and torch.equal(S_e, S_e2)
    assert torch.equal(o_io, o_e) and torch.equal(S_io, S_e)
    o, S = torch.empty_like(o_e), torch.empty_like(S_e)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ops.chunk_fwd(q, k, v, la, b, S0=S0, cu_seqlens=cu, o=o, S_final=S, workspace=ws,
                      stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_e) and torch.equal(S, S_e)
    assert ops.read_device_status(ws) == 0
    o_ref, S_ref = oracle_prefill(inp)
    assert rel_err(f64(o_e), o_ref) <= TOL["bf16"] and rel_err(f64(S_e), S_ref) <= TOL["bf16"]


def test_tensor_path_rates_at_a_4_byte_offset():
    # log_alpha needs only 4-byte alignment; at an offset that is not a multiple of 16
    # bytes the operands kernel has no tensor map of it (no L2 prefetch), same results
    inp = inputs.prefill_inputs([300, 77], H=2, dk=128, dv=128, dtype="bf16", seed=656,
                                s0_std=0.3, gate="default", decay="channel")
    d = lambda t: None if t is None else t.cuda()
    flat = torch.empty(inp.log_alpha.numel() + 1, dtype=torch.float32, device="cuda")
    la_off = flat[1:].view(inp.log_alpha.shape)
    la_off.copy_(inp.log_alpha)
    assert la_off.data_ptr() % 16 == 4
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), la_off, d(inp.beta), S0=d(inp.S0),
                     cu_seqlens=d(inp.cu_seqlens))
    o_a, S_a = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta),
                         S0=d(inp.S0), cu_seqlens=d(inp.cu_seqlens))
    torch.cuda.synchronize()
    assert torch.equal(o, o_a) and torch.equal(S, S_a)
    o_ref, S_ref = oracle_prefill(inp)
    assert rel_err(f64(o), o_ref) <= TOL["bf16"] and rel_err(f64(S), S_ref) <= TOL["bf16"]


@pytest.mark.parametrize("steep", [False, True])
def test_tensor_path_prologue(steep):
    # raw q, k and per-channel gate pre-activations on the tensor-core path; steep: rates
    # large enough that chunks take the exact element-wise Gram
    rng = np.random.default_rng(657 + steep)
    lens, H, dk = [300, 64, 33], 2, 128
    T = sum(lens)
    assert ops.chunk_fwd_path(dk, dk, torch.bfloat16, "channel", prologue=True) == \
        ops.PATH_CHANNEL_TENSOR
    st = lambda x: torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    q, k = st(rng.standard_normal((T, H, dk))), st(3.0 * rng.standard_normal((T, H, dk)))
    v = st(rng.standard_normal((T, H, dk)))
    a = torch.from_numpy((rng.standard_normal((T, H, dk)) + (3.0 if steep else -4.0)).astype(np.float32))
    b = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32))
    A = torch.from_numpy(rng.uniform(0.2, 2.0, H).astype(np.float32))
    S0 = torch.from_numpy((0.3 * rng.standard_normal((3, H, dk, dk))).astype(np.float32))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    c = lambda t: t.cuda()
    o, S = chunk_fwd(c(q), c(k), c(v), c(a), c(b), S0=c(S0), cu_seqlens=c(cu), prologue=True,
                     gate_A=c(A))
    torch.cuda.synchronize()
    qn, kn, la, beta = oracle.layer_prologue(f64(q), f64(k), f64(a), f64(b), f64(A))
    o_ref, S_ref = oracle.forward(qn, kn, f64(v), la, beta, S0=f64(S0),
                                  cu_seqlens=cu.numpy().astype(np.int64))
    assert rel_err(f64(o), o_ref) <= TOL["bf16"] and rel_err(f64(S), S_ref) <= TOL["bf16"]


def test_log_alpha_shape_is_checked():
    inp = inputs.prefill_inputs([64], H=2, dk=64, dv=64, dtype="f32", seed=615)
    c = lambda t: t.cuda()
    bad = torch.zeros((64, 2, 32), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        chunk_fwd(c(inp.q), c(inp.k), c(inp.v), bad, c(inp.beta))


# --------------------------------------------------------------------------- decode

def decode_steps(d, **kw):
    S = d.S.cuda()
    outs = []
    for s in range(d.steps):
        outs.append(decode_step(d.q[s].cuda(), d.k[s].cuda(), d.v[s].cuda(),
                                d.log_alpha[s].cuda(), d.beta[s].cuda(), S, **kw))
    torch.cuda.synchronize()
    return [f64(o) for o in outs], f64(S)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 256), (128, 64), (128, 128), (128, 256)])
def test_decode_shapes(dtype, dk, dv):
    d = inputs.decode_inputs(N=5, H=3, dk=dk, dv=dv, steps=4, dtype=dtype, seed=620 + dk + dv,
                             s0_std=0.5, decay="channel")
    outs, S = decode_steps(d)
    S_ref = f64(d.S)
    for s in range(d.steps):
        o_ref, S_ref = oracle.decode(f64(d.q[s]), f64(d.k[s]), f64(d.v[s]), f64(d.log_alpha[s]),
                                     f64(d.beta[s]), S_ref)
        assert rel_err(outs[s], o_ref) <= TOL[dtype], s
    assert rel_err(S, S_ref) <= TOL[dtype]


def test_decode_workload_shape():
    # decode_bf16's shapes (256 sequences x 32 heads, d = 128) with per-channel rates
    d = inputs.decode_inputs(N=256, H=32, dk=128, dv=128, steps=2, dtype="bf16", seed=3,
                             s0_std=0.02, decay="channel")
    outs, S = decode_steps(d)
    sel = slice(0, 16)  # the oracle on the first 16 sequences
    S_ref = f64(d.S)[sel]
    for s in range(d.steps):
        o_ref, S_ref = oracle.decode(f64(d.q[s])[sel], f64(d.k[s])[sel], f64(d.v[s])[sel],
                                     f64(d.log_alpha[s])[sel], f64(d.beta[s])[sel], S_ref)
        assert rel_err(outs[s][sel], o_ref) <= TOL["bf16"], s
    assert rel_err(S[sel], S_ref) <= TOL["bf16"]


def test_prefill_then_decode_equals_longer_prefill():
    full = inputs.prefill_inputs([150], H=2, dk=128, dv=128, dtype="f32", seed=630,
                                 s0_std=0.2, gate="slow", decay="channel")
    c = lambda t: t.cuda()
    q, k, v, la, b = c(full.q), c(full.k), c(full.v), c(full.log_alpha), c(full.beta)
    tau = 140
    _, S = chunk_fwd(q[:tau].contiguous(), k[:tau].contiguous(), v[:tau].contiguous(),
                     la[:tau].contiguous(), b[:tau].contiguous(), S0=c(full.S0))
    outs = [decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1], b[t:t + 1], S)
            for t in range(tau, 150)]
    o_all, S_all = chunk_fwd(q, k, v, la, b, S0=c(full.S0))
    torch.cuda.synchronize()
    assert rel_err(f64(torch.cat(outs)), f64(o_all[tau:])) <= 1e-5
    assert rel_err(f64(S), f64(S_all)) <= 1e-5


@pytest.mark.parametrize("rule", ["delta", "additive"])
def test_decode_rule_prologue_and_output_step(rule):
    rng = np.random.default_rng(640)
    N, H, dk, dv = 6, 4, 128, 128
    st = lambda x: torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    q, k, v = (st(rng.standard_normal((N, H, n))) for n in (dk, dk, dv))
    a = torch.from_numpy((rng.standard_normal((N, H, dk)) - 3.0).astype(np.float32))
    b = torch.from_numpy(rng.standard_normal((N, H)).astype(np.float32))
    A = torch.from_numpy(rng.uniform(0.2, 2.0, H).astype(np.float32))
    S = torch.from_numpy((0.3 * rng.standard_normal((N, H, dk, dv))).astype(np.float32))
    z = st(2.0 * rng.standard_normal((N, H, dv)))
    c = lambda t: t.cuda()
    Sg = c(S)
    o = decode_step(c(q), c(k), c(v), c(a), c(b), Sg, rule=rule, prologue=True, gate_A=c(A),
                    out_gate=c(z))
    torch.cuda.synchronize()
    qn, kn, la, beta = oracle.layer_prologue(f64(q), f64(k), f64(a), f64(b), f64(A))
    o_ref, S_ref = oracle.forward(qn, kn, f64(v), la, beta, S0=f64(S), num_seqs=N,
                                  additive=rule == "additive")
    o_ref = oracle.out_norm_gate(o_ref, f64(z))
    assert rel_err(f64(o), o_ref) <= TOL["bf16"] and rel_err(f64(Sg), S_ref) <= TOL["bf16"]
