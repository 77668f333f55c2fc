"""GPU parity of the layer prologue (gdr_options.prologue = GDR_PROLOGUE_LAYER): raw q and
k scaled to unit length inside the kernels, and the gates from their pre-activations
(log alpha = -A_h softplus(a), beta = sigmoid(b)).

The reference is oracle.layer_prologue on the exact raw inputs the GPU receives, then
oracle.forward / oracle.decode, all float64. Raw q, k ~ N(0, 1) of length about
sqrt(d_k) (not unit), gates a ~ N(0, 1) + offset, b ~ N(0, 1), A_h ~ U(0.2, 2). Tolerances
as for the recurrence (1e-4 fp32 inputs, 2e-2 bf16 inputs); with bf16 the kernels scale
the bf16 raw vectors, the reference the same bf16 values in float64.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_03_gb300 import inputs
from tests.helpers import TOL, chunk_fwd, decode_step, f64, rel_err

pytestmark = pytest.mark.gpu


def raw_inputs(lens, H, dk, dv, dtype, seed, s0_std=0.3, a_shift=-4.0):
    """Raw (un-normalised) q, k, v; gate pre-activations a, b; per-head A; S0."""
    rng = np.random.default_rng(seed)
    T = int(sum(lens))
    st = lambda x: torch.from_numpy(x.astype(np.float32)).to(inputs.TORCH_DTYPES[dtype])
    q, k = st(rng.standard_normal((T, H, dk))), st(rng.standard_normal((T, H, dk)))
    v = st(rng.standard_normal((T, H, dv)))
    a = torch.from_numpy((rng.standard_normal((T, H)) + a_shift).astype(np.float32))
    b = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32))
    A = torch.from_numpy(rng.uniform(0.2, 2.0, H).astype(np.float32))
    S0 = torch.from_numpy((s0_std * rng.standard_normal((len(lens), H, dk, dv))).astype(np.float32))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32) \
        if len(set(lens)) > 1 else None
    return q, k, v, a, b, A, S0, cu


def reference(q, k, v, a, b, A, S0, cu, num_seqs):
    qn, kn, la, beta = oracle.layer_prologue(f64(q), f64(k), f64(a), f64(b), f64(A))
    return oracle.forward(qn, kn, f64(v), la, beta, S0=f64(S0),
                          cu_seqlens=None if cu is None else cu.numpy().astype(np.int64),
                          num_seqs=num_seqs)


def run(q, k, v, a, b, A, S0, cu, num_seqs):
    c = lambda t: None if t is None else t.cuda()
    o, S = chunk_fwd(c(q), c(k), c(v), c(a), c(b), S0=c(S0), cu_seqlens=c(cu), num_seqs=num_seqs,
                     prologue=True, gate_A=c(A))
    torch.cuda.synchronize()
    return f64(o), f64(S)


@pytest.mark.parametrize("dtype,dk,dv", [("f32", 64, 64), ("bf16", 64, 128), ("bf16", 128, 128),
                                         ("bf16", 128, 256)])
@pytest.mark.parametrize("a_shift", [-4.0, 0.0])
def test_prefill_packed(dtype, dk, dv, a_shift):
    lens = [200, 64, 1, 130]
    args = raw_inputs(lens, 3, dk, dv, dtype, seed=140 + dk + dv, a_shift=a_shift)
    o, S = run(*args, len(lens))
    o_ref, S_ref = reference(*args, len(lens))
    tol = TOL[dtype]
    assert rel_err(o, o_ref) <= tol and rel_err(S, S_ref) <= tol


@pytest.mark.parametrize("S_,T,H,dv", [(2, 1000, 3, 128), (3, 640, 2, 256)])
def test_prefill_fused_schedule(S_, T, H, dv, monkeypatch):
    # equal lengths take the fused schedule; the phased one gives the same bits
    args = raw_inputs([T] * S_, H, 128, dv, "bf16", seed=150 + S_)
    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    o_f, S_f = run(*args, S_)
    monkeypatch.setenv("GDR_PREFILL_PHASES", "1")
    o_p, S_p = run(*args, S_)
    np.testing.assert_array_equal(o_f, o_p)
    np.testing.assert_array_equal(S_f, S_p)
    o_ref, S_ref = reference(*args, S_)
    assert rel_err(o_f, o_ref) <= TOL["bf16"] and rel_err(S_f, S_ref) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 256)])
def test_decode_steps(dtype, dk, dv):
    N, H = 5, 3
    q, k, v, a, b, A, S0, _ = raw_inputs([1] * N, H, dk, dv, dtype, seed=160 + dk + dv)
    S = S0.cuda()
    S_ref = f64(S0)
    for step in range(3):
        rng = np.random.default_rng(170 + step)
        qs = q if step == 0 else torch.from_numpy(rng.standard_normal(q.shape).astype(np.float32)).to(q.dtype)
        o = decode_step(qs.cuda(), k.cuda(), v.cuda(), a.cuda(), b.cuda(), S, prologue=True,
                        gate_A=A.cuda())
        torch.cuda.synchronize()
        qn, kn, la, beta = oracle.layer_prologue(f64(qs), f64(k), f64(a), f64(b), f64(A))
        o_ref, S_ref = oracle.decode(qn, kn, f64(v), la, beta, S_ref)
        assert rel_err(f64(o), o_ref) <= TOL[dtype], step
    assert rel_err(f64(S), S_ref) <= TOL[dtype]
