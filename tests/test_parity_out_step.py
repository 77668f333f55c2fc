"""GPU parity of the layer's output step (gdr_options.out_gate) against the oracle:
o <- o / sqrt(mean(o^2) + eps) * w * silu(z) per token and head, after the recurrence.

The reference is oracle.forward followed by oracle.out_norm_gate, both float64, on the
exact inputs the GPU receives. The step runs fused in the decode kernel and in the
tensor-core chain's epilogue (d_v = 128), and as its own kernel on the exact path and
for d_v = 256. Tolerances as for the recurrence: max |gpu - ref| / max |ref| <= 1e-4
(fp32 inputs) and 2e-2 (bf16 inputs).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_03_gb300 import inputs
from tests.helpers import TOL, chunk_fwd, decode_step, f64, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu


def gate_inputs(shape, dtype, seed, with_weight):
    rng = np.random.default_rng(seed)
    z = torch.from_numpy((2.0 * rng.standard_normal(shape)).astype(np.float32)).to(
        inputs.TORCH_DTYPES[dtype])
    w = torch.from_numpy(rng.uniform(0.5, 1.5, shape[-1]).astype(np.float32)) if with_weight else None
    return z, w


@pytest.mark.parametrize("dtype,dk,dv", [("f32", 64, 64), ("bf16", 64, 128), ("bf16", 128, 128),
                                         ("bf16", 128, 256), ("f32", 128, 96)])
@pytest.mark.parametrize("with_weight", [False, True])
def test_prefill_packed(dtype, dk, dv, with_weight):
    inp = inputs.prefill_inputs([200, 64, 1, 130], H=3, dk=dk, dv=dv, dtype=dtype,
                                seed=80 + dk + dv, s0_std=0.5, gate="slow")
    z, w = gate_inputs((inp.total_tokens, inp.H, dv), dtype, 90 + dv, with_weight)
    d = lambda t: None if t is None else t.cuda()
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), S0=d(inp.S0),
                     cu_seqlens=d(inp.cu_seqlens), num_seqs=inp.num_seqs, out_gate=d(z),
                     out_norm_weight=d(w), out_norm_eps=1e-5)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle_prefill(inp)
    o_ref = oracle.out_norm_gate(o_ref, f64(z), None if w is None else f64(w), eps=1e-5)
    tol = TOL[dtype]
    assert rel_err(f64(o), o_ref) <= tol and rel_err(f64(S), S_ref) <= tol


@pytest.mark.parametrize("S,T,H", [(2, 1000, 3), (4, 4096, 16)])
def test_prefill_fused_schedule(S, T, H, monkeypatch):
    # equal lengths, d_v = 128: the step runs inside the fused kernel's chain epilogue;
    # the phased schedule gives the same bits
    inp = inputs.prefill_inputs([T] * S, H=H, dk=128, dv=128, dtype="bf16", seed=100 + S,
                                s0_std=0.5, gate="slow")
    z, w = gate_inputs((inp.total_tokens, H, 128), "bf16", 110 + S, True)
    d = lambda t: None if t is None else t.cuda()

    def run():
        o, S_ = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta),
                          S0=d(inp.S0), num_seqs=S, out_gate=d(z), out_norm_weight=d(w))
        torch.cuda.synchronize()
        return f64(o), f64(S_)

    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    o_f, S_f = run()
    monkeypatch.setenv("GDR_PREFILL_PHASES", "1")
    o_p, S_p = run()
    np.testing.assert_array_equal(o_f, o_p)
    np.testing.assert_array_equal(S_f, S_p)
    if S * T <= 4000:
        o_ref, S_ref = oracle_prefill(inp)
        o_ref = oracle.out_norm_gate(o_ref, f64(z), f64(w), eps=1e-6)
        assert rel_err(o_f, o_ref) <= TOL["bf16"] and rel_err(S_f, S_ref) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 256)])
def test_decode_fused(dtype, dk, dv):
    dd = inputs.decode_inputs(N=5, H=3, dk=dk, dv=dv, steps=3, dtype=dtype, seed=120 + dk + dv,
                              s0_std=0.3, gate="slow")
    S = dd.S.cuda()
    S_ref = f64(dd.S)
    for s in range(dd.steps):
        z, w = gate_inputs((dd.N, dd.H, dv), dtype, 130 + s, s % 2 == 1)
        o = decode_step(dd.q[s].cuda(), dd.k[s].cuda(), dd.v[s].cuda(), dd.log_alpha[s].cuda(),
                        dd.beta[s].cuda(), S, out_gate=z.cuda(),
                        out_norm_weight=None if w is None else w.cuda())
        torch.cuda.synchronize()
        o_ref, S_ref = oracle.decode(f64(dd.q[s]), f64(dd.k[s]), f64(dd.v[s]), f64(dd.log_alpha[s]),
                                     f64(dd.beta[s]), S_ref)
        o_ref = oracle.out_norm_gate(o_ref, f64(z), None if w is None else f64(w), eps=1e-6)
        assert rel_err(f64(o), o_ref) <= TOL[dtype], s
    assert rel_err(f64(S), S_ref) <= TOL[dtype]
