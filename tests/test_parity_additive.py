"""GPU parity of the additive rule (gdr_options.rule = GDR_RULE_ADDITIVE) against the
float64 oracle's additive mode, S_t = alpha_t S_{t-1} + beta_t k_t v_t^T, o_t = S_t^T q_t.

The same tolerances as the delta rule: max |gpu - oracle| / max |oracle| per output
tensor <= 1e-4 for fp32 inputs and <= 2e-2 for bf16 inputs. The rule runs through every
kernel path: the exact fp32 path, the tensor-core path in both its schedules (phased
for packed sequences, fused for equal lengths) and the decode step.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_03_gb300 import inputs
from tests.helpers import TOL, chunk_fwd, decode_step, f64, rel_err

pytestmark = pytest.mark.gpu


def gpu_additive(inp):
    d = lambda t: None if t is None else t.cuda()
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), S0=d(inp.S0),
                     cu_seqlens=d(inp.cu_seqlens), num_seqs=inp.num_seqs, rule="additive")
    torch.cuda.synchronize()
    return f64(o), f64(S)


def oracle_additive(inp):
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy().astype(np.int64)
    return oracle.forward(f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.log_alpha), f64(inp.beta),
                          S0=None if inp.S0 is None else f64(inp.S0), cu_seqlens=cu,
                          num_seqs=inp.num_seqs, additive=True)


def check(inp):
    o, S = gpu_additive(inp)
    o_ref, S_ref = oracle_additive(inp)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    tol = TOL[inp.dtype]
    eo, es = rel_err(o, o_ref), rel_err(S, S_ref)
    assert eo <= tol and es <= tol, (eo, es)
    return eo, es


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 256)])
@pytest.mark.parametrize("gate", ["default", "slow", "none"])
def test_ragged_packed(dtype, dk, dv, gate):
    inp = inputs.prefill_inputs([200, 64, 1, 130], H=3, dk=dk, dv=dv, dtype=dtype,
                                seed=40 + dk + dv, s0_std=0.5, gate=gate)
    check(inp)


@pytest.mark.parametrize("S,T,H,dv", [(2, 1000, 3, 128), (4, 4096, 16, 128), (1, 700, 2, 256)])
def test_equal_lengths_fused(S, T, H, dv, monkeypatch):
    # equal-length batches take the fused cooperative schedule; the phased one gives the
    # same bits
    monkeypatch.delenv("GDR_PREFILL_PHASES", raising=False)
    inp = inputs.prefill_inputs([T] * S, H=H, dk=128, dv=dv, dtype="bf16", seed=50 + S,
                                s0_std=0.5, gate="slow")
    o_f, S_f = gpu_additive(inp)
    monkeypatch.setenv("GDR_PREFILL_PHASES", "1")
    o_p, S_p = gpu_additive(inp)
    np.testing.assert_array_equal(o_f, o_p)
    np.testing.assert_array_equal(S_f, S_p)
    if S * T <= 4000:
        check(inp)


def test_plain_linear_attention():
    # alpha = 1 and beta = 1: S_T = S_0 + K^T V and o_t = (S_0 + sum_{i<=t} k_i v_i^T)^T q_t
    inp = inputs.prefill_inputs([300], H=2, dk=64, dv=64, dtype="f32", seed=61, s0_std=0.3,
                                gate="none")
    inp.beta.fill_(1.0)
    o, S = gpu_additive(inp)
    q, k, v, S0 = f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.S0)
    S_ref = S0[0] + np.einsum("thd,the->hde", k, v)
    pref = S0[0][None] + np.cumsum(np.einsum("thd,the->thde", k, v), axis=0)
    o_ref = np.einsum("thd,thde->the", q, pref)
    assert rel_err(S[0], S_ref) <= TOL["f32"] and rel_err(o, o_ref) <= TOL["f32"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 128), (128, 256)])
def test_decode_steps(dtype, dk, dv):
    # a decode step is a one-token forward from the current state
    d = inputs.decode_inputs(N=6, H=3, dk=dk, dv=dv, steps=4, dtype=dtype, seed=70 + dk + dv,
                             s0_std=0.3, gate="slow")
    S = d.S.cuda()
    S_ref = f64(d.S)
    for s in range(d.steps):
        o = decode_step(d.q[s].cuda(), d.k[s].cuda(), d.v[s].cuda(), d.log_alpha[s].cuda(),
                        d.beta[s].cuda(), S, rule="additive")
        torch.cuda.synchronize()
        # N sequences of one token each, packed
        cu = np.arange(d.N + 1, dtype=np.int64)
        o_ref, S_ref = oracle.forward(f64(d.q[s]), f64(d.k[s]), f64(d.v[s]),
                                      f64(d.log_alpha[s]), f64(d.beta[s]), S0=S_ref,
                                      cu_seqlens=cu, num_seqs=d.N, additive=True)
        assert rel_err(f64(o), o_ref) <= TOL[dtype], s
    assert rel_err(f64(S), S_ref) <= TOL[dtype]
