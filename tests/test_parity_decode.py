"""GPU parity of gdr_decode_step against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_03_gb300 import inputs
from tests.helpers import TOL, chunk_fwd, decode_step, f64, rel_err

pytestmark = pytest.mark.gpu


def run_steps(d, steps=None):
    steps = d.steps if steps is None else steps
    S = d.S.cuda()
    outs = []
    for s in range(steps):
        outs.append(decode_step(d.q[s].cuda(), d.k[s].cuda(), d.v[s].cuda(),
                                d.log_alpha[s].cuda(), d.beta[s].cuda(), S))
    torch.cuda.synchronize()
    return [f64(o) for o in outs], f64(S)


def oracle_steps(d, steps=None, seqs=None):
    steps = d.steps if steps is None else steps
    sel = slice(None) if seqs is None else slice(0, seqs)
    S = f64(d.S)[sel]
    outs = []
    for s in range(steps):
        o, S = oracle.decode(f64(d.q[s])[sel], f64(d.k[s])[sel], f64(d.v[s])[sel],
                             f64(d.log_alpha[s])[sel], f64(d.beta[s])[sel], S)
        outs.append(o)
    return outs, S


def test_decode_workload_16_steps():
    d = inputs.workload_decode()
    outs, S = run_steps(d)
    ref_outs, S_ref = oracle_steps(d)
    for s in range(d.steps):
        assert rel_err(outs[s], ref_outs[s]) <= TOL["bf16"], s
    assert rel_err(S, S_ref) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (64, 256), (128, 64), (128, 128),
                                   (128, 256)])
def test_decode_shapes(dtype, dk, dv):
    d = inputs.decode_inputs(N=5, H=3, dk=dk, dv=dv, steps=4, dtype=dtype, seed=dk * dv,
                             s0_std=0.5)
    outs, S = run_steps(d)
    ref_outs, S_ref = oracle_steps(d)
    for s in range(d.steps):
        assert rel_err(outs[s], ref_outs[s]) <= TOL[dtype], s
    assert rel_err(S, S_ref) <= TOL[dtype]


def test_prefill_then_decode_equals_longer_prefill():
    full = inputs.prefill_inputs([150], H=2, dk=128, dv=128, dtype="bf16", seed=13, s0_std=0.2,
                                 gate="slow")
    dev = lambda t: t.cuda()
    q, k, v, la, b = (dev(full.q), dev(full.k), dev(full.v), dev(full.log_alpha),
                      dev(full.beta))
    tau = 140
    _, S = chunk_fwd(q[:tau].contiguous(), k[:tau].contiguous(), v[:tau].contiguous(),
                     la[:tau].contiguous(), b[:tau].contiguous(), S0=dev(full.S0))
    outs = []
    for t in range(tau, 150):
        outs.append(decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1], b[t:t + 1], S))
    o_all, S_all = chunk_fwd(q, k, v, la, b, S0=dev(full.S0))
    torch.cuda.synchronize()
    assert rel_err(f64(torch.cat(outs)), f64(o_all[tau:])) <= 2e-2
    assert rel_err(f64(S), f64(S_all)) <= 2e-2


def test_decode_zero_sequences_is_a_no_op():
    S = torch.zeros((0, 2, 64, 64), device="cuda")
    q = torch.zeros((0, 2, 64), device="cuda")
    o = decode_step(q, q, q, torch.zeros((0, 2), device="cuda"),
                    torch.zeros((0, 2), device="cuda"), S)
    assert o.shape == (0, 2, 64)
