"""A seeded sweep of decode steps that combine the options, each against the oracle.

Each case draws N sequences, heads, d_k / d_v, storage dtype, forget-rate granularity,
rule, the layer prologue and the output step, then runs three consecutive steps on one
state. The reference for a step is the oracle's prefill over N one-token sequences from the
same state (a decode step is that prefill), which covers every rule. Tolerances as for
every path: max |gpu - oracle| / max |oracle| <= 1e-4 for fp32 inputs and <= 2e-2 for
bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import TOL, decode_step, f64, rel_err

pytestmark = pytest.mark.gpu

SHAPES = [(64, 64), (128, 128), (128, 256), (64, 256), (128, 64), (64, 128)]  # d_v in {64, 128, 256}


@pytest.mark.parametrize("seed", range(24))
def test_random_decode_option_combinations(seed):
    rng = np.random.default_rng(8000 + seed)
    N, H = int(rng.integers(1, 41)), int(rng.integers(1, 5))
    dk, dv = SHAPES[int(rng.integers(0, len(SHAPES)))]
    bf16 = bool(rng.random() < 0.7)
    channel, additive = bool(rng.random() < 0.5), bool(rng.random() < 0.25)
    prologue, out_step = bool(rng.random() < 0.3), bool(rng.random() < 0.3)
    st = torch.bfloat16 if bf16 else torch.float32
    to = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x).astype(np.float32)).to(dt)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    S = to(0.3 * rng.standard_normal((N, H, dk, dv)), torch.float32)
    S_ref = f64(S)
    Sg = S.cuda()
    A = to(rng.uniform(0.2, 2.0, H), torch.float32)
    w = to(rng.uniform(0.5, 1.5, dv), torch.float32)
    cu = np.arange(N + 1, dtype=np.int64)
    for step in range(3):
        q64 = rng.standard_normal((N, H, dk))
        k64 = rng.standard_normal((N, H, dk))
        if not prologue:
            q64, k64 = unit(q64), unit(k64)
        q, k, v = to(q64, st), to(k64, st), to(rng.standard_normal((N, H, dv)), st)
        a64 = rng.standard_normal((N, H, dk) if channel else (N, H))
        b64 = rng.standard_normal((N, H))
        if prologue:
            la, beta = to(a64, torch.float32), to(b64, torch.float32)
        else:
            la = to(-np.logaddexp(0.0, a64), torch.float32)
            beta = to(1.0 / (1.0 + np.exp(-b64)), torch.float32)
        z = to(2.0 * rng.standard_normal((N, H, dv)), st)
        kw = dict(rule="additive" if additive else "delta")
        if prologue:
            kw.update(prologue=True, gate_A=A.cuda())
        if out_step:
            kw.update(out_gate=z.cuda(), out_norm_weight=w.cuda(), out_norm_eps=1e-5)
        c = lambda t: t.cuda()
        o = decode_step(c(q), c(k), c(v), c(la), c(beta), Sg, **kw)
        torch.cuda.synchronize()
        qo, ko, lao, bo = f64(q), f64(k), f64(la), f64(beta)
        if prologue:
            qo, ko, lao, bo = oracle.layer_prologue(qo, ko, lao, bo, f64(A))
        o_ref, S_ref = oracle.forward(qo, ko, f64(v), lao, bo, S0=S_ref, cu_seqlens=cu,
                                      additive=additive)
        if out_step:
            o_ref = oracle.out_norm_gate(o_ref, f64(z), f64(w), eps=1e-5)
        tol = TOL["bf16" if bf16 else "f32"]
        desc = dict(seed=seed, N=N, H=H, dk=dk, dv=dv, bf16=bf16, channel=channel,
                    additive=additive, prologue=prologue, out_step=out_step, step=step)
        assert rel_err(f64(o), o_ref) <= tol, (rel_err(f64(o), o_ref), desc)
    assert rel_err(f64(Sg), S_ref) <= tol, (rel_err(f64(Sg), S_ref), desc)
