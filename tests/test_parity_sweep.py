"""A seeded sweep of prefill calls that combine the options, each against the oracle.

Each case draws its own packed sequence lengths (empty, single-token, ragged and whole
chunks), head count, d_k / d_v, storage dtype, forget-rate granularity (one rate per head
or per key channel), rule (the gated delta rule or the decayed additive write), the layer
prologue (raw q, k and gate pre-activations), the output step and an initial state. The
combination picks the kernel path (exact fp32, tensor cores with one rate per head, or per
key channel), so every path meets options it is not tested with elsewhere. Tolerances as
for every path: max |gpu - oracle| / max |oracle| <= 1e-4 for fp32 inputs and <= 2e-2 for
bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_03_gb300 import ops
from tests.helpers import TOL, chunk_fwd, f64, rel_err

pytestmark = pytest.mark.gpu

SHAPES = [(64, 64), (128, 128), (128, 256), (64, 32), (128, 96)]
SHAPE_P = [0.1, 0.5, 0.2, 0.1, 0.1]  # (d = 128 reaches both tensor-core paths)


def draw_case(seed):
    rng = np.random.default_rng(7000 + seed)
    n = int(rng.integers(1, 5))
    lens = [int(x) for x in rng.choice([0, 1, 17, 63, 64, 65, 128, 200, 333], size=n)]
    if sum(lens) == 0:
        lens[0] = 70
    H = int(rng.integers(1, 4))
    dk, dv = SHAPES[int(rng.choice(len(SHAPES), p=SHAPE_P))]
    dtype = "bf16" if rng.random() < 0.7 else "f32"
    channel = bool(rng.random() < 0.5)
    additive = bool(rng.random() < 0.25)
    prologue = bool(rng.random() < 0.3)
    out_step = bool(rng.random() < 0.3)
    with_s0 = bool(rng.random() < 0.6)
    return dict(seed=seed, lens=lens, H=H, dk=dk, dv=dv, dtype=dtype, channel=channel,
                additive=additive, prologue=prologue, out_step=out_step, with_s0=with_s0,
                rng=rng)


@pytest.mark.parametrize("seed", range(48))
def test_random_option_combinations(seed):
    cs = draw_case(seed)
    rng, lens, H, dk, dv = cs["rng"], cs["lens"], cs["H"], cs["dk"], cs["dv"]
    T, n = sum(lens), len(lens)
    st = torch.bfloat16 if cs["dtype"] == "bf16" else torch.float32
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    if cs["prologue"]:  # raw projections: the kernels scale them
        q64, k64 = 2.0 * rng.standard_normal((T, H, dk)), 2.0 * rng.standard_normal((T, H, dk))
    else:
        q64, k64 = unit(rng.standard_normal((T, H, dk))), unit(rng.standard_normal((T, H, dk)))
    v64 = rng.standard_normal((T, H, dv))
    gshape = (T, H, dk) if cs["channel"] else (T, H)
    a64 = rng.standard_normal(gshape) - (3.0 if cs["prologue"] else 0.0)
    b64 = rng.standard_normal((T, H))
    A64 = rng.uniform(0.2, 2.0, H)
    to = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x).astype(np.float32)).to(dt)
    q, k, v = to(q64, st), to(k64, st), to(v64, st)
    if cs["prologue"]:
        la, beta, A = to(a64, torch.float32), to(b64, torch.float32), to(A64, torch.float32)
    else:
        la = to(-np.logaddexp(0.0, a64), torch.float32)
        beta = to(1.0 / (1.0 + np.exp(-b64)), torch.float32)
        A = None
    S0 = to(0.3 * rng.standard_normal((n, H, dk, dv)), torch.float32) if cs["with_s0"] else None
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    z = to(2.0 * rng.standard_normal((T, H, dv)), st) if cs["out_step"] else None
    w = to(rng.uniform(0.5, 1.5, dv), torch.float32) if cs["out_step"] else None

    c = lambda t: None if t is None else t.cuda()
    kw = dict(S0=c(S0), cu_seqlens=c(cu), rule="additive" if cs["additive"] else "delta")
    if cs["prologue"]:
        kw.update(prologue=True, gate_A=c(A))
    if cs["out_step"]:
        kw.update(out_gate=c(z), out_norm_weight=c(w), out_norm_eps=1e-5)
    o, S = chunk_fwd(c(q), c(k), c(v), c(la), c(beta), **kw)
    torch.cuda.synchronize()

    # the oracle on the same stored values
    qo, ko, lao, bo = f64(q), f64(k), f64(la), f64(beta)
    if cs["prologue"]:
        qo, ko, lao, bo = oracle.layer_prologue(qo, ko, lao, bo, f64(A))
    o_ref, S_ref = oracle.forward(qo, ko, f64(v), lao, bo,
                                  S0=None if S0 is None else f64(S0),
                                  cu_seqlens=cu.numpy().astype(np.int64),
                                  additive=cs["additive"])
    if cs["out_step"]:
        o_ref = oracle.out_norm_gate(o_ref, f64(z), f64(w), eps=1e-5)
    tol = TOL[cs["dtype"]]
    desc = {k_: v_ for k_, v_ in cs.items() if k_ != "rng"}
    desc["path"] = ops.chunk_fwd_path(dk, dv, st, "channel" if cs["channel"] else "head",
                                      prologue=cs["prologue"])
    assert np.isfinite(f64(o)).all() and np.isfinite(f64(S)).all(), desc
    assert rel_err(f64(o), o_ref) <= tol, (rel_err(f64(o), o_ref), desc)
    assert rel_err(f64(S), S_ref) <= tol, (rel_err(f64(S), S_ref), desc)
