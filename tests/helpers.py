"""Shared helpers for the parity tests: run both sides on the same inputs, compare."""
import numpy as np
import torch

import oracle


def f64(t):
    """Exact float64 copy of a CPU or GPU tensor (bf16 and fp32 widen exactly)."""
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(got, want):
    """max |got - want| / max |want| (0 when both are zero)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    denom = np.abs(want).max() if want.size else 0.0
    diff = np.abs(got - want).max() if want.size else 0.0
    if denom == 0.0:
        return float(diff)
    return float(diff / denom)


TOL = {"f32": 1e-4, "bf16": 2e-2}


def oracle_prefill(inp, heads=None):
    """Oracle result for a PrefillInputs (optionally only the given heads)."""
    sel = slice(None) if heads is None else list(heads)
    q, k, v = f64(inp.q)[:, sel], f64(inp.k)[:, sel], f64(inp.v)[:, sel]
    la, b = f64(inp.log_alpha)[:, sel], f64(inp.beta)[:, sel]
    S0 = None if inp.S0 is None else f64(inp.S0)[:, sel]
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy().astype(np.int64)
    return oracle.forward(q, k, v, la, b, S0=S0, cu_seqlens=cu, num_seqs=inp.num_seqs)


def gpu_prefill(inp, device="cuda"):
    from gated_delta_rule_03_gb300 import chunk_fwd
    d = lambda t: None if t is None else t.to(device)
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), S0=d(inp.S0),
                     cu_seqlens=d(inp.cu_seqlens), num_seqs=inp.num_seqs, chunk=inp.chunk)
    torch.cuda.synchronize()
    return o, S
