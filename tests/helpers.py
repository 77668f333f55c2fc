"""Shared helpers for the parity tests: run both sides on the same inputs, compare.

`chunk_fwd` and `decode_step` here wrap the binding's calls of the same names for the GPU
tests. Every output the caller does not pass in is allocated NaN-filled, inside a larger
NaN-filled buffer with a guard band of at least one leading-dimension row before and after
it. After the call the guard bands must still be NaN: an element the kernels forget to
write stays NaN and fails the comparison with the oracle, and a write outside the output
fails the guard check. A state updated in place (decode) is copied into such a buffer for
the call and copied back.
"""
import math

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


def _guard_elems(shape):
    """Guard band length: one row of the leading dimension, at least 256 elements, rounded
    up to 64 elements so that the tensor inside keeps 128-byte alignment."""
    row = math.prod(shape[1:]) if len(shape) > 1 else 1
    return (max(row, 256) + 63) // 64 * 64


def poisoned(shape, dtype, device, fill=None):
    """(tensor, guard) -- a NaN-filled tensor of `shape` (or a copy of `fill`) inside a
    NaN-filled buffer with a guard band before and after it."""
    n, g = math.prod(shape), _guard_elems(shape)
    buf = torch.full((g + n + g,), float("nan"), dtype=dtype, device=device)
    t = buf[g:g + n].view(shape)
    if fill is not None:
        t.copy_(fill)
    return t, (buf, g, n)


def check_guards(guards):
    """Every guard band is still all NaN (synchronises the device)."""
    if not guards:
        return
    torch.cuda.synchronize()
    for buf, g, n in guards:
        head, tail = buf[:g], buf[g + n:]
        assert bool(torch.isnan(head).all()), "a kernel wrote before the start of an output"
        assert bool(torch.isnan(tail).all()), "a kernel wrote past the end of an output"


def chunk_fwd(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, num_seqs=None, o=None,
              S_final=None, **kw):
    """ops.chunk_fwd with NaN-poisoned, guard-banded o and S_final (when not passed in)."""
    from gated_delta_rule_03_gb300 import ops
    T, H, dk = q.shape
    dv = v.shape[-1]
    n = cu_seqlens.numel() - 1 if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    guards = []
    if o is None:
        o, g = poisoned((T, H, dv), q.dtype, q.device)
        guards.append(g)
    if S_final is None:
        S_final, g = poisoned((n, H, dk, dv), torch.float32, q.device)
        guards.append(g)
    out = ops.chunk_fwd(q, k, v, log_alpha, beta, S0=S0, cu_seqlens=cu_seqlens, num_seqs=num_seqs,
                        o=o, S_final=S_final, **kw)
    check_guards(guards)
    return out


def decode_step(q, k, v, log_alpha, beta, S, o=None, **kw):
    """ops.decode_step with a NaN-poisoned, guard-banded o (when not passed in) and the
    state updated inside a guard-banded copy."""
    from gated_delta_rule_03_gb300 import ops
    N, H, dk = q.shape
    dv = v.shape[-1]
    guards = []
    if o is None:
        o, g = poisoned((N, H, dv), q.dtype, q.device)
        guards.append(g)
    Sg, g = poisoned(tuple(S.shape), S.dtype, S.device, fill=S)
    guards.append(g)
    ops.decode_step(q, k, v, log_alpha, beta, Sg, o=o, **kw)
    S.copy_(Sg)
    check_guards(guards)
    return o


def gpu_prefill(inp, device="cuda"):
    d = lambda t: None if t is None else t.to(device)
    o, S = chunk_fwd(d(inp.q), d(inp.k), d(inp.v), d(inp.log_alpha), d(inp.beta), S0=d(inp.S0),
                     cu_seqlens=d(inp.cu_seqlens), num_seqs=inp.num_seqs, chunk=inp.chunk)
    torch.cuda.synchronize()
    return o, S
