"""Float64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline / reference legs
of `bench.py` may import this package. The product path (the CUDA library in
`gated_delta_rule_03_gb300` and its binding) never imports it; the two share no
code. The arithmetic lives in `gdr_oracle.c` (the token-by-token recurrence of
"Linear attention" (arsalanzafar.ai), "How it works", Eqs. (1)-(4), keys x
values layout, update before read); this module only marshals numpy arrays.

Every array is converted to contiguous float64 before the call, so callers can
pass the exact values the GPU receives (bf16 or fp32, widened exactly).
"""
import ctypes
import os

import numpy as np

from .build import ensure_built

_lib = None


def _load():
    global _lib
    if _lib is None:
        # GDR_ORACLE_LIB points the wrapper at another build of the same source; the
        # mutation tests use it to check that the pins catch planted mistakes.
        path = os.environ.get("GDR_ORACLE_LIB") or ensure_built()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.gdr_oracle_forward.argtypes = [dp, dp, dp, dp, dp, dp, lp, i64, i64, i64, i64, i64,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp]
        lib.gdr_oracle_forward.restype = ctypes.c_int
        lib.gdr_oracle_decode.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                          ctypes.c_int, ctypes.c_int]
        lib.gdr_oracle_decode.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads():
    """Host threads the oracle uses by default: the cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def forward(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, num_seqs=None,
            additive=False, threads=None):
    """Run the recurrence over packed sequences.

    q, k: [total_T, H, dk]; v: [total_T, H, dv]; beta: [total_T, H]; log_alpha:
    [total_T, H] (one rate per head), or [total_T, H, dk] (one rate per key channel);
    S0: [num_seqs, H, dk, dv] or None (zero state); cu_seqlens: [num_seqs+1]
    token offsets or None (then `num_seqs` equal sequences, default 1).
    Returns (o [total_T, H, dv], S_final [num_seqs, H, dk, dv]) in float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, b = _f64(log_alpha), _f64(beta)
    T, H, dk = q.shape
    dv = v.shape[2]
    assert k.shape == (T, H, dk) and v.shape[:2] == (T, H)
    per_channel = la.ndim == 3
    assert la.shape == ((T, H, dk) if per_channel else (T, H)) and b.shape == (T, H)
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        n = len(cu) - 1
    else:
        n = 1 if num_seqs is None else int(num_seqs)
    s0 = None if S0 is None else _f64(S0)
    if s0 is not None:
        assert s0.shape == (n, H, dk, dv)
    o = np.zeros((T, H, dv), dtype=np.float64)
    S = np.zeros((n, H, dk, dv), dtype=np.float64)
    rc = _load().gdr_oracle_forward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(s0), _ptr(cu, ctypes.c_int64),
        n, T, H, dk, dv, int(bool(additive)), int(per_channel), int(threads or default_threads()),
        _ptr(o), _ptr(S))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (status {rc})")
    return o, S


def decode(q, k, v, log_alpha, beta, S, threads=None):
    """One decode step for N sequences: q, k [N, H, dk]; v [N, H, dv];
    log_alpha [N, H] (or [N, H, dk], one rate per key channel), beta [N, H];
    S [N, H, dk, dv]. Returns (o, S_new) in float64; the input S is not modified."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, b = _f64(log_alpha), _f64(beta)
    S_new = np.array(S, dtype=np.float64, copy=True, order="C")
    N, H, dk = q.shape
    dv = v.shape[2]
    o = np.zeros((N, H, dv), dtype=np.float64)
    per_channel = la.ndim == 3
    assert la.shape == ((N, H, dk) if per_channel else (N, H))
    rc = _load().gdr_oracle_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(S_new),
                                   _ptr(o), N, H, dk, dv, int(per_channel),
                                   int(threads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (status {rc})")
    return o, S_new


def out_norm_gate(o, gate, weight=None, eps=1e-6):
    """The layer's output step after the recurrence, in float64 ("Linear attention"
    (arsalanzafar.ai), "A naive PyTorch implementation": the output is normalised over
    the head dimension, then multiplied by SiLU of the input-dependent output gate):

        o'_tj = o_tj / sqrt(mean_j' o_tj'^2 + eps) * weight_j * gate_tj * sigmoid(gate_tj)

    per token and head; o and gate [..., d_v], weight [d_v] (None: ones). The mean runs
    over the last axis (the head's value entries). Written out with numpy, elementwise."""
    o = _f64(o)
    g = _f64(gate)
    w = np.ones(o.shape[-1]) if weight is None else _f64(weight)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o / rms * w * (g / (1.0 + np.exp(-g)))


def layer_prologue(q, k, a, b, A=None):
    """The layer's steps before the recurrence, in float64 ("Linear attention"
    (arsalanzafar.ai), "A naive PyTorch implementation"): each token's query and key
    vector per head scaled to unit length (x / max(|x|, 1e-12), as F.normalize), and the
    gates from their pre-activations,

        log alpha = -A_h softplus(a),    beta = sigmoid(b),

    q, k [..., H, d_k]; b [..., H]; a [..., H], or [..., H, d_k] for one rate per key
    channel; A [H] (None: ones). Returns (q, k, log_alpha, beta) for forward() / decode()."""
    q, k, a, b = _f64(q), _f64(k), _f64(a), _f64(b)
    per_channel = a.ndim == q.ndim
    H = a.shape[-2] if per_channel else a.shape[-1]
    A = np.ones(H) if A is None else _f64(A)
    if per_channel:
        A = A[:, None]
    qn = q / np.maximum(np.linalg.norm(q, axis=-1, keepdims=True), 1e-12)
    kn = k / np.maximum(np.linalg.norm(k, axis=-1, keepdims=True), 1e-12)
    softplus = np.logaddexp(0.0, a)
    return qn, kn, -A * softplus, 1.0 / (1.0 + np.exp(-b))
