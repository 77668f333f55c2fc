"""Seeded synthetic inputs for the gated delta rule workloads.

This module is shared by the CUDA path's callers (tests, benchmark) and by the
oracle's callers, and for that reason it holds none of the recurrence's
arithmetic: it only draws random numbers, shapes them, applies the layer
prologue the workloads specify (unit-length q and k, gate activations) and
rounds them to the storage type. Both sides then consume the identical values.

Recipe (one numpy PCG64 generator per workload, `numpy.random.default_rng(seed)`):
  * draw order: [sequence lengths], q, k, v, a, b, [S0]; decode draws S first and
    then q, k, v, a, b for every step;
  * q, k ~ N(0, 1), each token's per-head vector scaled to unit L2 norm in
    float64 (the unit-length queries and keys of "Linear attention"
    (arsalanzafar.ai), "A naive PyTorch implementation", F.normalize);
  * v ~ N(0, 1);
  * log alpha = -softplus(a), beta = sigmoid(b), a, b ~ N(0, 1), stored fp32
    (the gate parameterisation of the same section, with A = 1); with one rate per
    key channel a has one more axis of d_k entries, drawn in its place;
  * S0 ~ N(0, std^2) in fp32 when a workload asks for an initial state;
  * storage rounding: float64 -> float32 -> bf16 (round to nearest even, by torch).
Gate variants used by stress cases: "slow" gives log alpha = -softplus(a - 6)
(alpha about 0.9975), "none" gives log alpha = 0 (alpha = 1, the ungated
delta rule) and "strong" gives log alpha = -softplus(a + 1.5) (a chunk of 64
tokens decays by about e^-110).
"""
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

# The five workloads, with their sizes. `seed` is the generator seed.
WORKLOADS = {
    "tiny_fp32": dict(seed=0, num_seqs=1, seq_len=256, H=2, dk=64, dv=64, chunk=64,
                      dtype="f32", s0_std=0.0),
    "prefill_bf16": dict(seed=1, num_seqs=4, seq_len=4096, H=16, dk=128, dv=128, chunk=64,
                         dtype="bf16", s0_std=0.0),
    "varlen_bf16": dict(seed=2, num_seqs=8, len_range=(512, 8192), H=16, dk=128, dv=128,
                        chunk=64, dtype="bf16", s0_std=0.02),
    "decode_bf16": dict(seed=3, N=256, H=32, dk=128, dv=128, steps=16, dtype="bf16",
                        s0_std=0.02),
    "long_bf16": dict(seed=4, num_seqs=1, seq_len=65536, H=8, dk=128, dv=256, chunk=64,
                      dtype="bf16", s0_std=0.0),
}

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class PrefillInputs:
    q: torch.Tensor            # [total_T, H, dk], storage dtype
    k: torch.Tensor            # [total_T, H, dk]
    v: torch.Tensor            # [total_T, H, dv]
    log_alpha: torch.Tensor    # [total_T, H] fp32
    beta: torch.Tensor         # [total_T, H] fp32
    S0: Optional[torch.Tensor]  # [num_seqs, H, dk, dv] fp32 or None
    cu_seqlens: Optional[torch.Tensor]  # [num_seqs+1] int32 or None (equal lengths)
    num_seqs: int
    seq_lens: list
    H: int
    dk: int
    dv: int
    chunk: int
    dtype: str

    @property
    def total_tokens(self):
        return int(self.q.shape[0])


@dataclass
class DecodeInputs:
    S: torch.Tensor            # [N, H, dk, dv] fp32 initial state
    q: torch.Tensor            # [steps, N, H, dk]
    k: torch.Tensor            # [steps, N, H, dk]
    v: torch.Tensor            # [steps, N, H, dv]
    log_alpha: torch.Tensor    # [steps, N, H] fp32
    beta: torch.Tensor         # [steps, N, H] fp32
    N: int
    H: int
    dk: int
    dv: int
    steps: int
    dtype: str


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _store(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(TORCH_DTYPES[dtype])


def _gates(rng, shape, gate, channels=None):
    # channels: one forget rate per key channel, log alpha of shape shape + (channels,)
    a = rng.standard_normal(shape if channels is None else tuple(shape) + (channels,))
    b = rng.standard_normal(shape)
    if gate == "default":
        log_alpha = -np.logaddexp(0.0, a)
    elif gate == "slow":
        log_alpha = -np.logaddexp(0.0, a - 6.0)
    elif gate == "none":
        log_alpha = np.zeros(a.shape)
    elif gate == "strong":
        log_alpha = -np.logaddexp(0.0, a + 1.5)
    else:
        raise ValueError(f"unknown gate variant {gate!r}")
    beta = 1.0 / (1.0 + np.exp(-b))
    return (torch.from_numpy(log_alpha.astype(np.float32)),
            torch.from_numpy(beta.astype(np.float32)))


def prefill_inputs(seq_lens, H, dk, dv, dtype="bf16", seed=0, s0_std=0.0, chunk=64,
                   gate="default", rng=None, packed=None, decay="head"):
    """Packed inputs for sequences of the given lengths.

    `packed` chooses whether cu_seqlens is produced; by default it is when the
    lengths differ. Equal-length batches are passed without cu_seqlens. decay
    "channel" draws one forget rate per key channel (log_alpha [T, H, dk]).
    """
    rng = np.random.default_rng(seed) if rng is None else rng
    seq_lens = [int(x) for x in seq_lens]
    total = int(sum(seq_lens))
    q = _unit_rows(rng.standard_normal((total, H, dk)))
    k = _unit_rows(rng.standard_normal((total, H, dk)))
    v = rng.standard_normal((total, H, dv))
    log_alpha, beta = _gates(rng, (total, H), gate, dk if decay == "channel" else None)
    S0 = None
    if s0_std > 0:
        S0 = torch.from_numpy(
            (s0_std * rng.standard_normal((len(seq_lens), H, dk, dv))).astype(np.float32))
    if packed is None:
        packed = len(set(seq_lens)) > 1
    cu = None
    if packed:
        cu = torch.tensor(np.concatenate([[0], np.cumsum(seq_lens)]), dtype=torch.int32)
    return PrefillInputs(q=_store(q, dtype), k=_store(k, dtype), v=_store(v, dtype),
                         log_alpha=log_alpha, beta=beta, S0=S0, cu_seqlens=cu,
                         num_seqs=len(seq_lens), seq_lens=seq_lens, H=H, dk=dk, dv=dv,
                         chunk=chunk, dtype=dtype)


def workload_prefill(name, gate="default", decay="head"):
    """Inputs of one of the prefill workloads in WORKLOADS (decay "channel": the same
    shapes with one forget rate per key channel)."""
    w = WORKLOADS[name]
    rng = np.random.default_rng(w["seed"])
    if "len_range" in w:
        lo, hi = w["len_range"]
        seq_lens = rng.integers(lo, hi + 1, size=w["num_seqs"]).tolist()
    else:
        seq_lens = [w["seq_len"]] * w["num_seqs"]
    return prefill_inputs(seq_lens, w["H"], w["dk"], w["dv"], dtype=w["dtype"],
                          s0_std=w["s0_std"], chunk=w["chunk"], gate=gate, rng=rng, decay=decay)


def decode_inputs(N, H, dk, dv, steps, dtype="bf16", seed=3, s0_std=0.02, gate="default",
                  decay="head"):
    """State plus per-step inputs for `steps` consecutive decode steps."""
    rng = np.random.default_rng(seed)
    S = torch.from_numpy((s0_std * rng.standard_normal((N, H, dk, dv))).astype(np.float32))
    qs, ks, vs, las, bs = [], [], [], [], []
    for _ in range(steps):
        qs.append(_store(_unit_rows(rng.standard_normal((N, H, dk))), dtype))
        ks.append(_store(_unit_rows(rng.standard_normal((N, H, dk))), dtype))
        vs.append(_store(rng.standard_normal((N, H, dv)), dtype))
        la, b = _gates(rng, (N, H), gate, dk if decay == "channel" else None)
        las.append(la)
        bs.append(b)
    return DecodeInputs(S=S, q=torch.stack(qs), k=torch.stack(ks), v=torch.stack(vs),
                        log_alpha=torch.stack(las), beta=torch.stack(bs), N=N, H=H, dk=dk,
                        dv=dv, steps=steps, dtype=dtype)


def workload_decode(name="decode_bf16", steps=None, gate="default", decay="head"):
    w = WORKLOADS[name]
    return decode_inputs(w["N"], w["H"], w["dk"], w["dv"], steps or w["steps"],
                         dtype=w["dtype"], seed=w["seed"], s0_std=w["s0_std"], gate=gate,
                         decay=decay)
