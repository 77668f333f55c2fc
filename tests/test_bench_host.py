"""Host-side pieces of bench.py and of the input generator, on CPU: the algorithmic byte
counts the roofline divides by, the workload description, the argument checks, and the
shapes of the per-channel gates."""
import pytest
import torch

import bench
from gated_delta_rule_03_gb300 import inputs


def test_prefill_bytes_head_and_channel_rates():
    inp = inputs.prefill_inputs([100, 28], H=3, dk=64, dv=32, dtype="bf16", seed=1)
    th = inp.total_tokens * inp.H
    state = inp.num_seqs * inp.H * 64 * 32 * 4
    # q, k (d_k each), v, o (d_v each) in bf16; one log alpha and one beta per token-head
    assert bench.prefill_bytes(inp) == th * (2 * 64 + 2 * 32) * 2 + th * 8 + state
    pc = inputs.prefill_inputs([100, 28], H=3, dk=64, dv=32, dtype="bf16", seed=1,
                               decay="channel", s0_std=0.1)
    # d_k fp32 rates per token-head; S0 read as well as S written
    assert bench.prefill_bytes(pc) == th * (2 * 64 + 2 * 32) * 2 + th * (64 + 1) * 4 + 2 * state


def test_workload_config_names_the_workload():
    cfg = bench.workload_config(inputs.prefill_inputs([64] * 2, H=2, dk=64, dv=64, seed=3),
                                "prefill_bf16")
    assert cfg["workload"].startswith("prefill_bf16: B=2 H=2 T=64")
    assert cfg["seq_len"] == 64 and cfg["global_batch"] == 2
    var = bench.workload_config(inputs.prefill_inputs([64, 100], H=2, dk=64, dv=64, seed=3,
                                                      decay="channel"), "varlen_bf16")
    assert "one forget rate per key channel" in var["workload"]
    assert "T in 64..100 packed (164 tokens)" in var["workload"] and var["seq_len"] == 82


def test_arguments_are_checked():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
    with pytest.raises(SystemExit):
        bench.main(["--workload", "tiny_fp32"])
    with pytest.raises(SystemExit):
        bench.main(["--decay", "row"])


@pytest.mark.parametrize("gate", ["default", "slow", "none", "strong"])
def test_per_channel_gates(gate):
    inp = inputs.prefill_inputs([70, 3], H=2, dk=16, dv=8, seed=5, gate=gate, decay="channel")
    assert tuple(inp.log_alpha.shape) == (73, 2, 16) and tuple(inp.beta.shape) == (73, 2)
    assert inp.log_alpha.dtype == torch.float32 and bool((inp.log_alpha <= 0).all())
    if gate == "none":
        assert bool((inp.log_alpha == 0).all())
    else:  # the channels differ
        assert float(inp.log_alpha.std(dim=-1).min()) > 0
    d = inputs.decode_inputs(N=3, H=2, dk=16, dv=8, steps=2, seed=5, gate=gate, decay="channel")
    assert tuple(d.log_alpha.shape) == (2, 3, 2, 16)


def test_head_rate_draws_are_unchanged_by_the_option():
    a = inputs.prefill_inputs([50], H=2, dk=8, dv=8, seed=9)
    b = inputs.prefill_inputs([50], H=2, dk=8, dv=8, seed=9, decay="head")
    assert torch.equal(a.log_alpha, b.log_alpha) and torch.equal(a.q, b.q)


def test_prefill_flops_is_the_chunk_count():
    inp = inputs.prefill_inputs([4096] * 4, H=16, dk=128, dv=128, dtype="bf16", seed=1)
    # 155,648 flops per token-head at d = 128, C = 64
    assert bench.prefill_flops(inp) == 4 * 4096 * 16 * 155648


def test_decode_cpu_baseline_sample():
    dec = inputs.decode_inputs(N=4, H=2, dk=16, dv=8, steps=3, seed=7)
    out = bench.cpu_decode_baseline(dec, 0.05, seqs=2)
    assert out["kind"] == "oracle" and out["value"] > 0 and out["cores"] >= 1
    assert out["sample"].startswith("2 of 4 sequences x 2 heads")


def test_cpu_baseline_compares_the_given_outputs_with_the_oracle():
    import numpy as np
    import oracle
    inp = inputs.prefill_inputs([70, 30], H=3, dk=16, dv=8, dtype="f32", seed=5, s0_std=0.1)
    full = oracle.forward(**bench.oracle_prefill_sample(inp))
    sel = [0, 2]
    o, S = full[0][:, sel], full[1][:, sel]
    out = bench.cpu_baseline(inp, 0.0, "small", heads=sel, gpu_out=(o, S))
    assert out["parity"]["o_rel_err"] < 1e-12 and out["parity"]["S_rel_err"] < 1e-12
    assert out["parity"]["tolerance"] == 1e-4 and out["parity"]["heads"] == sel
    bad = o.copy()
    bad[5, 1, 3] += 0.5 * np.abs(o).max()  # one wrong element of head 2
    out = bench.cpu_baseline(inp, 0.0, "small", heads=sel, gpu_out=(bad, S))
    assert out["parity"]["o_rel_err"] == pytest.approx(0.5, rel=1e-9)
