"""Pins for the float64 oracle: the pages' printed values, closed forms and brute force.

The oracle (oracle/gdr_oracle.c) is the token recurrence of "Linear attention"
(arsalanzafar.ai), "How it works", Eqs. (1)-(4). None of these tests re-types
that loop: each checks it against something fixed independently -- a worked
example or table printed on a page (tests/golden/*.json, each with its
citation), a closed form, an identity, or the unrolled product of transitions.
"""
import json
import os

import numpy as np
import pytest

import oracle
from tests import chunk_form

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def run(q, k, v, alpha=None, beta=None, S0=None, log_alpha=None, additive=False):
    """Single head, single sequence: q, k [T, dk], v [T, dv] -> (o [T, dv], S [dk, dv])."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    T = len(k)
    if log_alpha is None:
        log_alpha = np.log(np.broadcast_to(np.asarray(1.0 if alpha is None else alpha,
                                                      dtype=np.float64), (T,)))
    log_alpha = np.broadcast_to(np.asarray(log_alpha, dtype=np.float64), (T,))
    beta = np.broadcast_to(np.asarray(1.0 if beta is None else beta, dtype=np.float64), (T,))
    s0 = None if S0 is None else np.asarray(S0, dtype=np.float64)[None, None]
    o, S = oracle.forward(q[:, None, :], k[:, None, :], v[:, None, :], log_alpha[:, None],
                          beta[:, None], S0=s0, additive=additive, threads=1)
    return o[:, 0, :], S[0, 0]


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


# --------------------------------------------------------------------------- pages' examples

def test_p1_worked_example():
    g = golden("p1_worked_example.json")
    S_old = np.array(g["S_old"], dtype=float).T          # keys x values
    q, k, v = (np.array(g[x], dtype=float) for x in ("q", "k", "v"))
    alpha, beta = g["alpha"], g["beta"]
    # beta = 0 leaves only the decay: the decayed memory, and reading it with k is the prediction
    _, decayed = run([q], [k], [v], alpha=alpha, beta=0.0, S0=S_old)
    np.testing.assert_array_equal(decayed.T, np.array(g["decayed"], dtype=float))
    pred, _ = run([k], [k], [v], alpha=alpha, beta=0.0, S0=S_old)
    np.testing.assert_array_equal(pred[0], g["prediction"])
    np.testing.assert_array_equal(v - pred[0], g["error"])
    # the full step
    y, S_new = run([q], [k], [v], alpha=alpha, beta=beta, S0=S_old)
    np.testing.assert_allclose(S_new.T, g["S_new"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(y[0], g["y"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(S_new.T @ k, g["read_with_k"], rtol=0, atol=1e-15)
    ortho = g["read_with_orthogonal_key"]
    np.testing.assert_allclose(S_new.T @ np.array(ortho["key"], dtype=float), ortho["value"],
                               rtol=0, atol=1e-15)


def test_p1_memory_built_from_two_writes_then_worked_step():
    g = golden("p1_reading_and_writing.json")
    e1 = golden("p1_worked_example.json")
    w1, w2 = g["writes"]
    q = np.array(g["q"], dtype=float)
    ks = [w1["k"], w2["k"], e1["k"]]
    vs = [w1["v"], w2["v"], e1["v"]]
    # first write alone from a zero state: the outer product v k^T
    _, S1 = run([q], [w1["k"]], [w1["v"]])
    np.testing.assert_array_equal(S1.T, np.array(w1["outer_v_kT"], dtype=float))
    # two writes with alpha = beta = 1 build the memory that the query reads
    o2, S2 = run([q, q], ks[:2], vs[:2])
    np.testing.assert_array_equal(S2.T, np.array(g["S_after_both_writes"], dtype=float))
    np.testing.assert_allclose(o2[1], g["y"], rtol=0, atol=1e-15)
    # then the worked step (alpha = 0.5, beta = 1) on top
    o3, S3 = run([q, q, q], ks, vs, log_alpha=[0.0, 0.0, np.log(e1["alpha"])])
    np.testing.assert_allclose(o3[2], e1["y"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(S3.T, e1["S_new"], rtol=0, atol=1e-15)


def test_p5_figure6_delta_rule_overwrites():
    g = golden("p5_figure6.json")
    K, V = np.array(g["keys"], dtype=float), np.array(g["values"], dtype=float)
    _, S2 = run(K[:2], K[:2], V[:2])
    _, S3 = run(K, K, V)
    np.testing.assert_array_equal(S3, g["delta_S_3"])
    _, S3_add = run(K, K, V, additive=True)
    np.testing.assert_array_equal(S3_add, g["additive_S_3"])
    # S_3 - S_2 = k_3 u_3^T, and k_3 has unit length
    np.testing.assert_array_equal((S3 - S2).T @ K[2], g["pseudo_value_u_3"])


def test_p5_figure5_additive_crosstalk():
    g = golden("p5_figure5.json")
    K, V = np.array(g["keys"], dtype=float), np.array(g["values"], dtype=float)
    _, S2 = run(K[:2], K[:2], V[:2], additive=True)
    _, S3 = run(K, K, V, additive=True)
    np.testing.assert_array_equal(S2, g["S_2"])
    np.testing.assert_array_equal(S3, g["S_3"])
    reads = K @ S3 / (K ** 2).sum(axis=1, keepdims=True)
    np.testing.assert_array_equal(reads - V, g["crosstalk_after_third_write"])


def test_p5_table1_read_errors():
    g = golden("p5_table1.json")
    half_ulp = 0.5 * 10.0 ** (-g["printed_decimals"]) + 1e-12
    for row in g["rows"]:
        n, r = row["n"], 32
        rng = np.random.default_rng(2)
        sq_all, sq_new, sq_add = [], [], []
        for _ in range(200):
            K = unit(rng.standard_normal((n, r)))
            V = unit(rng.standard_normal((n, r)))
            _, S = run(K, K, V, alpha=1.0, beta=1.0)
            _, S_add = run(K, K, V, alpha=1.0, beta=1.0, additive=True)
            err = ((K @ S - V) ** 2).sum(axis=1)
            sq_all.append(err.mean())
            sq_new.append(err[-8:].mean())
            sq_add.append(((K @ S_add - V) ** 2).sum(axis=1).mean())
        assert abs(np.sqrt(np.mean(sq_all)) - row["delta_all"]) <= half_ulp, row
        assert abs(np.sqrt(np.mean(sq_new)) - row["delta_newest8"]) <= half_ulp, row
        assert abs(np.sqrt(np.mean(sq_add)) - row["additive"]) <= half_ulp, row


def test_p5_kaczmarz_sweeps_converge():
    g = golden("p5_kaczmarz.json")
    rng = np.random.default_rng(4)
    K = unit(rng.standard_normal((24, 32)))
    V = unit(rng.standard_normal((24, 32)))
    Kr, Vr = np.tile(K, (200, 1)), np.tile(V, (200, 1))
    _, S = run(Kr, Kr, Vr, alpha=1.0, beta=1.0)
    err = np.abs(K @ S - V).max()
    assert err < g["tolerance"]
    assert float(f"{err:.1e}") == g["printed_largest_error"]


# --------------------------------------------------------------------------- closed forms

def _random_case(rng, T, dk, dv, unit_keys=True):
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk))
    if unit_keys:
        k = unit(k)
    v = rng.standard_normal((T, dv))
    la = -np.logaddexp(0.0, rng.standard_normal(T))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    S0 = rng.standard_normal((dk, dv))
    return q, k, v, la, b, S0


def test_alpha_one_beta_zero_leaves_state_unchanged():
    rng = np.random.default_rng(10)
    q, k, v, _, _, S0 = _random_case(rng, 20, 6, 5)
    o, S = run(q, k, v, alpha=1.0, beta=0.0, S0=S0)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o, q @ S0, rtol=0, atol=1e-13)


def test_beta_zero_is_pure_decay():
    rng = np.random.default_rng(11)
    q, k, v, la, _, S0 = _random_case(rng, 15, 4, 7)
    o, S = run(q, k, v, log_alpha=la, beta=0.0, S0=S0)
    decay = np.exp(np.cumsum(la))
    np.testing.assert_allclose(S, decay[-1] * S0, rtol=1e-13, atol=0)
    np.testing.assert_allclose(o, decay[:, None] * (q @ S0), rtol=1e-12, atol=1e-15)


def test_beta_one_unit_key_reads_back_its_value_exactly():
    # keys with entries +-1/2 in four dimensions have exactly unit length in binary
    rng = np.random.default_rng(12)
    T, dk, dv = 12, 4, 3
    k = 0.5 * rng.choice([-1.0, 1.0], size=(T, dk))
    v = rng.integers(-8, 9, size=(T, dv)).astype(float)
    S = rng.integers(-4, 5, size=(dk, dv)).astype(float)
    for t in range(T):
        _, S = run([k[t]], [k[t]], [v[t]], alpha=0.5, beta=1.0, S0=S)
        np.testing.assert_array_equal(S.T @ k[t], v[t])


def test_read_back_mixes_old_read_and_new_value():
    # "How linear attention works", section "Correct the association at this key":
    # for a unit key, S_t^T k = (1 - beta) alpha S_{t-1}^T k + beta v.
    rng = np.random.default_rng(7)
    dk, dv = 8, 8
    for beta in (0.0, 0.3, 0.7, 1.0):
        S0 = rng.standard_normal((dk, dv))
        k = unit(rng.standard_normal(dk))
        v = rng.standard_normal(dv)
        alpha = 0.8
        _, S1 = run([k], [k], [v], alpha=alpha, beta=beta, S0=S0)
        np.testing.assert_allclose(S1.T @ k, (1 - beta) * alpha * (S0.T @ k) + beta * v,
                                   rtol=0, atol=1e-13)


def test_factored_householder_form_equals_the_recurrence():
    # "How linear attention works", section "A runnable check": the factored form
    # alpha (I - beta k k^T) S + beta k v^T (keys x values) equals decay-predict-correct,
    # here also for non-unit keys.
    rng = np.random.default_rng(13)
    dk, dv = 6, 5
    for unit_keys in (True, False):
        S = rng.standard_normal((dk, dv))
        k = rng.standard_normal(dk)
        if unit_keys:
            k = unit(k)
        v, q = rng.standard_normal(dv), rng.standard_normal(dk)
        alpha, beta = 0.6, 0.45
        factored = alpha * (np.eye(dk) - beta * np.outer(k, k)) @ S + beta * np.outer(k, v)
        o, S1 = run([q], [k], [v], alpha=alpha, beta=beta, S0=S)
        np.testing.assert_allclose(S1, factored, rtol=0, atol=1e-13)
        np.testing.assert_allclose(o[0], factored.T @ q, rtol=0, atol=1e-13)


def test_additive_rule_without_decay_is_one_matmul():
    rng = np.random.default_rng(14)
    T, dk, dv = 33, 5, 7
    K, V, Q = rng.standard_normal((T, dk)), rng.standard_normal((T, dv)), rng.standard_normal((T, dk))
    o, S = run(Q, K, V, alpha=1.0, beta=1.0, additive=True)
    np.testing.assert_allclose(S, K.T @ V, rtol=0, atol=1e-12)
    # every read is the masked product: o_t = sum_{j<=t} (q_t . k_j) v_j
    np.testing.assert_allclose(o, np.tril(Q @ K.T) @ V, rtol=0, atol=1e-12)
    # with a write strength: one gradient step of size beta_t on the dot-product loss per
    # token ("From KV Cache to a State Matrix", section "Associating keys and values"),
    # so S = K^T diag(beta) V
    beta = rng.uniform(0.1, 0.9, size=T)
    o, S = run(Q, K, V, alpha=1.0, beta=beta, additive=True)
    np.testing.assert_allclose(S, K.T @ (beta[:, None] * V), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- brute force

def _unrolled(q, k, v, la, b, S0):
    """S_t = (A_t...A_1) S0 + sum_i (A_t...A_{i+1}) B_i, A_t = alpha_t (I - beta_t k_t k_t^T),
    B_t = beta_t k_t v_t^T ("From KV Cache to a State Matrix", section "The same pattern
    over more steps", with the decay gate of section "Why DeltaNet may forget too slowly")."""
    T, dk = k.shape
    A = [np.exp(la[t]) * (np.eye(dk) - b[t] * np.outer(k[t], k[t])) for t in range(T)]
    B = [b[t] * np.outer(k[t], v[t]) for t in range(T)]
    outs, states = [], []
    for t in range(T):
        prod = np.eye(dk)
        for j in range(t, -1, -1):
            prod = prod @ A[j]                       # A_t ... A_j
        S_t = prod @ S0
        for i in range(t + 1):
            P = np.eye(dk)
            for j in range(t, i, -1):
                P = P @ A[j]                         # A_t ... A_{i+1}
            S_t = S_t + P @ B[i]
        states.append(S_t)
        outs.append(S_t.T @ q[t])
    return np.array(outs), states


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_unrolled_products(seed):
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(1, 9))
    dk, dv = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    q, k, v, la, b, S0 = _random_case(rng, T, dk, dv, unit_keys=bool(seed % 2))
    o_ref, states = _unrolled(q, k, v, la, b, S0)
    o, S = run(q, k, v, log_alpha=la, beta=b, S0=S0)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, states[-1], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- structure

def test_linearity_in_initial_state_and_values():
    rng = np.random.default_rng(15)
    q, k, va, la, b, Sa = _random_case(rng, 40, 8, 6)
    vb, Sb = rng.standard_normal(va.shape), rng.standard_normal(Sa.shape)
    oa, Ta = run(q, k, va, log_alpha=la, beta=b, S0=Sa)
    ob, Tb = run(q, k, vb, log_alpha=la, beta=b, S0=Sb)
    oab, Tab = run(q, k, va + vb, log_alpha=la, beta=b, S0=Sa + Sb)
    np.testing.assert_allclose(oab, oa + ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Tab, Ta + Tb, rtol=0, atol=1e-12)


def test_value_columns_evolve_independently():
    rng = np.random.default_rng(16)
    q, k, v, la, b, S0 = _random_case(rng, 30, 5, 6)
    o, S = run(q, k, v, log_alpha=la, beta=b, S0=S0)
    for cols in ([0], [2, 5], [1, 3, 4]):
        oc, Sc = run(q, k, v[:, cols], log_alpha=la, beta=b, S0=S0[:, cols])
        np.testing.assert_allclose(oc, o[:, cols], rtol=0, atol=1e-13)
        np.testing.assert_allclose(Sc, S[:, cols], rtol=0, atol=1e-13)


@pytest.mark.parametrize("tau", [0, 1, 17, 64, 99, 100])
def test_split_and_resume_equals_one_pass(tau):
    rng = np.random.default_rng(17)
    q, k, v, la, b, S0 = _random_case(rng, 100, 6, 4)
    o, S = run(q, k, v, log_alpha=la, beta=b, S0=S0)
    o1, S1 = run(q[:tau], k[:tau], v[:tau], log_alpha=la[:tau], beta=b[:tau], S0=S0) \
        if tau else (np.zeros((0, 4)), S0)
    o2, S2 = run(q[tau:], k[tau:], v[tau:], log_alpha=la[tau:], beta=b[tau:], S0=S1) \
        if tau < 100 else (np.zeros((0, 4)), S1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S2, S, rtol=0, atol=1e-13)


def test_packed_sequences_equal_separate_calls():
    rng = np.random.default_rng(18)
    lens = [5, 0, 13, 1, 8]
    H, dk, dv = 3, 4, 5
    total = sum(lens)
    q, k = rng.standard_normal((total, H, dk)), unit(rng.standard_normal((total, H, dk)))
    v = rng.standard_normal((total, H, dv))
    la = -np.logaddexp(0.0, rng.standard_normal((total, H)))
    b = 1 / (1 + np.exp(-rng.standard_normal((total, H))))
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, S = oracle.forward(q, k, v, la, b, S0=S0, cu_seqlens=cu, threads=2)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        if lens[n] == 0:
            np.testing.assert_array_equal(S[n], S0[n])
            continue
        on, Sn = oracle.forward(q[sl], k[sl], v[sl], la[sl], b[sl], S0=S0[n:n + 1], threads=1)
        np.testing.assert_array_equal(o[sl], on)
        np.testing.assert_array_equal(S[n], Sn[0])


def test_decode_step_equals_one_token_forward():
    rng = np.random.default_rng(19)
    N, H, dk, dv = 3, 2, 4, 6
    q, k = rng.standard_normal((N, H, dk)), unit(rng.standard_normal((N, H, dk)))
    v = rng.standard_normal((N, H, dv))
    la = -np.logaddexp(0.0, rng.standard_normal((N, H)))
    b = 1 / (1 + np.exp(-rng.standard_normal((N, H))))
    S = rng.standard_normal((N, H, dk, dv))
    o, S_new = oracle.decode(q, k, v, la, b, S)
    of, Sf = oracle.forward(q, k, v, la, b, S0=S, num_seqs=N)
    np.testing.assert_array_equal(o, of)
    np.testing.assert_array_equal(S_new, Sf)


# --------------------------------------------------------------------------- chunk form

def test_gated_chunk_form_equals_the_recurrence():
    # the derivation the kernels use; residuals of the same order as the pages' own
    # chunk checks ("Attention as Matrix Algebra", section 8, printed <= 1.1e-15)
    rng = np.random.default_rng(20)
    T, dk, dv = 150, 8, 6
    for gate in ("default", "slow", "none"):
        q, k, v, la, b, S0 = _random_case(rng, T, dk, dv)
        if gate == "slow":
            la = -np.logaddexp(0.0, rng.standard_normal(T) - 6)
        elif gate == "none":
            la = np.zeros(T)
        o, S = run(q, k, v, log_alpha=la, beta=b, S0=S0)
        for C in (1, 5, 16, 64, 150):
            oc, Sc = chunk_form.chunked_forward(q, k, v, la, b, C, S0=S0)
            np.testing.assert_allclose(oc, o, rtol=0, atol=1e-12)
            np.testing.assert_allclose(Sc, S, rtol=0, atol=1e-12)


def test_segment_summaries_chain_to_the_recurrence():
    # the state map of a run of chunks is affine, S_end = P S + R (P independent of the
    # values): chaining the segments' maps from S0 gives every segment's start state, and
    # each segment run from its start reproduces the recurrence (the segmented schedule)
    rng = np.random.default_rng(22)
    T, dk, dv, C = 300, 8, 5, 16
    for shift in (-6.0, 0.0):
        q, k, v, _, b, S0 = _random_case(rng, T, dk, dv)
        la = -np.logaddexp(0.0, rng.standard_normal(T) + shift)
        o, S = run(q, k, v, log_alpha=la, beta=b, S0=S0)
        bounds = [0, 64, 128, 192, 300]  # segments of whole chunks, a ragged last one
        X, outs = S0, []
        for a, e in zip(bounds[:-1], bounds[1:]):
            P, R = chunk_form.segment_summary(k[a:e], v[a:e], la[a:e], b[a:e], C)
            oc, Sc = chunk_form.chunked_forward(q[a:e], k[a:e], v[a:e], la[a:e], b[a:e], C, S0=X)
            np.testing.assert_allclose(P @ X + R, Sc, rtol=0, atol=1e-11)
            outs.append(oc)
            X = P @ X + R
        np.testing.assert_allclose(np.concatenate(outs), o, rtol=0, atol=1e-11)
        np.testing.assert_allclose(X, S, rtol=0, atol=1e-11)


def test_pages_ungated_chunk_experiment():
    g = golden("p5_chunk_checks.json")
    rng = np.random.default_rng(3)
    Q = unit(rng.standard_normal((64, 8)))
    K = unit(rng.standard_normal((64, 8)))
    V = rng.standard_normal((64, 8))
    beta = 1 / (1 + np.exp(-rng.standard_normal(64)))
    rec, _ = run(Q, K, V, alpha=1.0, beta=beta)
    for C in g["chunk_sizes"]:
        oc, _ = chunk_form.chunked_forward(Q, K, V, np.zeros(64), beta, C)
        assert np.abs(oc - rec).max() < g["tolerance"]
    # WY: the product of the first 6 transitions
    prod = np.eye(8)
    for t in range(g["wy_tokens"]):
        prod = (np.eye(8) - beta[t] * np.outer(K[t], K[t])) @ prod
    wy = chunk_form.chunk_transition(K[:6], np.zeros(6), beta[:6])
    assert np.abs(prod - wy).max() < g["tolerance"]


def test_gated_wy_form_is_the_product_of_transitions():
    rng = np.random.default_rng(21)
    C, dk = 9, 5
    k = unit(rng.standard_normal((C, dk)))
    la = -np.logaddexp(0.0, rng.standard_normal(C))
    b = 1 / (1 + np.exp(-rng.standard_normal(C)))
    prod = np.eye(dk)
    for t in range(C):
        prod = np.exp(la[t]) * (np.eye(dk) - b[t] * np.outer(k[t], k[t])) @ prod
    np.testing.assert_allclose(chunk_form.chunk_transition(k, la, b), prod, rtol=0, atol=1e-13)
    # and it is what the oracle applies to S0 when V = 0
    S0 = rng.standard_normal((dk, 3))
    _, S = run(np.zeros((C, dk)), k, np.zeros((C, 3)), log_alpha=la, beta=b, S0=S0)
    np.testing.assert_allclose(S, prod @ S0, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- per-channel decay
# One rate per key channel ("Attention as Matrix Algebra", section 10 "Where this goes
# next": Kimi Delta Attention gives each feature channel its own rate). In the keys x
# values layout channel c is row c of S: S'_t = diag(alpha_t) S_{t-1}.

def run_pc(q, k, v, log_alpha, beta, S0=None, additive=False):
    """Single head, single sequence, log_alpha [T, dk]."""
    s0 = None if S0 is None else np.asarray(S0, dtype=np.float64)[None, None]
    o, S = oracle.forward(q[:, None, :], k[:, None, :], v[:, None, :], log_alpha[:, None, :],
                          np.asarray(beta)[:, None], S0=s0, additive=additive, threads=1)
    return o[:, 0, :], S[0, 0]


def _pc_case(rng, T, dk, dv):
    q, k, v, _, b, S0 = _random_case(rng, T, dk, dv)
    la = -np.logaddexp(0.0, rng.standard_normal((T, dk)))
    return q, k, v, la, b, S0


@pytest.mark.parametrize("seed", range(6))
def test_per_channel_brute_force_unrolled_products(seed):
    # S_t = A_t S_{t-1} + B_t with A_t = (I - beta_t k_t k_t^T) diag(alpha_t) (decay, then
    # the rank-one correction), B_t = beta_t k_t v_t^T, unrolled as explicit products
    rng = np.random.default_rng(400 + seed)
    T = int(rng.integers(2, 9))
    dk, dv = int(rng.integers(2, 5)), int(rng.integers(1, 5))
    q, k, v, la, b, S0 = _pc_case(rng, T, dk, dv)
    A = [(np.eye(dk) - b[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(la[t])) for t in range(T)]
    states, S_t = [], S0
    for t in range(T):
        prod = np.eye(dk)
        for j in range(t, -1, -1):
            prod = prod @ A[j]
        S_t = prod @ S0
        for i in range(t + 1):
            P = np.eye(dk)
            for j in range(t, i, -1):
                P = P @ A[j]
            S_t = S_t + P @ (b[i] * np.outer(k[i], v[i]))
        states.append(S_t)
    o, S = run_pc(q, k, v, la, b, S0)
    np.testing.assert_allclose(S, states[-1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, np.array([states[t].T @ q[t] for t in range(T)]), rtol=0,
                               atol=1e-12)


def test_per_channel_equal_rates_are_the_head_rate():
    rng = np.random.default_rng(410)
    q, k, v, la, b, S0 = _random_case(rng, 40, 6, 5)
    o, S = run(q, k, v, log_alpha=la, beta=b, S0=S0)
    op, Sp = run_pc(q, k, v, np.repeat(la[:, None], 6, axis=1), b, S0)
    np.testing.assert_array_equal(op, o)
    np.testing.assert_array_equal(Sp, S)


def test_per_channel_unwritten_channel_only_decays():
    # a key channel that no key touches (k[:, c] = 0) is never corrected: row c of S is
    # S0's row c times the product of its own rates, and its rates reach no other row
    rng = np.random.default_rng(411)
    T, dk, dv, c = 30, 5, 4, 2
    q, k, v, la, b, S0 = _pc_case(rng, T, dk, dv)
    k[:, c] = 0.0
    _, S = run_pc(q, k, v, la, b, S0)
    np.testing.assert_allclose(S[c], np.exp(la[:, c].sum()) * S0[c], rtol=1e-13, atol=0)
    la2 = la.copy()
    la2[:, c] -= 0.7
    _, S2 = run_pc(q, k, v, la2, b, S0)
    rows = [r for r in range(dk) if r != c]
    np.testing.assert_array_equal(S2[rows], S[rows])


def test_per_channel_beta_zero_is_rowwise_decay():
    rng = np.random.default_rng(412)
    q, k, v, la, _, S0 = _pc_case(rng, 12, 4, 3)
    o, S = run_pc(q, k, v, la, np.zeros(12), S0)
    g = np.cumsum(la, axis=0)
    np.testing.assert_allclose(S, np.exp(g[-1])[:, None] * S0, rtol=1e-13, atol=0)
    np.testing.assert_allclose(o, np.einsum("tc,cj,tc->tj", q, S0, np.exp(g)), rtol=1e-12,
                               atol=1e-14)


def test_per_channel_decode_step_equals_one_token_forward():
    rng = np.random.default_rng(413)
    N, H, dk, dv = 3, 2, 4, 6
    q, k = rng.standard_normal((N, H, dk)), unit(rng.standard_normal((N, H, dk)))
    v = rng.standard_normal((N, H, dv))
    la = -np.logaddexp(0.0, rng.standard_normal((N, H, dk)))
    b = 1 / (1 + np.exp(-rng.standard_normal((N, H))))
    S = rng.standard_normal((N, H, dk, dv))
    o, S_new = oracle.decode(q, k, v, la, b, S)
    of, Sf = oracle.forward(q, k, v, la, b, S0=S, num_seqs=N)
    np.testing.assert_array_equal(o, of)
    np.testing.assert_array_equal(S_new, Sf)


def test_per_channel_chunk_form_equals_the_recurrence():
    # the chunk form the exact kernels follow for per-channel rates
    rng = np.random.default_rng(414)
    T, dk, dv = 150, 8, 6
    for shift in (0.0, -6.0):
        q, k, v, _, b, S0 = _random_case(rng, T, dk, dv)
        la = -np.logaddexp(0.0, rng.standard_normal((T, dk)) + shift)
        o, S = run_pc(q, k, v, la, b, S0)
        for C in (1, 5, 16, 64, 150):
            oc, Sc = chunk_form.chunked_forward_per_channel(q, k, v, la, b, C, S0=S0)
            np.testing.assert_allclose(oc, o, rtol=0, atol=1e-12)
            np.testing.assert_allclose(Sc, S, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- output step

def test_out_norm_gate_worked_values():
    # o = [3, 4]: mean square 12.5, so the row is divided by sqrt(12.5) (not by its L2 norm
    # 5); a gate of 40 has sigmoid(40) = 1 in float64, so SiLU(40) = 40
    o = np.array([[3.0, 4.0]])
    got = oracle.out_norm_gate(o, np.full((1, 2), 40.0), eps=0.0)
    np.testing.assert_allclose(got, [[3 / np.sqrt(12.5) * 40, 4 / np.sqrt(12.5) * 40]], rtol=1e-15)
    # SiLU(0) = 0 and SiLU(ln 3) = ln 3 * 3/4 (sigmoid(ln 3) = 3/4)
    got = oracle.out_norm_gate(o, np.array([[0.0, np.log(3.0)]]), eps=0.0)
    np.testing.assert_allclose(got, [[0.0, 4 / np.sqrt(12.5) * 0.75 * np.log(3.0)]], rtol=1e-15)


def test_out_norm_gate_weight_eps_and_scale():
    rng = np.random.default_rng(7)
    o = rng.standard_normal((5, 3, 8))
    big = np.full(o.shape, 40.0)
    # with unit weight and SiLU(40) = 40 every row has root-mean-square 40 (eps = 0)
    got = oracle.out_norm_gate(o, big, eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(got ** 2, axis=-1)), 40.0, rtol=1e-13)
    # the normalisation is invariant to the row's scale; the weight multiplies per column
    w = rng.uniform(0.5, 2.0, 8)
    np.testing.assert_allclose(oracle.out_norm_gate(7.5 * o, big, weight=w, eps=0.0),
                               oracle.out_norm_gate(o, big, eps=0.0) * w, rtol=1e-13)
    # eps keeps an all-zero row finite (zero) and shrinks a tiny row: rms = sqrt(1e-8 + eps)
    z = oracle.out_norm_gate(np.zeros((1, 4)), np.ones((1, 4)), eps=1e-6)
    np.testing.assert_array_equal(z, 0.0)
    t = oracle.out_norm_gate(np.full((1, 4), 1e-4), np.full((1, 4), 40.0), eps=1e-6)
    np.testing.assert_allclose(t, 1e-4 / np.sqrt(1e-8 + 1e-6) * 40.0, rtol=1e-13)


# --------------------------------------------------------------------------- layer prologue

def test_layer_prologue_closed_forms():
    # q = [3, 4] has length 5; softplus(0) = ln 2, sigmoid(0) = 1/2; A scales log alpha;
    # softplus(a) -> a for large a and -> e^a for very negative a
    q = np.array([[[3.0, 4.0]], [[0.0, 0.0]]])
    k = np.array([[[1.0, 0.0]], [[0.0, 2.0]]])
    a = np.array([[0.0], [30.0]])
    b = np.array([[0.0], [np.log(3.0)]])
    qn, kn, la, beta = oracle.layer_prologue(q, k, a, b, A=np.array([2.0]))
    np.testing.assert_allclose(qn[0, 0], [0.6, 0.8], rtol=1e-15)
    np.testing.assert_array_equal(qn[1, 0], [0.0, 0.0])        # zero stays zero (max(|x|, eps))
    np.testing.assert_allclose(kn[1, 0], [0.0, 1.0], rtol=1e-15)
    np.testing.assert_allclose(la[:, 0], [-2 * np.log(2.0), -2 * (30.0 + np.log1p(np.exp(-30.0)))],
                               rtol=1e-15)
    np.testing.assert_allclose(beta[:, 0], [0.5, 0.75], rtol=1e-15)
    _, _, la2, _ = oracle.layer_prologue(q, k, np.array([[-40.0], [0.0]]), b)
    np.testing.assert_allclose(la2[0, 0], -np.exp(-40.0), rtol=1e-12)


def test_layer_prologue_per_channel_rates():
    # a [T, H, d_k]: each channel's rate from its own pre-activation, A_h per head
    q = k = np.ones((1, 2, 3))
    a = np.array([[[0.0, 30.0, -40.0], [0.0, 0.0, 0.0]]])
    _, _, la, _ = oracle.layer_prologue(q, k, a, np.zeros((1, 2)), A=np.array([1.0, 3.0]))
    np.testing.assert_allclose(la[0, 0], [-np.log(2.0), -(30.0 + np.log1p(np.exp(-30.0))),
                                          -np.exp(-40.0)], rtol=1e-12)
    np.testing.assert_allclose(la[0, 1], [-3 * np.log(2.0)] * 3, rtol=1e-15)


def test_layer_prologue_makes_unit_vectors_and_gates_in_range():
    rng = np.random.default_rng(11)
    q, k = 5 * rng.standard_normal((2, 7, 3, 16))
    a, b = 3 * rng.standard_normal((2, 7, 3))
    qn, kn, la, beta = oracle.layer_prologue(q, k, a, b, A=rng.uniform(0.1, 4.0, 3))
    np.testing.assert_allclose(np.linalg.norm(qn, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(kn, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(qn * np.linalg.norm(q, axis=-1, keepdims=True), q, rtol=1e-13)
    assert (la < 0).all() and (np.exp(la) < 1).all()
    assert (beta > 0).all() and (beta < 1).all()
