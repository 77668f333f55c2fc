"""Float64 NumPy statement of the gated chunk form, used only to check its derivation.

The CUDA prefill kernels compute the recurrence chunk by chunk. The pages print
the chunk algorithm only without decay ("Attention as Matrix Algebra: From
Softmax to the Delta Rule", section 8 "Training the delta rule in chunks":
(I + L) U = diag(beta) (V - K S), O = Q S + (Q K^T . L_C) U, S <- S + K^T U) and
derive the chunk update for two tokens ("From KV Cache to a State Matrix",
section "Chunkwise training for DeltaNet"). With the decay gate the same
substitution gives, per chunk of C tokens entering with state S,

    g_t = sum_{i<=t} log alpha_i (inside the chunk),  gamma_t = exp(g_t),
    Gamma_ti = exp(g_t - g_i) for i <= t,
    L_ti = beta_t Gamma_ti k_t^T k_i  (i < t),  T = (I + L)^{-1} diag(beta),
    U = T V - T diag(gamma) K S,
    O = diag(gamma) Q S + (Q K^T . Gamma . [i <= t]) U,
    S <- gamma_C S + Ktilde^T U,  Ktilde_i = exp(g_C - g_i) k_i,

and the product of the chunk's transitions alpha_t (I - beta_t k_t k_t^T) is
gamma_C I - Ktilde^T T diag(gamma) K.

With one rate per key channel (log alpha_t a d_k vector, the state's row c decayed
by alpha_t[c]) the same substitution holds with the decay moved inside the key
products: g_t is a vector, every Gamma_ti k_t^T k_i becomes
sum_c k_t[c] k_i[c] exp(g_t[c] - g_i[c]), diag(gamma) K becomes the rows
gamma_t . k_t, diag(gamma) Q the rows gamma_t . q_t, gamma_C S becomes
diag(gamma_C) S, and Ktilde_i = exp(g_C - g_i) . k_i (chunk_step_per_channel).

Tests compare this module with the token-by-token oracle; that pins the
derivation the kernels rely on. Nothing here is used by the CUDA path, and the
oracle does not use this module either.
"""
import numpy as np
from scipy.linalg import solve_triangular


def chunk_step(S, q, k, v, log_alpha, beta):
    """One chunk for one head. q, k [C, dk]; v [C, dv]; log_alpha, beta [C]; S [dk, dv]."""
    C = len(k)
    g = np.cumsum(log_alpha)
    gamma = np.exp(g)
    diff = g[:, None] - g[None, :]
    lower_incl = np.tril(np.ones((C, C), dtype=bool))
    Gamma = np.where(lower_incl, np.exp(np.where(lower_incl, diff, 0.0)), 0.0)
    L = np.tril(beta[:, None] * Gamma * (k @ k.T), -1)
    T = solve_triangular(np.eye(C) + L, np.diag(beta), lower=True)
    U = T @ v - T @ (gamma[:, None] * k) @ S
    O = gamma[:, None] * (q @ S) + ((q @ k.T) * Gamma) @ U
    k_tilde = np.exp(g[-1] - g)[:, None] * k
    S_next = gamma[-1] * S + k_tilde.T @ U
    return O, S_next


def chunked_forward(q, k, v, log_alpha, beta, C, S0=None):
    """Whole sequence for one head, chunk by chunk. Returns (O [T, dv], S [dk, dv])."""
    T_len, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    out = np.empty((T_len, dv))
    for c in range(0, T_len, C):
        sl = slice(c, c + C)
        out[sl], S = chunk_step(S, q[sl], k[sl], v[sl], log_alpha[sl], beta[sl])
    return out, S


def chunk_transition(k, log_alpha, beta):
    """gamma_C I - Ktilde^T T diag(gamma) K for one chunk (the WY form of its transitions)."""
    C, dk = k.shape
    g = np.cumsum(log_alpha)
    gamma = np.exp(g)
    diff = g[:, None] - g[None, :]
    lower = np.tril(np.ones((C, C), dtype=bool), -1)
    Gamma = np.where(lower, np.exp(np.where(lower, diff, 0.0)), 0.0)
    L = beta[:, None] * Gamma * (k @ k.T)
    T = solve_triangular(np.eye(C) + L, np.diag(beta), lower=True)
    k_tilde = np.exp(g[-1] - g)[:, None] * k
    return gamma[-1] * np.eye(dk) - k_tilde.T @ T @ (gamma[:, None] * k)


def chunk_step_per_channel(S, q, k, v, log_alpha, beta):
    """One chunk with one rate per key channel: log_alpha [C, dk]; otherwise as chunk_step.
    Every exponent is g_t - g_i with i <= t (or g_t, g_C - g_i), so every factor is <= 1."""
    C = len(k)
    g = np.cumsum(log_alpha, axis=0)                      # [C, dk]
    lower_incl = np.tril(np.ones((C, C), dtype=bool))
    diff = g[:, None, :] - g[None, :, :]                  # [t, i, c]
    dec = np.where(lower_incl[:, :, None], np.exp(np.where(lower_incl[:, :, None], diff, 0.0)), 0.0)
    KK = np.einsum("tc,ic,tic->ti", k, k, dec)
    QK = np.einsum("tc,ic,tic->ti", q, k, dec)
    L = np.tril(beta[:, None] * KK, -1)
    T = solve_triangular(np.eye(C) + L, np.diag(beta), lower=True)
    U = T @ v - T @ (np.exp(g) * k) @ S
    O = (np.exp(g) * q) @ S + QK @ U
    k_tilde = np.exp(g[-1][None, :] - g) * k
    S_next = np.exp(g[-1])[:, None] * S + k_tilde.T @ U
    return O, S_next


def chunked_forward_per_channel(q, k, v, log_alpha, beta, C, S0=None):
    """Whole sequence for one head with per-channel rates, chunk by chunk."""
    T_len, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    out = np.empty((T_len, dv))
    for c in range(0, T_len, C):
        sl = slice(c, c + C)
        out[sl], S = chunk_step_per_channel(S, q[sl], k[sl], v[sl], log_alpha[sl], beta[sl])
    return out, S


def segment_summary(k, v, log_alpha, beta, C):
    """The affine map of a run of chunks, S_end = P S + R: P is the end state from the
    identity with zero values (the product of the run's transitions), R the end state from
    zero with the values. The segmented GPU schedule computes these per segment."""
    dk, dv = k.shape[1], v.shape[1]
    q0 = np.zeros_like(k)
    _, P = chunked_forward(q0, k, np.zeros((len(k), dk)), log_alpha, beta, C, S0=np.eye(dk))
    _, R = chunked_forward(q0, k, v, log_alpha, beta, C, S0=np.zeros((dk, dv)))
    return P, R
