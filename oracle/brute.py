"""Brute-force expansion of the KDA recurrence for tiny T (T <= 8), FP64 numpy.

TEST INFRASTRUCTURE (see the package docstring).

This pins the C token loop by a construction that shares nothing with it: each
token's transition is formed as an explicit dk x dk matrix

    A_t = (I - beta_t k_t k_t^T) Diag(exp g_t),    B_t = beta_t k_t v_t^T,

and every state is the closed sum of products

    S_t = (A_t ... A_0) S_init + sum_{j <= t} (A_t ... A_{j+1}) B_j ,

with o_t = scale * S_t^T q_t (the KDA definition whose chunked kernel form is
"FlashInfer PR #4262: CAKE KDA Prefill Highlights" section 2). The gate is
taken from library routines (scipy's logistic function, numpy's logaddexp), not
from the oracle's own gate code.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit

MAX_T = 8


def gate_lib(a: np.ndarray, gate_mode: str, lower_bound: float) -> np.ndarray:
    """g from the raw gate a with library primitives: lb*expit(a), -logaddexp(0, a), or a."""
    a = np.asarray(a, dtype=np.float64)
    if gate_mode == "lower_bound":
        return lower_bound * expit(a)
    if gate_mode == "softplus":
        return -np.logaddexp(0.0, a)
    if gate_mode == "log_decay":
        return a
    raise ValueError(gate_mode)


def prefill_chain(q, k, v, a, beta, S0, *, scale, lower_bound=0.0, gate_mode="lower_bound"):
    """One chain: q, k, a [T, dk]; v [T, dv]; beta [T]; S0 [dk, dv]. Returns (o [T, dv], S_T)."""
    q, k, v, a, beta, S0 = (np.asarray(x, dtype=np.float64) for x in (q, k, v, a, beta, S0))
    T, dk = q.shape
    if T > MAX_T:
        raise ValueError("brute force is for T <= 8")
    eye = np.eye(dk)
    g = gate_lib(a, gate_mode, lower_bound)
    A = [(eye - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t])) for t in range(T)]
    B = [beta[t] * np.outer(k[t], v[t]) for t in range(T)]

    def chain_product(hi: int, lo: int) -> np.ndarray:
        """A_hi A_{hi-1} ... A_lo (identity when hi < lo)."""
        m = eye.copy()
        for s in range(lo, hi + 1):
            m = A[s] @ m
        return m

    outs = np.zeros((T, v.shape[1]))
    S_t = S0
    for t in range(T):
        S_t = chain_product(t, 0) @ S0
        for j in range(t + 1):
            S_t = S_t + chain_product(t, j + 1) @ B[j]
        outs[t] = scale * (S_t.T @ q[t])
    return outs, (S_t if T > 0 else S0.copy())
