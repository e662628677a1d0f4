"""The chunked closed form of KDA prefill, FP64 numpy, as a checker of the recurrence.

TEST INFRASTRUCTURE (see the package docstring).

Follows "FlashInfer PR #4262: CAKE KDA Prefill Highlights":
  * section 2, the seven per-chunk steps (gate prefix and centred Q/K; causal
    Mqk and the triangular system; inverse of the 32 x 32 lower-triangular
    matrix; state decay and projection; residual/beta transform; fused state and
    output update; output store), and the concatenated update
    [S_new | O] = [S_d | O_0] + U [K_r | Mqk^T] with U: [dv, L],
    [K_r | Mqk^T]: [L, dk + L], [S | O]: [dv, dk + L] (the page keeps S^T);
  * section 1, the fixed exponent anchor b = lower_bound * log2(e), C = 16 b, with
    operand factors 2^(G_i - C) and 2^(C - G_j) whose product is 2^(G_i - G_j).

With G_i the inclusive per-channel prefix of g in base-2 units, the chunk algebra
is (rows = tokens of the chunk, L <= 32 of them):
    Qbar = scale q (x) 2^G,  Kbar = k (x) 2^G,  Kr = k (x) 2^(G_last - G)
    Mqk[i, j] = scale sum_c q_i k_j 2^(G_i - G_j)   (j <= i)
    A[i, j]   =       sum_c k_i k_j 2^(G_i - G_j)   (j <  i)
    U = (I + Diag(beta) A)^-1 Diag(beta) (V - Kbar S)
    O = Qbar S + Mqk U,    S_new = Diag(2^G_last) S + Kr^T U

``pair_scheme`` selects how the pair factor 2^(G_i - G_j) is formed:
  * "direct"  -- the difference is exponentiated as is (reference);
  * "anchor"  -- the section-1 fixed anchor (lower-bound gate only);
  * "halves"  -- a per-channel anchor at the middle of each 16-token half for the
    two diagonal blocks and the factorisation 2^(G_i - G_15) 2^(G_15 - G_j)
    through the half boundary for the off-diagonal block.  This is the reading
    used where the fixed anchor leaves the float range (lower_bound = -8, and the
    softplus gate, which has no bound); the pages do not print it.
In FP64 all three agree to rounding; ``anchor_exponent_radius`` reports the
largest |exponent| an operand factor reaches, to compare with BF16/FP32's 127.
"""
from __future__ import annotations

import math

import numpy as np

from .brute import gate_lib

CHUNK = 32
HALF = 16
LOG2E = 1.0 / math.log(2.0)
FLOAT_MAX_EXP2 = 127  # largest finite binary exponent of FP32 and BF16


def fixed_anchor(lower_bound: float) -> float:
    """C = 16 * lower_bound * log2(e): the section-1 anchor, in base-2 units."""
    return HALF * lower_bound * LOG2E


def _pair_direct(left, right, G, causal_incl):
    L = G.shape[0]
    M = np.zeros((L, L))
    for i in range(L):
        for j in range(i + 1 if causal_incl else i):
            M[i, j] = np.sum(left[i] * right[j] * np.exp2(G[i] - G[j]))
    return M


def _pair_anchor(left, right, G, C, causal_incl):
    lhs = left * np.exp2(G - C)
    rhs = right * np.exp2(C - G)
    return np.tril(lhs @ rhs.T, 0 if causal_incl else -1)


def _pair_halves(left, right, G, causal_incl):
    L = G.shape[0]
    M = np.zeros((L, L))
    for lo in range(0, L, HALF):
        hi = min(lo + HALF, L)
        anchor = 0.5 * (G[lo] + G[hi - 1])
        lhs = left[lo:hi] * np.exp2(G[lo:hi] - anchor)
        rhs = right[lo:hi] * np.exp2(anchor - G[lo:hi])
        M[lo:hi, lo:hi] = lhs @ rhs.T
    if L > HALF:
        edge = G[HALF - 1]
        lhs = left[HALF:] * np.exp2(G[HALF:] - edge)
        rhs = right[:HALF] * np.exp2(edge - G[:HALF])
        M[HALF:, :HALF] = lhs @ rhs.T
    return np.tril(M, 0 if causal_incl else -1)


def pair_products(q, k, G, *, scale, scheme="direct", lower_bound=None):
    """(Mqk, A) of one chunk with the chosen exponent scheme (see module docstring)."""
    if scheme == "direct":
        mqk = _pair_direct(q, k, G, True)
        akk = _pair_direct(k, k, G, False)
    elif scheme == "anchor":
        if lower_bound is None:
            raise ValueError("the fixed anchor needs a lower bound")
        C = fixed_anchor(lower_bound)
        mqk = _pair_anchor(q, k, G, C, True)
        akk = _pair_anchor(k, k, G, C, False)
    elif scheme == "halves":
        mqk = _pair_halves(q, k, G, True)
        akk = _pair_halves(k, k, G, False)
    else:
        raise ValueError(scheme)
    return scale * mqk, akk


def anchor_exponent_radius(G, lower_bound) -> float:
    """Largest |G_i - C| over a chunk: the base-2 exponent the anchored operand factors reach."""
    return float(np.max(np.abs(G - fixed_anchor(lower_bound))))


def halves_exponent_radius(G) -> float:
    """Largest base-2 exponent any operand factor of the "halves" scheme reaches in one chunk.

    Diagonal-block factors 2^(G - anchor) and 2^(anchor - G) take both signs; the
    off-diagonal factors 2^(G_i - G_15) (i >= 16) and 2^(G_15 - G_j) (j < 16) never
    exceed 1 (exponent <= 0), so they can only underflow, where the true product is
    below 2^-126 anyway.
    """
    L = G.shape[0]
    r = -np.inf
    for lo in range(0, L, HALF):
        hi = min(lo + HALF, L)
        anchor = 0.5 * (G[lo] + G[hi - 1])
        r = max(r, float(np.max(np.abs(G[lo:hi] - anchor))))
    if L > HALF:
        edge = G[HALF - 1]
        r = max(r, float(np.max(G[HALF:] - edge)), float(np.max(edge - G[:HALF])))
    return r


def prefill_chain(q, k, v, a, beta, S0, *, scale, lower_bound=0.0, gate_mode="lower_bound",
                  scheme="direct", chunk=CHUNK):
    """One chain by the chunked closed form. Shapes as ``brute.prefill_chain``."""
    q, k, v, a, beta, S = (np.asarray(x, dtype=np.float64) for x in (q, k, v, a, beta, S0))
    T, dk = q.shape
    dv = v.shape[1]
    S = S.copy()
    out = np.zeros((T, dv))
    g = gate_lib(a, gate_mode, lower_bound)
    for c0 in range(0, T, chunk):
        L = min(chunk, T - c0)
        qc, kc, vc, bc = q[c0:c0 + L], k[c0:c0 + L], v[c0:c0 + L], beta[c0:c0 + L]
        # 1. gate prefix (inclusive, base 2) and the decayed operands
        G = np.cumsum(g[c0:c0 + L], axis=0) * LOG2E
        qbar = scale * qc * np.exp2(G)
        kbar = kc * np.exp2(G)
        kr = kc * np.exp2(G[L - 1] - G)
        # 2. causal Mqk and the strictly lower triangular system
        mqk, akk = pair_products(qc, kc, G, scale=scale, scheme=scheme,
                                 lower_bound=lower_bound if gate_mode == "lower_bound" else None)
        # 3. inverse of the unit lower-triangular (I + Diag(beta) A)
        tinv = np.linalg.inv(np.eye(L) + bc[:, None] * akk)
        # 4. state decay and projection
        s_d = np.exp2(G[L - 1])[:, None] * S
        proj_k = kbar @ S
        o_0 = qbar @ S
        # 5. residual / beta transform
        U = tinv @ (bc[:, None] * (vc - proj_k))
        # 6. fused state and output update, in the page's transposed layout
        SO = np.hstack([s_d.T, o_0.T]) + U.T @ np.hstack([kr, mqk.T])
        S = SO[:, :dk].T
        # 7. output transpose and store
        out[c0:c0 + L] = SO[:, dk:].T
    return out, S
