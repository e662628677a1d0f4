"""Pins of the FP64 oracle to things other than itself (CPU only).

* brute-force transition-matrix expansion for T <= 8 (oracle/brute.py);
* the chunked closed form of "FlashInfer PR #4262: CAKE KDA Prefill Highlights"
  section 2, under the direct, fixed-anchor (section 1) and half-chunk exponent schemes;
* the anchor-cancellation identity 2^(G_i - C) 2^(C - G_j) = 2^(G_i - G_j) and the
  range of the anchored operands;
* closed forms: beta = 0; beta = 0 with g = 0; the delta-rule write at beta = 1;
* invariants: linearity in (S0, V), split at any token, the window affine composite
  S_end = M S_start + E, varlen = separate sequences, dk-channel permutation, decode =
  prefill of length one;
* the gate against library routines, and a two-token d = 2 example worked by hand;
* planted mistakes (a dropped decay, a transposed read-out, a misplaced beta, a wrong
  prefix) that at least one pin must reject.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
from oracle import brute, chunked

HERE = os.path.dirname(os.path.abspath(__file__))
RNG = np.random.default_rng(1234)
MODES = [("lower_bound", -5.0), ("lower_bound", -8.0), ("softplus", 0.0), ("log_decay", 0.0)]


def make_case(T, H=1, dk=16, dv=16, *, seed=0, mode="lower_bound", unit_k=True, init_std=0.1, lens=None):
    rng = np.random.default_rng(seed)
    lens = [T] if lens is None else lens
    T = sum(lens)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    a = rng.standard_normal((T, H, dk))
    if mode == "log_decay":
        a = -np.abs(a)
    beta = expit(rng.standard_normal((T, H)))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    s0 = init_std * rng.standard_normal((len(lens), H, dk, dv))
    return dict(q=q, k=k, v=v, a=a, beta=beta, cu=cu, s0=s0)


def run(c, mode, lb, scale=0.3, **kw):
    return oracle.prefill(c["q"], c["k"], c["v"], c["a"], c["beta"], c["cu"], c["s0"], scale=scale,
                          lower_bound=lb, gate_mode=mode, **kw)


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(b), 1e-300))


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("mode,lb", MODES)
@pytest.mark.parametrize("dk,dv", [(16, 16), (8, 24), (128, 128)])
def test_loop_matches_brute_force(mode, lb, dk, dv):
    T = 8 if dk < 128 else 5
    c = make_case(T, 2, dk, dv, seed=dk + dv, mode=mode)
    out, fin, _ = run(c, mode, lb)
    for h in range(2):
        o_b, s_b = brute.prefill_chain(c["q"][:, h], c["k"][:, h], c["v"][:, h], c["a"][:, h], c["beta"][:, h],
                                       c["s0"][0, h], scale=0.3, lower_bound=lb, gate_mode=mode)
        assert rel(out[:, h], o_b) < 1e-12
        assert rel(fin[0, h], s_b) < 1e-12


# ---------------------------------------------------------------- chunked form

@pytest.mark.parametrize("mode,lb", MODES)
@pytest.mark.parametrize("scheme", ["direct", "halves", "anchor"])
def test_loop_matches_chunked_closed_form(mode, lb, scheme):
    if scheme == "anchor" and mode != "lower_bound":
        pytest.skip("the fixed anchor is defined by a lower bound only")
    lens = [64, 45, 1, 97]  # full chunks, a ragged tail, a single token, three-plus chunks
    c = make_case(0, 2, 128, 128, seed=7, mode=mode, lens=lens, init_std=0.02)
    out, fin, _ = run(c, mode, lb, scale=1 / math.sqrt(128))
    for n in range(len(lens)):
        s, e = c["cu"][n], c["cu"][n + 1]
        for h in range(2):
            o_c, s_c = chunked.prefill_chain(c["q"][s:e, h], c["k"][s:e, h], c["v"][s:e, h], c["a"][s:e, h],
                                             c["beta"][s:e, h], c["s0"][n, h], scale=1 / math.sqrt(128),
                                             lower_bound=lb, gate_mode=mode, scheme=scheme)
            assert rel(out[s:e, h], o_c) < 1e-11
            assert rel(fin[n, h], s_c) < 1e-11


def test_anchor_cancellation_identity():
    """2^(G_i - C) 2^(C - G_j) = 2^(G_i - G_j) (section 1 of the prefill note), in FP64."""
    for lb in (-5.0, -8.0, -1.0):
        C = chunked.fixed_anchor(lb)
        assert C == pytest.approx(16 * lb / math.log(2), rel=1e-15)
        g = lb * expit(RNG.standard_normal((32, 128)))
        G = np.cumsum(g, axis=0) / math.log(2)
        lhs = np.exp2(G[:, None, :] - C) * np.exp2(C - G[None, :, :])
        rhs = np.exp2(G[:, None, :] - G[None, :, :])
        assert np.max(np.abs(lhs / rhs - 1)) < 1e-13


def test_anchor_range_and_half_chunk_scheme():
    """The fixed anchor fits the float range at lb = -5 (<= 16|b| = 115.4 bits) but not at
    lb = -8 (up to 184.7 bits): anchored operands overflow FP32 there, while the
    half-chunk scheme stays within 8|b| bits and finite."""
    for lb, fits in ((-5.0, True), (-8.0, False)):
        b = lb / math.log(2)
        g = np.full((32, 128), lb)  # the steepest chunk the bound allows
        g[:, :64] = lb * expit(RNG.standard_normal((32, 64)))
        G = np.cumsum(g, axis=0) / math.log(2)
        r_anchor = chunked.anchor_exponent_radius(G, lb)
        r_halves = chunked.halves_exponent_radius(G)
        assert r_anchor <= 16 * abs(b) + 1e-9
        assert r_halves <= 8 * abs(b) + 1e-9
        assert (r_anchor < chunked.FLOAT_MAX_EXP2) == fits
        with np.errstate(over="ignore"):
            anchored = np.exp2(G - chunked.fixed_anchor(lb)).astype(np.float32)
        assert np.all(np.isfinite(anchored)) == fits
    assert 16 * abs(-5.0 / math.log(2)) == pytest.approx(115.4, abs=0.05)
    assert 16 * abs(-8.0 / math.log(2)) == pytest.approx(184.7, abs=0.05)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("mode,lb", MODES)
def test_beta_zero_closed_form(mode, lb):
    c = make_case(21, 1, 12, 10, seed=3, mode=mode)
    c["beta"][:] = 0.0
    out, fin, _ = run(c, mode, lb)
    g = brute.gate_lib(c["a"][:, 0], mode, lb)
    Gam = np.cumsum(g, axis=0)
    S0 = c["s0"][0, 0]
    for t in range(21):
        o_t = 0.3 * (np.exp(Gam[t])[:, None] * S0).T @ c["q"][t, 0]
        assert rel(out[t, 0], o_t) < 1e-13
    assert rel(fin[0, 0], np.exp(Gam[-1])[:, None] * S0) < 1e-13


def test_beta_zero_gate_zero_leaves_state_bitwise():
    c = make_case(40, 2, 16, 16, seed=4)
    c["beta"][:] = 0.0
    out, fin, _ = run(c, "lower_bound", 0.0)  # lower_bound = 0 gives g = 0
    assert np.array_equal(fin, c["s0"])
    for t in range(40):
        for h in range(2):
            assert rel(out[t, h], 0.3 * c["s0"][0, h].T @ c["q"][t, h]) < 1e-14


@pytest.mark.parametrize("unit", [True, False])
def test_beta_one_delta_rule_write(unit):
    """k_t^T S_t = (1 - |k_t|^2) k_t^T D_t S_{t-1} + |k_t|^2 v_t^T; = v_t^T for unit k."""
    c = make_case(6, 1, 16, 16, seed=5, unit_k=unit)
    c["beta"][:] = 1.0
    S = c["s0"][0, 0].copy()
    for t in range(6):
        one = {k2: (c[k2][t:t + 1] if k2 not in ("cu", "s0") else None) for k2 in c}
        _, fin, _ = oracle.prefill(one["q"], one["k"], one["v"], one["a"], one["beta"], np.array([0, 1]),
                                   S[None, None], scale=1.0, lower_bound=-5.0)
        k, v = c["k"][t, 0], c["v"][t, 0]
        DS = np.exp(-5.0 * expit(c["a"][t, 0]))[:, None] * S
        nk = float(k @ k)
        expect = (1 - nk) * (k @ DS) + nk * v
        assert rel(k @ fin[0, 0], expect) < 1e-12
        if unit:
            assert rel(k @ fin[0, 0], v) < 1e-12
        S = fin[0, 0]


def test_hand_worked_example():
    with open(os.path.join(HERE, "golden", "kda_tiny_d2.json")) as f:
        gd = json.load(f)
    q = np.array(gd["q"])[:, None, :]
    k = np.array(gd["k"])[:, None, :]
    v = np.array(gd["v"])[:, None, :]
    g = np.array(gd["g"])[:, None, :]
    beta = np.array(gd["beta"])[:, None]
    S0 = np.array(gd["S0"])[None, None]
    out, fin, _ = oracle.prefill(q, k, v, g, beta, np.array([0, 2]), S0, scale=gd["scale"], gate_mode="log_decay")
    np.testing.assert_allclose(out[:, 0], gd["expected_o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(fin[0, 0], gd["expected_S2"], rtol=0, atol=1e-14)
    _, fin1, _ = oracle.prefill(q[:1], k[:1], v[:1], g[:1], beta[:1], np.array([0, 1]), S0, scale=1.0,
                                gate_mode="log_decay")
    np.testing.assert_allclose(fin1[0, 0], gd["expected_S1"], rtol=0, atol=1e-14)


# ---------------------------------------------------------------- invariants

def test_linearity_in_state_and_values():
    c1 = make_case(50, 2, 16, 16, seed=6)
    c2 = make_case(50, 2, 16, 16, seed=6)
    rng = np.random.default_rng(9)
    c2["v"] = rng.standard_normal(c2["v"].shape)
    c2["s0"] = rng.standard_normal(c2["s0"].shape)
    a1, b1 = 0.7, -1.3
    c3 = dict(c1, v=a1 * c1["v"] + b1 * c2["v"], s0=a1 * c1["s0"] + b1 * c2["s0"])
    o1, f1, _ = run(c1, "softplus", 0.0)
    o2, f2, _ = run(c2, "softplus", 0.0)
    o3, f3, _ = run(c3, "softplus", 0.0)
    assert rel(o3, a1 * o1 + b1 * o2) < 1e-12
    assert rel(f3, a1 * f1 + b1 * f2) < 1e-12


@pytest.mark.parametrize("cut", [32, 64, 17, 1])
def test_split_and_carry_is_bitwise(cut):
    c = make_case(96, 2, 16, 16, seed=8)
    out, fin, _ = run(c, "lower_bound", -5.0)
    first = {k2: (c[k2][:cut] if k2 not in ("cu", "s0") else None) for k2 in c}
    rest = {k2: (c[k2][cut:] if k2 not in ("cu", "s0") else None) for k2 in c}
    o1, f1, _ = oracle.prefill(first["q"], first["k"], first["v"], first["a"], first["beta"], np.array([0, cut]),
                               c["s0"], scale=0.3, lower_bound=-5.0)
    o2, f2, _ = oracle.prefill(rest["q"], rest["k"], rest["v"], rest["a"], rest["beta"], np.array([0, 96 - cut]),
                               f1, scale=0.3, lower_bound=-5.0)
    assert np.array_equal(np.concatenate([o1, o2]), out)
    assert np.array_equal(f2, fin)


@pytest.mark.parametrize("mode,lb", [("lower_bound", -5.0), ("softplus", 0.0)])
def test_window_affine_composite(mode, lb):
    """The window schedule's reading of the composite schedule of FlashInfer PR #5573
    ("1. Composite schedule"): over a window, S_end = M S_start + E, where E is the window
    run from a zero state and M the window run from S_start = I with V = 0 (d_k = d_v), and
    the window's outputs are the zero-start outputs plus those of the V = 0 run from S_start."""
    d = 16
    c = make_case(150, 1, d, d, seed=12, mode=mode)
    cut = 64
    out, fin, _ = run(c, mode, lb)
    part = lambda x: x[cut:]
    win = dict(q=part(c["q"]), k=part(c["k"]), v=part(c["v"]), a=part(c["a"]), beta=part(c["beta"]),
               cu=np.array([0, 150 - cut], dtype=np.int32))
    _, s_start, _ = oracle.prefill(c["q"][:cut], c["k"][:cut], c["v"][:cut], c["a"][:cut], c["beta"][:cut],
                                   np.array([0, cut]), c["s0"], scale=0.3, lower_bound=lb, gate_mode=mode)
    o_e, e, _ = run(dict(win, s0=np.zeros((1, 1, d, d))), mode, lb)
    _, m, _ = run(dict(win, v=np.zeros_like(win["v"]), s0=np.eye(d)[None, None]), mode, lb)
    o_s, _, _ = run(dict(win, v=np.zeros_like(win["v"]), s0=s_start), mode, lb)
    assert rel(m[0, 0] @ s_start[0, 0] + e[0, 0], fin[0, 0]) < 1e-12
    assert rel(o_e + o_s, out[cut:]) < 1e-12


def test_varlen_equals_separate_sequences_bitwise():
    lens = [5, 0, 33, 64]
    c = make_case(0, 3, 16, 16, seed=10, lens=lens)
    out, fin, _ = run(c, "softplus", 0.0)
    for n, L in enumerate(lens):
        s, e = c["cu"][n], c["cu"][n + 1]
        o, f, _ = oracle.prefill(c["q"][s:e], c["k"][s:e], c["v"][s:e], c["a"][s:e], c["beta"][s:e],
                                 np.array([0, L]), c["s0"][n:n + 1], scale=0.3, gate_mode="softplus")
        assert np.array_equal(o, out[s:e])
        assert np.array_equal(f[0], fin[n])


def test_thread_count_does_not_change_results():
    c = make_case(0, 4, 16, 16, seed=11, lens=[30, 70, 3])
    o1, f1, _ = run(c, "lower_bound", -5.0, threads=1)
    o2, f2, _ = run(c, "lower_bound", -5.0, threads=5)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)


def test_dk_channel_permutation():
    c = make_case(37, 2, 16, 12, seed=12)
    out, fin, _ = run(c, "lower_bound", -5.0)
    p = np.random.default_rng(3).permutation(16)
    cp = dict(c, q=c["q"][..., p], k=c["k"][..., p], a=c["a"][..., p], s0=c["s0"][:, :, p, :])
    out_p, fin_p, _ = run(cp, "lower_bound", -5.0)
    assert rel(out_p, out) < 1e-13
    assert rel(fin_p, fin[:, :, p, :]) < 1e-13


def test_decode_equals_prefill_of_length_one():
    c = make_case(0, 3, 16, 16, seed=13, lens=[1, 1, 1, 1])
    out, fin, _ = run(c, "softplus", 0.0)
    o_d, s_d, _ = oracle.decode(c["q"], c["k"], c["v"], c["a"], c["beta"], c["s0"], scale=0.3, gate_mode="softplus")
    assert np.array_equal(o_d, out) and np.array_equal(s_d, fin)


def test_gate_against_library_routines():
    a = np.concatenate([RNG.standard_normal(200) * 4, [0.0, 30.0, -30.0, 1e-8]])
    for x in a:
        assert oracle.gate(x, "lower_bound", -5.0) == pytest.approx(-5.0 * expit(x), rel=1e-14, abs=1e-300)
        assert oracle.gate(x, "softplus") == pytest.approx(-np.logaddexp(0.0, x), rel=1e-14, abs=1e-300)
        assert oracle.gate(x, "log_decay") == x
    assert oracle.gate(0.0, "lower_bound", -5.0) == -2.5
    assert oracle.gate(0.0, "softplus") == pytest.approx(-math.log(2.0), rel=1e-15)


# ---------------------------------------------------------------- planted mistakes

def _mutant_loop(c, mutation, lb=-5.0, scale=0.3):
    """A copy of the token recurrence with one planted mistake (numpy, single chain)."""
    q, k, v, a, beta, S = c["q"][:, 0], c["k"][:, 0], c["v"][:, 0], c["a"][:, 0], c["beta"][:, 0], c["s0"][0, 0].copy()
    outs = []
    for t in range(q.shape[0]):
        g = lb * expit(a[t])
        if mutation != "no_decay":
            S = np.exp(g)[:, None] * S
        w = S.T @ k[t]
        u = (v[t] - w) * (beta[t] if mutation != "beta_on_w_only" else 1.0)
        if mutation == "beta_on_w_only":
            u = v[t] - beta[t] * w
        S = S + np.outer(k[t], u)
        outs.append(scale * (S @ q[t] if mutation == "transposed_readout" else S.T @ q[t]))
    return np.array(outs), S


@pytest.mark.parametrize("mutation", ["no_decay", "transposed_readout", "beta_on_w_only"])
def test_pins_reject_planted_mistakes(mutation):
    c = make_case(8, 1, 16, 16, seed=14)
    o_m, s_m = _mutant_loop(c, mutation)
    o_b, s_b = brute.prefill_chain(c["q"][:, 0], c["k"][:, 0], c["v"][:, 0], c["a"][:, 0], c["beta"][:, 0],
                                   c["s0"][0, 0], scale=0.3, lower_bound=-5.0)
    assert rel(o_m, o_b) > 1e-3 or rel(s_m, s_b) > 1e-3
    o_ok, s_ok = _mutant_loop(c, "none")
    assert rel(o_ok, o_b) < 1e-12 and rel(s_ok, s_b) < 1e-12


def test_chunked_form_rejects_exclusive_prefix():
    """An exclusive (instead of inclusive) gate prefix in the chunked form is caught."""
    c = make_case(40, 1, 16, 16, seed=15)
    out, fin, _ = run(c, "lower_bound", -5.0)
    a_shift = np.concatenate([np.full((1, 1, 16), -np.inf), c["a"][:-1]])  # g_0 = 0, g_t = g_{t-1}
    o_c, s_c = chunked.prefill_chain(c["q"][:, 0], c["k"][:, 0], c["v"][:, 0], a_shift[:, 0], c["beta"][:, 0],
                                     c["s0"][0, 0], scale=0.3, lower_bound=-5.0)
    assert rel(o_c, out[:, 0]) > 1e-3


# ---------------------------------------------------------------- decode input options

def test_decode_qk_normalisation_is_scale_invariant():
    """With in-step L2 normalisation, scaling q and k by positive factors changes nothing
    (up to the eps term), and unit inputs are left as they are."""
    c = make_case(0, 3, 16, 16, seed=16, lens=[1] * 5, unit_k=False)
    args = dict(scale=0.3, lower_bound=-5.0)
    o1, s1, _ = oracle.decode(c["q"], c["k"], c["v"], c["a"], c["beta"], c["s0"], norm_eps=0.0, **args)
    o2, s2, _ = oracle.decode(7.5 * c["q"], 0.02 * c["k"], c["v"], c["a"], c["beta"], c["s0"], norm_eps=0.0, **args)
    assert rel(o1, o2) < 1e-13 and rel(s1, s2) < 1e-13
    qn = c["q"] / np.linalg.norm(c["q"], axis=-1, keepdims=True)
    kn = c["k"] / np.linalg.norm(c["k"], axis=-1, keepdims=True)
    o3, s3, _ = oracle.decode(qn, kn, c["v"], c["a"], c["beta"], c["s0"], **args)
    assert rel(o1, o3) < 1e-13 and rel(s1, s3) < 1e-13
    o4, _, _ = oracle.decode(c["q"], c["k"], c["v"], c["a"], c["beta"], c["s0"], **args)
    assert rel(o1, o4) > 1e-3  # not normalising changes the result


def test_decode_beta_logits_match_library_logistic():
    c = make_case(0, 2, 16, 16, seed=17, lens=[1] * 4)
    logits = RNG.standard_normal(c["beta"].shape) * 3
    args = dict(scale=0.3, gate_mode="softplus")
    o1, s1, _ = oracle.decode(c["q"], c["k"], c["v"], c["a"], logits, c["s0"], beta_logits=True, **args)
    o2, s2, _ = oracle.decode(c["q"], c["k"], c["v"], c["a"], expit(logits), c["s0"], **args)
    assert rel(o1, o2) < 1e-14 and rel(s1, s2) < 1e-14
