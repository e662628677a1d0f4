"""GPU parity of the windowed (chunk-parallel) prefill schedule, kda_prefill_ex, against the
FP64 oracle and against the sequential schedule.

The window pass carries each window's linear map M through the same tcgen05 chain as the
state; the slow-decay cases make the carried part of the state dominate, so an error in M,
in the carry or in the window bookkeeping shows up there first.
"""
import pytest
import torch

import kda_recurrent_gb300 as K
import kda_synth as S
from helpers import assert_out_close, assert_state_close, oracle_prefill, rel_l2, slice_problem

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALE = S.DEFAULT_SCALE


def to_dev(inp):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def windowed(inp, *, lower_bound, gate_mode, init=True):
    d = to_dev(inp)
    N, T, H = d["cu_seqlens"].shape[0] - 1, d["q"].shape[0], d["q"].shape[1]
    ws = K.prefill_workspace(N, T, H, DEV)
    assert ws is not None, "this shape should take the windowed schedule"
    out, fin = K.prefill(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], d["cu_seqlens"],
                         d["init_state"] if init else None, scale=SCALE, lower_bound=lower_bound,
                         gate_mode=gate_mode, workspace=ws)
    st, detail = K.kda_device_status()
    assert st == K.KDA_OK, (st, detail)
    return out.cpu(), fin.cpu()


def check(inp, *, lower_bound, gate_mode):
    out, fin = windowed(inp, lower_bound=lower_bound, gate_mode=gate_mode)
    ref_out, ref_fin = oracle_prefill(inp, scale=SCALE, lower_bound=lower_bound, gate_mode=gate_mode)
    assert_out_close(out, ref_out)
    assert_state_close(fin, ref_fin)


def test_windowed_h8_t8192():
    cfg = S.configs()["prefill_h8_t8192"]
    check(S.config_inputs(cfg), lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)


def test_windowed_matches_sequential():
    cfg = S.configs()["prefill_h8_t8192"]
    inp = S.config_inputs(cfg)
    out_w, fin_w = windowed(inp, lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)
    d = to_dev(inp)
    out_s, fin_s = K.prefill(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], d["cu_seqlens"], d["init_state"],
                             scale=SCALE, lower_bound=cfg.lower_bound)
    assert rel_l2(out_w, out_s.cpu()) < 5e-3
    assert rel_l2(fin_w, fin_s.cpu()) < 1e-3


@pytest.mark.parametrize("rate", [0.002, 0.03])
def test_windowed_slow_decay_carries_the_state(rate):
    """g = -rate * |a| per token: the state remembers thousands of tokens, so the start state
    of late windows is mostly carried through the maps M of earlier windows."""
    inp = S.prefill_inputs([3000], 2, seed=31, init_std=0.02)
    inp["g_raw"] = (-rate * inp["g_raw"].float().abs()).to(torch.bfloat16)
    check(inp, lower_bound=0.0, gate_mode="log_decay")


def test_windowed_maps_zero_in_some_windows_only():
    """Slow decay, then g = -5 per token over tokens 1000-1999, then slow decay again: the maps
    of the windows inside the fast stretch underflow to zero and the others do not, so the
    carry mixes product steps with steps that take S_start[w+1] = E_w."""
    inp = S.prefill_inputs([3000], 2, seed=39, init_std=0.02)
    g = -0.002 * inp["g_raw"].float().abs()
    g[1000:2000] = -5.0
    inp["g_raw"] = g.to(torch.bfloat16)
    d = to_dev(inp)
    ws = K.prefill_workspace(1, 3000, 2, DEV)
    out, fin = K.prefill(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], d["cu_seqlens"], d["init_state"],
                         scale=SCALE, lower_bound=0.0, gate_mode="log_decay", workspace=ws)
    st, detail = K.kda_device_status()
    assert st == K.KDA_OK, (st, detail)
    # the per-window map flags after the state slots: 2 chains, W windows each; this sequence
    # has 94 chunks in windows of ceil(94 / W) chunks, and windows 1 .. wins - 2 carry a map
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    W = min(sms // 2 + 1, 94 // 4)
    lw = -(-94 // W)
    wins = -(-94 // lw)
    off = 2 * (3 * W - 5) * 128 * 128 * 4
    flags = ws[off:off + 2 * W * 4].view(torch.int32).view(2, W)[:, 1:wins - 1].cpu()
    assert (flags == 0).any() and (flags == 1).any(), flags
    ref_out, ref_fin = oracle_prefill(inp, scale=SCALE, lower_bound=0.0, gate_mode="log_decay")
    assert_out_close(out.cpu(), ref_out)
    assert_state_close(fin.cpu(), ref_fin)


@pytest.mark.parametrize("lens", [[3000], [1500, 3000, 610]], ids=["1x3000", "varlen3"])
def test_windowed_lower_bound_minus_8(lens):
    """lb = -8, the widest exponent range of the half-chunk anchors, on the window schedule with
    an initial state: the window maps M are built through the same anchored operands."""
    inp = S.prefill_inputs(lens, 2, seed=38 + len(lens), init_std=0.02)
    N, T = len(lens), sum(lens)
    slots = K.kda_prefill_workspace_size(N, T, 2, sm_count=152) // (N * 2 * 128 * 128 * 4)
    assert (slots + 5) // 3 >= 4, "a plan of at least 4 windows per chain (3 W - 5 state slots)"
    check(inp, lower_bound=-8.0, gate_mode="lower_bound")


def test_windowed_ragged_multi_sequence():
    inp = S.prefill_inputs([1000, 37, 0, 2500, 130], 2, seed=32, init_std=0.02)
    check(inp, lower_bound=0.0, gate_mode="softplus")


def test_windowed_zero_init_and_in_place():
    inp = to_dev(S.prefill_inputs([2048], 4, seed=33, init_std=0.02))
    ws = K.prefill_workspace(1, 2048, 4, DEV)
    args = dict(scale=SCALE, lower_bound=-5.0, gate_mode="lower_bound")
    out_ref = torch.empty_like(inp["q"])
    fin_ref = torch.empty_like(inp["init_state"])
    K.kda_prefill_ex(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"], inp["init_state"],
                     out_ref, fin_ref, workspace=ws, **args)
    state = inp["init_state"].clone()
    out = torch.empty_like(inp["q"])
    K.kda_prefill_ex(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"], state, out, state,
                     workspace=ws, **args)
    assert torch.equal(out, out_ref) and torch.equal(state, fin_ref)
    out0, fin0 = windowed({k: v.cpu() if isinstance(v, torch.Tensor) else v for k, v in inp.items()},
                          lower_bound=-5.0, gate_mode="lower_bound", init=False)
    ref_out, ref_fin = oracle_prefill({**{k: v.cpu() for k, v in inp.items() if k != "init_state"},
                                       "init_state": None}, scale=SCALE, lower_bound=-5.0, gate_mode="lower_bound")
    assert_out_close(out0, ref_out)
    assert_state_close(fin0, ref_fin)


def test_workspace_rules():
    inp = to_dev(S.prefill_inputs([1024], 2, seed=34, init_std=None))
    need = K.kda_prefill_workspace_size(1, 1024, 2)
    assert need > 0
    out = torch.empty_like(inp["q"])
    small = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(K.KdaError) as ei:
        K.kda_prefill_ex(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"], None, out, None,
                         SCALE, -5.0, workspace=small)
    assert ei.value.status == K.KDA_ERR_INVALID_ARG
    # no workspace: the sequential schedule, bitwise equal to kda_prefill
    out_a, fin_a = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"], None,
                             scale=SCALE, lower_bound=-5.0)
    out_b = torch.empty_like(out_a)
    fin_b = torch.empty_like(fin_a)
    K.kda_prefill_ex(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"], None, out_b, fin_b,
                     SCALE, -5.0, workspace=None)
    assert torch.equal(out_a, out_b) and torch.equal(fin_a, fin_b)


def test_windowed_tail_after_full_waves():
    """More chains than SMs with a short last wave: the full waves run one CTA per chain and
    only the last chains are windowed. Chains start longest sequence first, so the split falls
    inside the shorter (second) sequence, whose heads then run on both schedules."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tail = 4
    H = (sms + tail) // 2
    tail = 2 * H - sms
    lens = [1500, 900]
    inp = S.prefill_inputs(lens, H, seed=35, init_std=0.02)
    assert K.kda_prefill_workspace_size(2, sum(lens), H) > 0
    out, fin = windowed(inp, lower_bound=-5.0, gate_mode="lower_bound")
    d = to_dev(inp)
    out_s, fin_s = K.prefill(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], d["cu_seqlens"], d["init_state"],
                             scale=SCALE, lower_bound=-5.0)
    # the chains of the full waves take the sequential kernel unchanged: bitwise equal
    first = sms - H  # heads of sequence 1 that precede the windowed tail
    assert torch.equal(out[:lens[0]], out_s[:lens[0]].cpu()) and torch.equal(fin[0], fin_s[0].cpu())
    assert torch.equal(out[lens[0]:, :first], out_s[lens[0]:, :first].cpu())
    assert torch.equal(fin[1, :first], fin_s[1, :first].cpu())
    # the windowed tail against the oracle, and a few heads of the full waves
    heads = [0, first - 1] + list(range(first, H))
    sub = slice_problem(inp, heads=heads)
    ref_out, ref_fin = oracle_prefill(sub, scale=SCALE, lower_bound=-5.0, gate_mode="lower_bound")
    assert_out_close(out[:, heads], ref_out)
    assert_state_close(fin[:, heads], ref_fin)
    assert tail == H - first


def test_windowed_three_windows_minimum():
    """13 chunks on 2 chains: the smallest plan, windows 0, 1 and 2 of 5, 5 and 3 chunks
    (window 0 from the initial state, one window pass, one carry step)."""
    assert K.kda_prefill_workspace_size(1, 400, 2, sm_count=152) == 2 * 4 * 128 * 128 * 4 + 256  # + map flags
    inp = S.prefill_inputs([400], 2, seed=36, init_std=0.02)
    check(inp, lower_bound=-5.0, gate_mode="lower_bound")


def test_windowed_tail_of_a_varlen_batch():
    """39 sequences x 4 heads = 156 chains: the 4 chains of the shortest sequence, which
    start last, take the window schedule after the full wave; the full wave matches the
    chunk loop bitwise and the windowed chains match the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = 4
    N = sms // H + 1
    gen = torch.Generator().manual_seed(37)
    lens = (torch.randint(700, 1400, (N,), generator=gen)).tolist()
    lens[N // 2] = 520  # the shortest: 17 chunks in windows of at least 4
    inp = S.prefill_inputs(lens, H, seed=37, init_std=0.02)
    assert K.kda_prefill_workspace_size(N, sum(lens), H) > 0
    out, fin = windowed(inp, lower_bound=-5.0, gate_mode="lower_bound")
    d = to_dev(inp)
    out_s, fin_s = K.prefill(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], d["cu_seqlens"], d["init_state"],
                             scale=SCALE, lower_bound=-5.0)
    cu = inp["cu_seqlens"].tolist()
    short = N // 2
    others = [n for n in range(N) if n != short]
    for n in others:
        sl = slice(cu[n], cu[n + 1])
        assert torch.equal(out[sl], out_s[sl].cpu()) and torch.equal(fin[n], fin_s[n].cpu()), n
    sub = slice_problem(inp, seqs=[short, others[0], others[-1]])
    ref_out, ref_fin = oracle_prefill(sub, scale=SCALE, lower_bound=-5.0, gate_mode="lower_bound")
    assert_out_close(out[sub["token_index"]], ref_out)
    assert_state_close(fin[[short, others[0], others[-1]]], ref_fin)
