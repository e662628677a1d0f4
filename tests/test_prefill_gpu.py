"""GPU parity of kda_prefill (through the C ABI) against the FP64 oracle.

Tolerances: output relL2 <= 1e-2 and max-abs <= 3e-2 (BF16 I/O); final FP32 state
relL2 <= 2e-3. Bitwise properties (chunk-boundary split, varlen vs separate calls,
head permutation, beta = g = 0) are checked exactly.
"""
import pytest
import torch

import kda_recurrent_gb300 as K
import kda_synth as S
from helpers import (assert_out_close, assert_state_close, launch_order, oracle_prefill, slice_problem)

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALE = S.DEFAULT_SCALE


def to_dev(inp):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def gpu_prefill(inp, *, lower_bound, gate_mode, init="use"):
    d = to_dev(inp)
    init_state = d.get("init_state") if init == "use" else None
    out, fin = K.prefill(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], d["cu_seqlens"], init_state, scale=SCALE,
                         lower_bound=lower_bound, gate_mode=gate_mode)
    st, detail = K.kda_device_status()
    assert st == K.KDA_OK, f"device status {st} (detail {detail})"
    return out.cpu(), fin.cpu()


def check_against_oracle(inp, *, lower_bound, gate_mode):
    out, fin = gpu_prefill(inp, lower_bound=lower_bound, gate_mode=gate_mode)
    ref_out, ref_fin = oracle_prefill(inp, scale=SCALE, lower_bound=lower_bound, gate_mode=gate_mode)
    r_o, m_o = assert_out_close(out, ref_out)
    r_s = assert_state_close(fin, ref_fin)
    return r_o, m_o, r_s


RAGGED = [[1], [15], [16], [17], [31], [32], [33], [63], [64], [65], [100], [5, 0, 40, 1, 97]]


@pytest.mark.parametrize("seqlens", RAGGED, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("gate", [("lower_bound", -5.0), ("softplus", 0.0), ("lower_bound", -8.0)],
                         ids=lambda g: f"{g[0]}{g[1]:g}")
def test_prefill_ragged_small(seqlens, gate):
    inp = S.prefill_inputs(seqlens, 2, seed=11 + sum(seqlens), init_std=0.02)
    check_against_oracle(inp, lower_bound=gate[1], gate_mode=gate[0])


def test_prefill_log_decay_mode():
    inp = S.prefill_inputs([77], 2, seed=5, init_std=0.02)
    inp["g_raw"] = -inp["g_raw"].abs()
    check_against_oracle(inp, lower_bound=0.0, gate_mode="log_decay")


def test_cfg_h1_t64():
    cfg = S.configs()["prefill_h1_t64"]
    check_against_oracle(S.config_inputs(cfg), lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)


def test_cfg_h8_t8192():
    cfg = S.configs()["prefill_h8_t8192"]
    check_against_oracle(S.config_inputs(cfg), lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)


def test_cfg_varlen16_h32_sampled_heads():
    """Full launch (all 32 heads); the oracle checks 6 heads over all 16 sequences and all 32
    heads of four sequences: the longest (3747 tokens, ragged), the shortest (307), one whose
    last chunk holds a single token (449) and one that ends on a chunk boundary (2112)."""
    cfg = S.configs()["prefill_varlen16_h32"]
    inp = S.config_inputs(cfg)
    out, fin = gpu_prefill(inp, lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)
    heads = [0, 5, 11, 17, 26, 31]
    sub = slice_problem(inp, heads=heads)
    ref_out, ref_fin = oracle_prefill(sub, scale=SCALE, lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)
    assert_out_close(out[:, heads], ref_out)
    assert_state_close(fin[:, heads], ref_fin)
    lens = cfg.seqlens
    seqs = [lens.index(max(lens)), lens.index(min(lens)), lens.index(449), lens.index(2112)]
    assert lens[seqs[0]] % 32 and lens[seqs[2]] % 32 == 1 and lens[seqs[3]] % 32 == 0
    sub = slice_problem(inp, seqs=seqs)
    ref_out, ref_fin = oracle_prefill(sub, scale=SCALE, lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)
    assert_out_close(out[sub["token_index"]], ref_out)
    assert_state_close(fin[seqs], ref_fin)


@pytest.fixture(scope="module")
def cfg5():
    """The 8 x 16384 H96 lb = -8 workload on the device, drawn as the bench draws it."""
    cfg = S.configs()["prefill_8x16384_h96"]
    inp = S.config_inputs(cfg, device=DEV)
    yield cfg, inp
    del inp
    torch.cuda.empty_cache()


def test_cfg_8x16384_h96_sampled_chains(cfg5):
    """Full-size launch on the sequential schedule (kda_prefill); the oracle checks 2 heads of
    every sequence."""
    cfg, inp = cfg5
    out, fin = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                         inp["init_state"], scale=SCALE, lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)
    assert K.kda_device_status()[0] == K.KDA_OK
    heads = [3, 70]
    sub = slice_problem(inp, heads=heads)
    ref_out, ref_fin = oracle_prefill(sub, scale=SCALE, lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)
    assert_out_close(out[:, heads].cpu(), ref_out)
    assert_state_close(fin[:, heads].cpu(), ref_fin)


def test_cfg_8x16384_h96_as_benched(cfg5):
    """The schedule the bench times: kda_prefill_ex with its workspace, i.e. full waves of one
    CTA per chain and the chains of the short last wave cut into windows (window 0, window
    pass, carry, output pass) at lb = -8. The oracle checks every windowed chain and 2 heads of
    every sequence from the full waves."""
    cfg, inp = cfg5
    N, H, T = len(cfg.seqlens), cfg.num_heads, cfg.total_tokens
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    ws = K.prefill_workspace(N, T, H, DEV)
    tail = (N * H) % sms
    assert ws is not None and 0 < 3 * tail <= sms, "this workload has a windowed tail on this GPU"
    out, fin = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                         inp["init_state"], scale=SCALE, lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode,
                         workspace=ws)
    st, detail = K.kda_device_status()
    assert st == K.KDA_OK, (st, detail)
    order = launch_order(cfg.seqlens, H)
    windowed = order[N * H - tail:]
    assert len({n for n, _ in windowed}) == 1  # equal lengths: the last heads of the last sequence
    n_t = windowed[0][0]
    t_heads = [h for _, h in windowed]
    sub = slice_problem(inp, heads=t_heads, seqs=[n_t])
    ref_out, ref_fin = oracle_prefill(sub, scale=SCALE, lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)
    cu = inp["cu_seqlens"].tolist()
    assert_out_close(out[cu[n_t]:cu[n_t + 1], t_heads].cpu(), ref_out, what="windowed out")
    assert_state_close(fin[n_t, t_heads].cpu()[None], ref_fin, what="windowed state")
    full = [5, 61]
    assert not set(full) & set(t_heads)
    sub = slice_problem(inp, heads=full)
    ref_out, ref_fin = oracle_prefill(sub, scale=SCALE, lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)
    assert_out_close(out[:, full].cpu(), ref_out)
    assert_state_close(fin[:, full].cpu(), ref_fin)


def test_split_at_chunk_boundaries_is_bitwise():
    inp = to_dev(S.prefill_inputs([256], 4, seed=21, init_std=0.02))
    args = dict(scale=SCALE, lower_bound=-5.0, gate_mode="lower_bound")
    out_full, fin_full = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                                   inp["init_state"], **args)
    state = inp["init_state"]
    outs = []
    for a, b in [(0, 32), (32, 96), (96, 160), (160, 256)]:
        cu = torch.tensor([0, b - a], dtype=torch.int32, device=DEV)
        sl = slice(a, b)
        o, state = K.prefill(inp["q"][sl].contiguous(), inp["k"][sl].contiguous(), inp["v"][sl].contiguous(),
                             inp["g_raw"][sl].contiguous(), inp["beta"][sl].contiguous(), cu, state, **args)
        outs.append(o)
    assert torch.equal(torch.cat(outs), out_full)
    assert torch.equal(state, fin_full)


def test_varlen_equals_separate_calls_bitwise():
    lens = [40, 0, 129, 7, 64]
    inp = to_dev(S.prefill_inputs(lens, 3, seed=22, init_std=0.02))
    args = dict(scale=SCALE, lower_bound=0.0, gate_mode="softplus")
    out, fin = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                         inp["init_state"], **args)
    cu = inp["cu_seqlens"].tolist()
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        c1 = torch.tensor([0, lens[n]], dtype=torch.int32, device=DEV)
        o, f = K.prefill(inp["q"][sl].contiguous(), inp["k"][sl].contiguous(), inp["v"][sl].contiguous(),
                         inp["g_raw"][sl].contiguous(), inp["beta"][sl].contiguous(), c1,
                         inp["init_state"][n:n + 1].contiguous(), **args)
        assert torch.equal(o, out[sl])
        assert torch.equal(f[0], fin[n])


@pytest.mark.parametrize("lens", [
    [64, 64, 0, 130, 64, 7, 130, 0, 33, 7],           # ties: chains start longest first, ties by index
    [3 * (i % 7) + 32 * (i % 3) for i in range(300)],  # more sequences than are ranked: index order
])
def test_launch_order_runs_every_chain_once(lens):
    """Each chain's result is independent of when its CTA starts: bitwise equal to a call on
    that sequence alone, so every (sequence, head) ran exactly once on its own data."""
    inp = to_dev(S.prefill_inputs(lens, 2, seed=28, init_std=0.02))
    args = dict(scale=SCALE, lower_bound=-5.0, gate_mode="lower_bound")
    out, fin = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                         inp["init_state"], **args)
    assert K.kda_device_status()[0] == K.KDA_OK
    cu = inp["cu_seqlens"].tolist()
    for n in sorted(set(range(0, len(lens), max(1, len(lens) // 12))) | {len(lens) - 1}):
        sl = slice(cu[n], cu[n + 1])
        c1 = torch.tensor([0, lens[n]], dtype=torch.int32, device=DEV)
        o, f = K.prefill(inp["q"][sl].contiguous(), inp["k"][sl].contiguous(), inp["v"][sl].contiguous(),
                         inp["g_raw"][sl].contiguous(), inp["beta"][sl].contiguous(), c1,
                         inp["init_state"][n:n + 1].contiguous(), **args)
        assert torch.equal(o, out[sl]) and torch.equal(f[0], fin[n]), n
    sub = slice_problem({k: v.cpu() if isinstance(v, torch.Tensor) else v for k, v in inp.items()})
    ref_out, ref_fin = oracle_prefill(sub, scale=SCALE, **{k: v for k, v in args.items() if k != "scale"})
    assert_out_close(out.cpu(), ref_out)
    assert_state_close(fin.cpu(), ref_fin)


def test_zero_length_sequence_copies_initial_state():
    inp = to_dev(S.prefill_inputs([0, 33, 0], 2, seed=23, init_std=0.02))
    out, fin = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                         inp["init_state"], scale=SCALE, lower_bound=-5.0)
    assert torch.equal(fin[0], inp["init_state"][0])
    assert torch.equal(fin[2], inp["init_state"][2])
    _, fin0 = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"], None,
                        scale=SCALE, lower_bound=-5.0)
    assert torch.count_nonzero(fin0[0]) == 0 and torch.count_nonzero(fin0[2]) == 0


def test_in_place_state_carry():
    inp = to_dev(S.prefill_inputs([70, 33], 2, seed=24, init_std=0.02))
    args = dict(scale=SCALE, lower_bound=-5.0, gate_mode="lower_bound")
    out_ref, fin_ref = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                                 inp["init_state"], **args)
    state = inp["init_state"].clone()
    out = torch.empty_like(inp["q"])
    K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"], state, out, state,
                  **args)
    assert torch.equal(out, out_ref) and torch.equal(state, fin_ref)


def test_beta0_gate0_leaves_state_bitwise_unchanged():
    inp = S.prefill_inputs([45], 2, seed=25, init_std=0.02)
    inp["beta"] = torch.zeros_like(inp["beta"])
    out, fin = gpu_prefill(inp, lower_bound=0.0, gate_mode="lower_bound")  # lb = 0 gives g = 0
    assert torch.equal(fin, inp["init_state"])
    ref_out, _ = oracle_prefill(inp, scale=SCALE, lower_bound=0.0, gate_mode="lower_bound")
    assert_out_close(out, ref_out)


def test_head_permutation_is_bitwise_equivariant():
    inp = to_dev(S.prefill_inputs([50, 90], 5, seed=26, init_std=0.02))
    perm = torch.tensor([3, 0, 4, 1, 2], device=DEV)
    args = dict(scale=SCALE, lower_bound=-5.0, gate_mode="lower_bound")
    out, fin = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                         inp["init_state"], **args)
    p = {k: inp[k][:, perm].contiguous() for k in ("q", "k", "v", "g_raw", "beta")}
    out_p, fin_p = K.prefill(p["q"], p["k"], p["v"], p["g_raw"], p["beta"], inp["cu_seqlens"],
                             inp["init_state"][:, perm].contiguous(), **args)
    assert torch.equal(out_p, out[:, perm]) and torch.equal(fin_p, fin[:, perm])


def test_bad_cu_seqlens_is_reported_not_faulted():
    inp = to_dev(S.prefill_inputs([40, 40], 1, seed=27, init_std=None))
    K.kda_device_status()  # clear
    cu = torch.tensor([0, 60, 50], dtype=torch.int32, device=DEV)  # decreasing: invalid
    out = torch.zeros_like(inp["q"])
    fin = torch.zeros(2, 1, 128, 128, device=DEV)
    K.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], cu, None, out, fin, SCALE, -5.0)
    st, detail = K.kda_device_status()
    assert st == K.KDA_ERR_DEVICE_INPUT and detail == 1
    assert torch.isfinite(out.float()).all()


def test_more_than_2_31_elements_per_token_tensor():
    """4 x 32768 tokens x H144: each token tensor holds 2.4e9 elements (> 2^31), so every token
    and output offset needs 64 bits. The oracle checks the first and last head of every
    sequence, whose rows sit at both ends of each tensor."""
    lens, H = [32768] * 4, 144
    assert sum(lens) * H * 128 > 2 ** 31
    inp = S.prefill_inputs(lens, H, seed=29, init_std=0.02, device=DEV)
    out, fin = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                         inp["init_state"], scale=SCALE, lower_bound=-5.0)
    assert K.kda_device_status()[0] == K.KDA_OK
    heads = [0, H - 1]
    sub = slice_problem(inp, heads=heads)
    ref_out, ref_fin = oracle_prefill(sub, scale=SCALE, lower_bound=-5.0, gate_mode="lower_bound")
    assert_out_close(out[:, heads].cpu(), ref_out)
    assert_state_close(fin[:, heads].cpu(), ref_fin)
    # the last token of the last sequence, head H - 1, lies past element 2^31 of `out`
    assert (sum(lens) - 1) * H * 128 + (H - 1) * 128 > 2 ** 31
    del inp, out, fin
    torch.cuda.empty_cache()
