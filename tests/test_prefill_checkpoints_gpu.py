"""Intermediate FP32 state checkpoints of kda_prefill_ex, every `ckpt_every` tokens.

Checkpoint j of sequence n is, by definition, the final state after the first
(j + 1) * ckpt_every tokens of that sequence; the oracle computes it as the final state of
that prefix run as a sequence of its own.
"""
import pytest
import torch

import kda_recurrent_gb300 as K
import kda_synth as S
from helpers import assert_state_close, oracle_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALE = S.DEFAULT_SCALE


def prefix_problem(inp, every):
    """All checkpoint prefixes of every sequence as one varlen problem (CPU tensors)."""
    cu = inp["cu_seqlens"].tolist()
    toks, lens, inits, owners = [], [], [], []
    for n in range(len(cu) - 1):
        T = cu[n + 1] - cu[n]
        for j in range(T // every):
            L = (j + 1) * every
            toks.append(torch.arange(cu[n], cu[n] + L))
            lens.append(L)
            inits.append(n)
    idx = torch.cat(toks)
    sub = {key: inp[key].index_select(0, idx) for key in ("q", "k", "v", "g_raw", "beta")}
    sub["cu_seqlens"] = torch.tensor([0] + torch.tensor(lens).cumsum(0).tolist(), dtype=torch.int32)
    init = inp.get("init_state")
    sub["init_state"] = None if init is None else init[torch.tensor(inits)].contiguous()
    return sub


@pytest.mark.parametrize("windows", [False, True])
@pytest.mark.parametrize("every", [64, 96])
def test_checkpoints_match_oracle_prefixes(windows, every):
    lens = [700, 64, 5, 257] if not windows else [1500, 300]
    H = 2
    inp = S.prefill_inputs(lens, H, seed=60 + every, init_std=0.02)
    counts = [n // every for n in lens]
    offsets = torch.tensor([0] + torch.tensor(counts).cumsum(0).tolist()[:-1], dtype=torch.int32)
    rows = sum(counts)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    ws = K.prefill_workspace(len(lens), sum(lens), H, DEV) if windows else None
    assert (ws is not None) == windows
    ck = torch.full((rows + 1, H, 128, 128), float("nan"), device=DEV)  # one spare row must stay untouched
    out = torch.empty_like(d["q"])
    fin = torch.empty_like(d["init_state"])
    K.kda_prefill_ex(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], d["cu_seqlens"], d["init_state"], out, fin, SCALE,
                     -5.0, workspace=ws, checkpoints=ck, ckpt_offsets=offsets.to(DEV), ckpt_every=every)
    assert K.kda_device_status()[0] == K.KDA_OK
    assert torch.isnan(ck[rows]).all()
    ref_out, ref_fin = oracle_prefill(prefix_problem(inp, every), scale=SCALE, lower_bound=-5.0,
                                      gate_mode="lower_bound")
    assert_state_close(ck[:rows].cpu(), ref_fin)
    # the same call without checkpoints gives bitwise the same outputs and final states
    out2, fin2 = K.prefill(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], d["cu_seqlens"], d["init_state"],
                           scale=SCALE, lower_bound=-5.0, workspace=ws)
    assert torch.equal(out, out2) and torch.equal(fin, fin2)


def test_checkpoint_row_past_the_buffer_is_reported_not_written():
    inp = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v)
           for k, v in S.prefill_inputs([256], 1, seed=63, init_std=None).items()}
    ck = torch.zeros(3, 1, 128, 128, device=DEV)  # 4 checkpoints are due, 3 rows given
    K.kda_device_status()
    out = torch.empty_like(inp["q"])
    K.kda_prefill_ex(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"], None, out, None,
                     SCALE, -5.0, checkpoints=ck, ckpt_offsets=torch.zeros(1, dtype=torch.int32, device=DEV),
                     ckpt_every=64)
    st, detail = K.kda_device_status()
    assert st == K.KDA_ERR_DEVICE_INPUT and detail == 0
    assert torch.isfinite(ck).all() and torch.count_nonzero(ck[2]) > 0
