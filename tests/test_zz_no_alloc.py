"""kda_prefill_noalloc: the window-scheduled prefill for callers that cannot allocate device
memory (an application that owns all device allocations through its own pool, or a
latency-critical path that must not allocate). Its scratch is a fixed array inside the
library, so the test checks that two calls in a row -- the second one on different inputs,
with the first call's leftovers still in the array -- match kda_prefill_ex given a
workspace of its own, within the tolerances the other parity tests use.

This file is named to be collected last, so a run that stops at its first failure has
already run every other test.
"""
import pytest
import torch

import kda_recurrent_gb300 as K
import kda_synth as S
from helpers import OUT_MAX_ABS, OUT_REL_L2, STATE_REL_L2, max_abs, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_both(seed):
    cfg = S.configs()["prefill_h8_t8192"]
    inp = S.prefill_inputs(cfg.seqlens, cfg.num_heads, seed=seed, init_std=cfg.init_std, device=DEV)
    N, T, H = 1, cfg.total_tokens, cfg.num_heads
    ws = K.prefill_workspace(N, T, H, DEV)
    assert ws is not None and ws.numel() <= 32 << 20, "the window schedule is what this test exercises"
    args = (cfg.scale, cfg.lower_bound, cfg.gate_mode)
    out_ref, fin_ref = torch.empty_like(inp["q"]), torch.empty(N, H, 128, 128, device=DEV)
    K.kda_prefill_ex(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                     inp["init_state"], out_ref, fin_ref, *args, workspace=ws)
    out, fin = torch.empty_like(inp["q"]), torch.empty(N, H, 128, 128, device=DEV)
    K.kda_prefill_noalloc(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                          inp["init_state"], out, fin, *args)
    st, detail = K.kda_device_status()
    assert st == K.KDA_OK, (st, detail)
    return out.cpu(), fin.cpu(), out_ref.cpu(), fin_ref.cpu()


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    for seed in (101, 202):
        out, fin, out_ref, fin_ref = _run_both(seed)
        assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
        assert rel_l2(out, out_ref) <= OUT_REL_L2 and max_abs(out, out_ref) <= OUT_MAX_ABS
        assert rel_l2(fin, fin_ref) <= STATE_REL_L2
