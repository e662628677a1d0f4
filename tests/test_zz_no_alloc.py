"""kda_prefill_noalloc: the window-scheduled prefill for callers that cannot allocate device
memory -- an application that owns all device allocations through its own pool and forbids
raw cudaMalloc, or a latency-critical path that must not allocate. Its scratch is a fixed
array inside the library, shared by every call, so stale contents from an earlier call are
the hazard this file looks for.

The first call uses the largest window plan of a single chain (one window per SM plus one),
which writes nearly every state slot of the array. The calls after it (two in a row, on
different inputs) use the 8-head plan, whose slots sit at other offsets: a wrong index that
read a slot the current plan never writes would pick up the first call's values. Each call
is compared BITWISE with kda_prefill_ex given a workspace of its own: both run the same
plan and the same deterministic kernels, so any difference is a scratch fault.

This file is named to be collected last, so a run that stops at its first failure has
already run every other test.
"""
import pytest
import torch

import kda_recurrent_gb300 as K
import kda_synth as S

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _compare(seqlens, heads, seed, lower_bound=-5.0):
    N, T, H = len(seqlens), sum(seqlens), heads
    inp = S.prefill_inputs(seqlens, heads, seed=seed, init_std=0.02, device=DEV)
    ws = K.prefill_workspace(N, T, H, DEV)
    assert ws is not None and ws.numel() <= K.KDA_NOALLOC_SCRATCH_BYTES, "the window schedule is what this test exercises"
    args = (S.DEFAULT_SCALE, lower_bound, "lower_bound")
    out_ref, fin_ref = torch.empty_like(inp["q"]), torch.empty(N, H, 128, 128, device=DEV)
    K.kda_prefill_ex(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                     inp["init_state"], out_ref, fin_ref, *args, workspace=ws)
    out, fin = torch.empty_like(inp["q"]), torch.empty(N, H, 128, 128, device=DEV)
    K.kda_prefill_noalloc(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                          inp["init_state"], out, fin, *args)
    st, detail = K.kda_device_status()
    assert st == K.KDA_OK, (st, detail)
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    assert torch.equal(out, out_ref), "output differs from kda_prefill_ex"
    assert torch.equal(fin, fin_ref), "final state differs from kda_prefill_ex"
    return ws.numel()


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    # one chain cut into sms + 1 windows of 4 chunks: 3 (sms + 1) - 5 state slots
    big = _compare([(sms + 1) * 4 * 32], 1, seed=303)
    assert big == (3 * (sms + 1) - 5) * 128 * 128 * 4 + ((sms + 1) * 4 + 255) // 256 * 256  # states + map flags
    cfg = S.configs()["prefill_h8_t8192"]
    for seed in (101, 202):
        _compare(cfg.seqlens, cfg.num_heads, seed=seed, lower_bound=cfg.lower_bound)

