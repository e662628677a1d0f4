"""GPU parity of kda_decode (through the C ABI) against the FP64 oracle.

The sweep is the decode workload: H = 8, rows 1, 2, 4, ..., 4096, a 16384-slot pool
(8 GiB FP32 / 4 GiB BF16, so slot offsets need 64 bits), unique scattered slots, the
pool updated in place. Every slot outside slot_idx must stay byte-identical.
"""
import pytest
import torch

import kda_recurrent_gb300 as K
import kda_synth as S
import oracle
from helpers import assert_out_close, assert_state_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALE = S.DEFAULT_SCALE


def bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def run_and_check(pool, rows, H, seed, *, lower_bound=-5.0, gate_mode="lower_bound", slots=None):
    inp = S.decode_inputs(rows, H, seed=seed, device=DEV)
    if slots is None:
        slots = S.slot_indices(rows, pool.shape[0], seed=seed, device=DEV)
    sl = slots.long()
    before = pool.clone()
    gathered = before[sl].double().cpu()
    out = K.decode(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], slots, pool, scale=SCALE,
                   lower_bound=lower_bound, gate_mode=gate_mode)
    st, detail = K.kda_device_status()
    assert st == K.KDA_OK, (st, detail)
    # bookkeeping: every other slot byte-identical
    after_sel = pool[sl].clone()
    before[sl] = after_sel
    assert torch.equal(bits(before), bits(pool)), "a slot outside slot_idx changed"
    del before
    ref_out, ref_state, _ = oracle.decode(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], gathered,
                                          scale=SCALE, lower_bound=lower_bound, gate_mode=gate_mode)
    assert_out_close(out.cpu(), ref_out)
    assert_state_close(after_sel.cpu(), ref_state)
    return inp, out


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decode_sweep_pool16384(state_dtype):
    cfg = S.configs()["decode_h8_pool16384"]
    pool = S.state_pool(cfg.num_slots, cfg.num_heads, state_dtype, std=cfg.pool_std, seed=cfg.seed, device=DEV)
    for rows in cfg.rows:
        run_and_check(pool, rows, cfg.num_heads, cfg.seed, lower_bound=cfg.lower_bound, gate_mode=cfg.gate_mode)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows", [3, 37, 300])
def test_decode_softplus_small_pool(state_dtype, rows):
    pool = S.state_pool(512, 3, state_dtype, std=0.05, seed=9, device=DEV)
    run_and_check(pool, rows, 3, 9, lower_bound=0.0, gate_mode="softplus")


def test_decode_padding_and_out_of_range_slots():
    pool = S.state_pool(64, 2, "f32", std=0.02, seed=4, device=DEV)
    before = pool.clone()
    inp = S.decode_inputs(3, 2, seed=4, device=DEV)
    K.kda_device_status()
    slots = torch.tensor([-1, 5, 64], dtype=torch.int32, device=DEV)  # padding, valid, past the pool
    out = K.decode(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], slots, pool, scale=SCALE,
                   lower_bound=-5.0)
    st, detail = K.kda_device_status()
    assert st == K.KDA_ERR_DEVICE_INPUT and detail == 2
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
    mask = torch.ones(64, dtype=torch.bool, device=DEV)
    mask[5] = False
    assert torch.equal(bits(pool[mask]), bits(before[mask]))
    assert not torch.equal(pool[5], before[5])


def test_decode_matches_prefill_of_length_one():
    H = 4
    inp = S.decode_inputs(6, H, seed=8, device=DEV)
    pool = S.state_pool(16, H, "f32", std=0.02, seed=8, device=DEV)
    slots = torch.tensor([9, 2, 15, 0, 7, 11], dtype=torch.int32, device=DEV)
    init = pool[slots.long()].clone()
    out_d = K.decode(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], slots, pool, scale=SCALE,
                     lower_bound=-5.0)
    cu = torch.arange(7, dtype=torch.int32, device=DEV)
    out_p, fin_p = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], cu, init, scale=SCALE,
                             lower_bound=-5.0)
    assert_out_close(out_d.cpu(), out_p.double().cpu())
    assert_state_close(pool[slots.long()].cpu(), fin_p.double().cpu(), tol=1e-3)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decode_streaming_schedule_with_padding_rows(state_dtype):
    """Enough items for the streaming (bulk-copy ring) schedule, with padding rows and a slot
    past the pool mixed in: those rows give zero outputs and touch no state."""
    rows, H, slots_n = 700, 2, 2048
    pool = S.state_pool(slots_n, H, state_dtype, std=0.02, seed=12, device=DEV)
    before = pool.clone()
    inp = S.decode_inputs(rows, H, seed=12, device=DEV)
    slots = S.slot_indices(rows, slots_n, seed=12, device=DEV)
    slots[5] = -1
    slots[300] = -7
    slots[611] = slots_n + 3
    K.kda_device_status()
    out = K.decode(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], slots, pool, scale=SCALE,
                   lower_bound=-5.0)
    st, detail = K.kda_device_status()
    assert st == K.KDA_ERR_DEVICE_INPUT and detail == 611
    pad = torch.tensor([5, 300, 611], device=DEV)
    assert torch.count_nonzero(out[pad]) == 0
    live = torch.ones(rows, dtype=torch.bool, device=DEV)
    live[pad] = False
    sl = slots[live].long()
    after_sel = pool[sl].clone()
    restored = pool.clone()
    restored[sl] = before[sl]
    assert torch.equal(bits(restored), bits(before)), "a slot outside the live rows changed"
    ref_out, ref_state, _ = oracle.decode(inp["q"][live], inp["k"][live], inp["v"][live], inp["g_raw"][live],
                                          inp["beta"][live], before[sl].double().cpu(), scale=SCALE, lower_bound=-5.0)
    assert_out_close(out[live].cpu(), ref_out)
    assert_state_close(after_sel.cpu(), ref_state)
