"""Canary bands around every buffer the library writes, in place of a memory checker: each
output is a view into a larger allocation whose bands before and after it hold a fixed byte
pattern, and after the call the bands must be byte-identical. Covers the prefill (sequential
and window schedules, checkpoints, final state) and the decode (register and streaming
schedules, several tokens per row)."""
import pytest
import torch

import kda_recurrent_gb300 as K
import kda_synth as S

pytestmark = pytest.mark.gpu
DEV = "cuda"
BAND = 4096  # bytes on each side, a multiple of 16 so the view keeps the 16-byte alignment


def banded(shape, dtype):
    """(view, raw): `view` of `shape` inside `raw`, with BAND bytes of pattern on both sides."""
    n = torch.Size(shape).numel() * torch.tensor([], dtype=dtype).element_size()
    raw = torch.full((n + 2 * BAND,), 0xA5, dtype=torch.uint8, device=DEV)
    return raw[BAND:BAND + n].view(dtype).view(shape), raw


def bands_intact(raw):
    return bool((raw[:BAND] == 0xA5).all() and (raw[-BAND:] == 0xA5).all())


@pytest.mark.parametrize("lens,H,windows", [([100, 37], 3, False), ([1500], 2, True), ([700, 64, 300], 4, True)])
def test_prefill_writes_stay_inside_out_and_final_state(lens, H, windows):
    inp = S.prefill_inputs(lens, H, seed=71, init_std=0.02, device=DEV)
    N, T = len(lens), sum(lens)
    out, raw_o = banded((T, H, 128), torch.bfloat16)
    fin, raw_f = banded((N, H, 128, 128), torch.float32)
    ck_rows = sum(n // 64 for n in lens)
    ck, raw_c = banded((max(ck_rows, 1), H, 128, 128), torch.float32)
    offs = torch.tensor([sum(n // 64 for n in lens[:i]) for i in range(N)], dtype=torch.int32, device=DEV)
    ws = K.prefill_workspace(N, T, H, DEV) if windows else None
    assert (ws is not None) == windows
    K.kda_prefill_ex(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"], inp["init_state"],
                     out, fin, S.DEFAULT_SCALE, -5.0, workspace=ws, checkpoints=ck, ckpt_offsets=offs, ckpt_every=64)
    assert K.kda_device_status()[0] == K.KDA_OK
    assert bands_intact(raw_o) and bands_intact(raw_f) and bands_intact(raw_c)
    ref_out, ref_fin = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                                 inp["init_state"], scale=S.DEFAULT_SCALE, lower_bound=-5.0, workspace=ws)
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)


@pytest.mark.parametrize("rows,tokens,state_dtype", [(5, 1, "f32"), (40, 1, "bf16"), (700, 1, "f32"),
                                                     (700, 1, "bf16"), (160, 3, "f32"), (160, 8, "bf16")])
def test_decode_writes_stay_inside_out(rows, tokens, state_dtype):
    H = 8
    pool = S.state_pool(rows + 8, H, state_dtype, std=0.02, seed=72, device=DEV)
    d = S.decode_inputs(rows * tokens, H, seed=72, device=DEV)
    if tokens > 1:
        d = {k: v.view(rows, tokens, *v.shape[1:]) for k, v in d.items()}
    slots = S.slot_indices(rows, rows + 8, seed=72, device=DEV)
    out, raw_o = banded(tuple(d["q"].shape), torch.bfloat16)
    K.kda_decode_ex(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], slots, pool, out, S.DEFAULT_SCALE, -5.0)
    assert K.kda_device_status()[0] == K.KDA_OK
    assert bands_intact(raw_o)
    assert torch.isfinite(out.float()).all()
