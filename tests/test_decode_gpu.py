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
@pytest.mark.parametrize("rows", [3, 37, 160, 300])  # 480 items: BF16 states stream, FP32 ones do not
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


@pytest.mark.parametrize("rows", [5, 900])  # the register schedule and the streaming schedule
@pytest.mark.parametrize("flags", [K.KDA_DECODE_L2NORM_QK, K.KDA_DECODE_BETA_LOGITS,
                                   K.KDA_DECODE_L2NORM_QK | K.KDA_DECODE_BETA_LOGITS])
def test_decode_input_options(rows, flags):
    """Raw N(0,1) q, k (normalised in the kernel when asked) and beta given as N(0,1) logits."""
    H = 2
    gen = torch.Generator(device="cpu").manual_seed(40 + rows + flags)
    q = torch.randn(rows, H, 128, generator=gen).to(torch.bfloat16)
    k = torch.randn(rows, H, 128, generator=gen).to(torch.bfloat16)
    if not flags & K.KDA_DECODE_L2NORM_QK:  # keep the state contractive without normalisation
        q = (q.float() / 11.3).to(torch.bfloat16)
        k = (k.float() / 11.3).to(torch.bfloat16)
    v = torch.randn(rows, H, 128, generator=gen).to(torch.bfloat16)
    g = torch.randn(rows, H, 128, generator=gen).to(torch.bfloat16)
    b = torch.randn(rows, H, generator=gen)
    if not flags & K.KDA_DECODE_BETA_LOGITS:
        b = torch.sigmoid(b)
    pool = S.state_pool(1024, H, "f32", std=0.02, seed=41, device=DEV)
    slots = S.slot_indices(rows, 1024, seed=41, device=DEV)
    before = pool[slots.long()].double().cpu()
    out = K.decode(*(t.to(DEV) for t in (q, k, v, g, b)), slots, pool, scale=SCALE, lower_bound=-5.0, flags=flags,
                   norm_eps=1e-6)
    assert K.kda_device_status()[0] == K.KDA_OK
    ref_out, ref_state, _ = oracle.decode(q, k, v, g, b, before, scale=SCALE, lower_bound=-5.0,
                                          norm_eps=1e-6 if flags & K.KDA_DECODE_L2NORM_QK else None,
                                          beta_logits=bool(flags & K.KDA_DECODE_BETA_LOGITS))
    assert_out_close(out.cpu(), ref_out)
    assert_state_close(pool[slots.long()].cpu(), ref_state)


def test_decode_and_windowed_prefill_replay_in_a_cuda_graph():
    """Captured once, replayed twice: the same bytes as eager calls on the same inputs."""
    H, rows = 8, 700
    d = S.decode_inputs(rows, H, seed=42, device=DEV)
    slots = S.slot_indices(rows, 4096, seed=42, device=DEV)
    pool0 = S.state_pool(4096, H, "f32", std=0.02, seed=42, device=DEV)
    p = S.prefill_inputs([2048], 4, seed=43, init_std=0.02, device=DEV)
    ws = K.prefill_workspace(1, 2048, 4, DEV)
    out_p, fin_p = torch.empty_like(p["q"]), torch.empty_like(p["init_state"])
    out_d = torch.empty_like(d["q"])

    def step(pool):
        K.kda_prefill_ex(p["q"], p["k"], p["v"], p["g_raw"], p["beta"], p["cu_seqlens"], p["init_state"], out_p,
                         fin_p, SCALE, -5.0, workspace=ws)
        K.kda_decode(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], slots, pool, out_d, SCALE, -5.0)

    eager_pool = pool0.clone()
    step(eager_pool)                      # first calls (one-time set-up) happen before capture
    eager = (out_p.clone(), fin_p.clone(), out_d.clone(), eager_pool.clone())
    graph_pool = pool0.clone()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=s):
            step(graph_pool)
    for _ in range(2):
        graph_pool.copy_(pool0)
        out_p.zero_(), fin_p.zero_(), out_d.zero_()
        gph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_p, eager[0]) and torch.equal(fin_p, eager[1]) and torch.equal(out_d, eager[2])
        assert torch.equal(graph_pool, eager[3])
    assert K.kda_device_status()[0] == K.KDA_OK


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,tokens", [(3, 2), (600, 2), (200, 3), (200, 4), (40, 5), (300, 16), (900, 7)])
def test_multi_token_decode_equals_prefill_of_short_sequences(state_dtype, rows, tokens):
    """T tokens per row applied in order to the row's slot: the oracle's prefill of T-token
    sequences started from the gathered pool states. Row 1 is a padding row. (900, 7) gives
    each CTA of the streaming schedule a dozen items with 3-15 tokens each, so every ring
    stage is refilled several times. BF16 states take the two-group layout up to 3 tokens
    per row and the register layout from 4, so (200, 3) and (200, 4) straddle the switch."""
    H, slots_n = 2, 2048
    p = S.prefill_inputs([tokens] * rows, H, seed=50 + rows + tokens, init_std=None)
    shape4 = (rows, tokens, H, 128)
    q, k, v, g = (p[n].reshape(shape4).contiguous() for n in ("q", "k", "v", "g_raw"))
    beta = p["beta"].reshape(rows, tokens, H).contiguous()
    pool = S.state_pool(slots_n, H, state_dtype, std=0.02, seed=51, device=DEV)
    slots = S.slot_indices(rows, slots_n, seed=51, device=DEV)
    if rows > 1:
        slots[1] = -1
    before = pool.clone()
    out = torch.empty(shape4, dtype=torch.bfloat16, device=DEV)
    K.kda_decode_ex(*(t.to(DEV) for t in (q, k, v, g, beta)), slots, pool, out, SCALE, -5.0)
    assert K.kda_device_status()[0] == K.KDA_OK
    live = torch.ones(rows, dtype=torch.bool)
    if rows > 1:
        live[1] = False
        assert torch.count_nonzero(out[1]) == 0
    sl = slots.cpu()[live].long()
    init = before[sl.to(DEV)].double().cpu()
    n_live = int(live.sum())
    cu = torch.arange(0, (n_live + 1) * tokens, tokens, dtype=torch.int32)
    flat = lambda t: t[live].reshape(n_live * tokens, H, *t.shape[3:]) if t.dim() == 4 else \
        t[live].reshape(n_live * tokens, H)
    ref_out, ref_fin, _ = oracle.prefill(flat(q), flat(k), flat(v), flat(g), flat(beta), cu, init, scale=SCALE,
                                         lower_bound=-5.0)
    assert_out_close(out.cpu()[live].reshape(n_live * tokens, H, 128), ref_out)
    assert_state_close(pool[sl.to(DEV)].cpu(), ref_fin)
    restored = pool.clone()
    restored[sl.to(DEV)] = before[sl.to(DEV)]
    assert torch.equal(bits(restored), bits(before)), "a slot outside the live rows changed"


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,tokens", [(900, 3), (50, 8)])
def test_multi_token_decode_with_input_options(state_dtype, rows, tokens):
    """Several tokens per row with q/k normalised in the kernel and beta given as logits: the
    oracle's decode applied token by token, the state carried between tokens."""
    H = 2
    gen = torch.Generator(device="cpu").manual_seed(60 + rows + tokens)
    shape4 = (rows, tokens, H, 128)
    q, k, v, g = (torch.randn(shape4, generator=gen).to(torch.bfloat16) for _ in range(4))
    b = torch.randn(rows, tokens, H, generator=gen)
    flags = K.KDA_DECODE_L2NORM_QK | K.KDA_DECODE_BETA_LOGITS
    pool = S.state_pool(2048, H, state_dtype, std=0.02, seed=61, device=DEV)
    slots = S.slot_indices(rows, 2048, seed=61, device=DEV)
    state = pool[slots.long()].double().cpu()
    out = torch.empty(shape4, dtype=torch.bfloat16, device=DEV)
    K.kda_decode_ex(*(t.to(DEV) for t in (q, k, v, g, b)), slots, pool, out, SCALE, -5.0, flags=flags, norm_eps=1e-6)
    assert K.kda_device_status()[0] == K.KDA_OK
    outs = []
    for t in range(tokens):
        o, state, _ = oracle.decode(q[:, t], k[:, t], v[:, t], g[:, t], b[:, t], state, scale=SCALE, lower_bound=-5.0,
                                    norm_eps=1e-6, beta_logits=True)
        outs.append(o)
    assert_out_close(out.cpu().transpose(0, 1).reshape(tokens * rows, H, 128),
                     torch.stack([torch.as_tensor(o) for o in outs]).reshape(tokens * rows, H, 128))
    assert_state_close(pool[slots.long()].cpu(), state)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("gate_mode", ["lower_bound", "softplus", "log_decay"])
def test_multi_token_decode_extreme_gates(state_dtype, gate_mode):
    """16 tokens per row with gates whose per-channel decay products leave [2^-60, 2^60] within
    the row, so that a kernel that defers the decay to the end of the row has to fold it into
    the state mid-row: lower bound -8 with saturated gates (a decay product below 2^-60 after 6
    tokens); softplus gates of 60 (e^-60 in one token) and 200 (a decay that underflows FP32);
    log-decay gates alternating +45 / -45 on channels whose k and q are zero (the row grows
    past 2^60 and shrinks back without reaching any output). The oracle's decode applied token
    by token, in FP64."""
    H, rows, tokens = 4, 300, 16
    gen = torch.Generator(device="cpu").manual_seed(70)
    shape4 = (rows, tokens, H, 128)
    q, k, v = (torch.randn(shape4, generator=gen) for _ in range(3))
    g = torch.randn(shape4, generator=gen)
    lb = 0.0
    if gate_mode == "lower_bound":
        lb = -8.0
        g[..., :64] = 8.0
    elif gate_mode == "softplus":
        g[:, 2::5, :, :32] = 60.0
        g[:, 3::7, :, 32:40] = 200.0
    else:
        g = -0.3 * g.abs()
        sign = torch.tensor([45.0 if t % 2 == 0 else -45.0 for t in range(tokens)])
        g[..., 100:104] = sign.view(1, tokens, 1, 1)
        q[..., 100:104] = 0.0
        k[..., 100:104] = 0.0
    # unit q and k per token (zero rows stay zero), as the model's normalised projections
    q, k = (x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6) for x in (q, k))
    q, k, v, g = (t.to(torch.bfloat16) for t in (q, k, v, g))
    b = torch.rand(rows, tokens, H, generator=gen)
    pool = S.state_pool(1024, H, state_dtype, std=0.02, seed=71, device=DEV)
    slots = S.slot_indices(rows, 1024, seed=71, device=DEV)
    state = pool[slots.long()].double().cpu()
    out = torch.empty(shape4, dtype=torch.bfloat16, device=DEV)
    K.kda_decode_ex(*(t.to(DEV) for t in (q, k, v, g, b)), slots, pool, out, SCALE, lb, gate_mode=gate_mode)
    assert K.kda_device_status()[0] == K.KDA_OK
    outs = []
    for t in range(tokens):
        o, state, _ = oracle.decode(q[:, t], k[:, t], v[:, t], g[:, t], b[:, t], state, scale=SCALE, lower_bound=lb,
                                    gate_mode=gate_mode)
        outs.append(o)
    assert_out_close(out.cpu().transpose(0, 1).reshape(tokens * rows, H, 128),
                     torch.stack([torch.as_tensor(o) for o in outs]).reshape(tokens * rows, H, 128))
    assert_state_close(pool[slots.long()].cpu(), state)
