"""Host-side pieces of bench.py that need no GPU: argument parsing, the synthetic workloads'
shapes and the algorithmic byte counts behind the roofline fractions."""
import json

import pytest

import bench
import kda_synth as S


def test_options_parse():
    a = bench.parse_args(["--decode-tokens", "4", "--ckpt-every", "64", "--state-dtype", "bf16"])
    assert a.decode_tokens == 4 and a.ckpt_every == 64 and a.state_dtype == "bf16"
    d = bench.parse_args([])
    assert d.gpus == 1 and d.decode_tokens == 1 and d.ckpt_every == 0 and d.warmup >= 3


def test_decode_bytes_count_state_both_ways_and_each_token_row():
    # FP32 state read and written, the q, k, v, g_raw rows, beta and the output per token,
    # and one slot index per row
    assert bench.decode_bytes(4096, 8, "f32") == 4096 * 8 * (2 * 65536 + 1284) + 4096 * 4
    assert bench.decode_bytes(10, 2, "bf16") == 10 * 2 * (2 * 32768 + 1284) + 40
    assert bench.decode_bytes(10, 2, "f32", tokens=3) == 10 * 2 * (2 * 65536 + 3 * 1284) + 40


def test_prefill_bytes_count_tokens_and_states():
    cfg = S.configs()["prefill_h8_t8192"]
    chains = len(cfg.seqlens) * cfg.num_heads
    states = 2 if cfg.init_std is not None else 1
    assert bench.prefill_bytes(cfg) == cfg.total_tokens * cfg.num_heads * 1284 + chains * states * 65536


@pytest.mark.parametrize("tokens", [1, 3])
def test_decode_workload_shapes(tokens):
    cfg, pool, inp = bench.decode_workload(6, "f32", "cpu", pool_slots=32, tokens=tokens)
    H = cfg.num_heads
    tok = (6, H, 128) if tokens == 1 else (6, tokens, H, 128)
    for k in ("q", "k", "v", "g_raw"):
        assert tuple(inp[k].shape) == tok and inp[k].is_contiguous()
    assert tuple(inp["beta"].shape) == tok[:-1]
    assert tuple(inp["slot_idx"].shape) == (6,) and len(set(inp["slot_idx"].tolist())) == 6
    assert tuple(pool.shape) == (32, H, 128, 128)


def test_decode_kernel_choice_follows_the_library_thresholds():
    assert bench.decode_kernel_name(4 * 152, 152) == "kda_decode_stream_kernel"
    assert bench.decode_kernel_name(4 * 152 - 1, 152) == "kda_decode_kernel"
    assert bench.decode_kernel_name(3 * 152, 152, "bf16") == "kda_decode_stream_kernel"
    assert bench.decode_kernel_name(3 * 152 - 1, 152, "bf16") == "kda_decode_kernel"


def test_traffic_record_matches_the_kernel_sources():
    """Every per-unit DRAM figure in profiles/traffic.json is keyed to the SHA-256 of its
    kernel source; bench.py drops a figure whose source has changed since the capture."""
    t = bench.load_traffic()
    with open(bench.os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        raw = json.load(f)
    for name, rec in raw.items():
        assert rec["unit"] in ("token*head", "row*head")
        assert rec["dram_bytes_per_unit"] > 0
        if rec["source_sha256_16"] == bench.source_digest(rec["source"]):
            assert bench.scaled_traffic(t, name, 10) == pytest.approx(10 * rec["dram_bytes_per_unit"], rel=1e-6)
        else:
            assert bench.scaled_traffic(t, name, 10) is None


def test_decode_flag_names():
    assert bench.decode_flags("") == 0
    assert bench.decode_flags("l2norm") == 1
    assert bench.decode_flags("beta_logits, l2norm") == 3
    with pytest.raises(SystemExit):
        bench.decode_flags("l2norm,unknown")
