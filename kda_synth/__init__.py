"""Seeded synthetic inputs for the KDA hot path, shared by the tests, the smoke check and the bench.

This module holds input recipes only -- none of the method's arithmetic. Both the
CUDA path and the oracle consume what it returns; neither is imported here.

Recipe (the pages' workloads are model-shaped K3 / Kimi-Linear layers with
d = 128; these five configurations stand in for them):
  * q, k: N(0, 1) in FP32, L2-normalised per (token, head) as x * (sum x^2 + 1e-6)^-1/2,
    then rounded to BF16 (round-to-nearest-even, torch's cast);
  * v: N(0, 1) rounded to BF16;  raw gate a: N(0, 1) rounded to BF16;
  * beta = sigmoid(N(0, 1)) kept in FP32 (post-sigmoid, in (0, 1));
  * initial states (when present) N(0, std^2) in FP32; the decode pool likewise,
    stored in the pool's dtype;
  * decode slots: the first ``rows`` entries of a seeded permutation of the pool.
Draw order is fixed (q, k, v, a, beta, then states), so one seed gives one input
set on a given generator device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

D = 128
DEFAULT_SCALE = 1.0 / math.sqrt(D)


@dataclass
class PrefillConfig:
    name: str
    seqlens: List[int]
    num_heads: int
    gate_mode: str
    lower_bound: float
    init_std: Optional[float]
    seed: int
    scale: float = DEFAULT_SCALE
    note: str = ""

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))


@dataclass
class DecodeConfig:
    name: str
    rows: List[int]
    num_heads: int
    num_slots: int
    gate_mode: str
    lower_bound: float
    pool_std: float
    seed: int
    state_dtypes: List[str] = field(default_factory=lambda: ["f32", "bf16"])
    scale: float = DEFAULT_SCALE
    note: str = ""


def varlen_lengths(count: int, lo: int, hi: int, seed: int) -> List[int]:
    """``count`` lengths drawn uniformly from [lo, hi] with a seeded CPU generator."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (count,), generator=gen)]


def _cfg3_lengths() -> List[int]:
    lens = varlen_lengths(16, 256, 4096, seed=2)
    assert any(n % 32 for n in lens), "the varlen workload must contain a ragged length"
    return lens


def configs():
    """The five workloads: three prefill shapes, the decode sweep and the large prefill."""
    return {
        "prefill_h1_t64": PrefillConfig("prefill_h1_t64", [64], 1, "lower_bound", -5.0, None, 0,
                                        note="1 seq, H1, T64 (2 chunks), lb=-5, zero initial state"),
        "prefill_h8_t8192": PrefillConfig("prefill_h8_t8192", [8192], 8, "lower_bound", -5.0, 0.02, 1,
                                          note="1 seq, H8 small-BH, T8192, lb=-5, initial state N(0,0.02)"),
        "prefill_varlen16_h32": PrefillConfig("prefill_varlen16_h32", _cfg3_lengths(), 32, "softplus", 0.0,
                                              None, 2,
                                              note="16 seqs, lengths U[256,4096], H32, softplus gate, zero init"),
        "decode_h8_pool16384": DecodeConfig("decode_h8_pool16384", [1 << i for i in range(13)], 8, 16384,
                                            "lower_bound", -5.0, 0.02, 3,
                                            note="T=1 decode, H8, rows 1..4096, 16384-slot pool"),
        "prefill_8x16384_h96": PrefillConfig("prefill_8x16384_h96", [16384] * 8, 96, "lower_bound", -8.0,
                                             0.02, 4,
                                             note="8 seqs x 16384, H96, lb=-8, initial state N(0,0.02)"),
    }


def _l2norm_bf16(x: torch.Tensor) -> torch.Tensor:
    return (x * torch.rsqrt((x * x).sum(-1, keepdim=True) + 1e-6)).to(torch.bfloat16)


def cu_seqlens_of(seqlens: List[int]) -> torch.Tensor:
    cu = [0]
    for n in seqlens:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def prefill_inputs(seqlens: List[int], num_heads: int, *, seed: int, init_std: Optional[float],
                   device="cpu", d: int = D):
    """Packed varlen prefill inputs: q, k, v, g_raw [T, H, d] BF16; beta [T, H] FP32;
    cu_seqlens [N+1] int32; init_state [N, H, d, d] FP32 or None."""
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(seed)
    T, H, N = int(sum(seqlens)), num_heads, len(seqlens)

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)

    q = _l2norm_bf16(randn(T, H, d))
    k = _l2norm_bf16(randn(T, H, d))
    v = randn(T, H, d).to(torch.bfloat16)
    g_raw = randn(T, H, d).to(torch.bfloat16)
    beta = torch.sigmoid(randn(T, H))
    init = None if init_std is None else randn(N, H, d, d) * init_std
    return {"q": q, "k": k, "v": v, "g_raw": g_raw, "beta": beta,
            "cu_seqlens": cu_seqlens_of(seqlens).to(device), "init_state": init}


def config_inputs(cfg: PrefillConfig, device="cpu"):
    return prefill_inputs(cfg.seqlens, cfg.num_heads, seed=cfg.seed, init_std=cfg.init_std, device=device)


def decode_inputs(rows: int, num_heads: int, *, seed: int, device="cpu", d: int = D):
    """Per-row decode inputs: q, k, v, g_raw [rows, H, d] BF16; beta [rows, H] FP32."""
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(seed * 7919 + rows)

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)

    return {"q": _l2norm_bf16(randn(rows, num_heads, d)), "k": _l2norm_bf16(randn(rows, num_heads, d)),
            "v": randn(rows, num_heads, d).to(torch.bfloat16),
            "g_raw": randn(rows, num_heads, d).to(torch.bfloat16),
            "beta": torch.sigmoid(randn(rows, num_heads))}


def slot_indices(rows: int, num_slots: int, *, seed: int, device="cpu") -> torch.Tensor:
    """``rows`` unique slots scattered uniformly over the pool (int32)."""
    gen = torch.Generator(device="cpu").manual_seed(seed * 104729 + rows)
    return torch.randperm(num_slots, generator=gen)[:rows].to(torch.int32).to(device)


def state_pool(num_slots: int, num_heads: int, state_dtype: str, *, std: float, seed: int, device="cpu",
               d: int = D) -> torch.Tensor:
    """[num_slots, H, d, d] pool filled with N(0, std^2), stored as FP32 or BF16."""
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(seed)
    dt = {"f32": torch.float32, "bf16": torch.bfloat16}[state_dtype]
    pool = torch.empty(num_slots, num_heads, d, d, dtype=dt, device=device)
    step = max(1, (1 << 28) // (num_heads * d * d))  # fill in slabs to bound the FP32 temporary
    for s in range(0, num_slots, step):
        e = min(num_slots, s + step)
        pool[s:e] = (torch.randn(e - s, num_heads, d, d, generator=gen, device=device) * std).to(dt)
    return pool
