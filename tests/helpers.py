"""Test helpers: parity metrics, tolerances and oracle runs on head/sequence subsets."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

# Tolerances against the FP64 oracle (BF16 inputs/outputs, FP32 state).
OUT_REL_L2 = 1e-2
OUT_MAX_ABS = 3e-2
STATE_REL_L2 = 2e-3


def to_np(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def rel_l2(got, ref) -> float:
    got, ref = to_np(got), to_np(ref)
    den = math.sqrt(float(np.sum(ref * ref)))
    num = math.sqrt(float(np.sum((got - ref) ** 2)))
    return num / den if den > 0 else num


def max_abs(got, ref) -> float:
    got, ref = to_np(got), to_np(ref)
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


def assert_out_close(got, ref, what="out"):
    r, m = rel_l2(got, ref), max_abs(got, ref)
    assert np.all(np.isfinite(to_np(got))), f"{what}: non-finite values"
    assert r <= OUT_REL_L2 and m <= OUT_MAX_ABS, f"{what}: relL2 {r:.3e} (<= {OUT_REL_L2}), max-abs {m:.3e} (<= {OUT_MAX_ABS})"
    return r, m


def assert_state_close(got, ref, what="state", tol=STATE_REL_L2):
    r = rel_l2(got, ref)
    assert np.all(np.isfinite(to_np(got))), f"{what}: non-finite values"
    assert r <= tol, f"{what}: relL2 {r:.3e} (<= {tol})"
    return r


def slice_problem(inp: dict, heads=None, seqs=None) -> dict:
    """The sub-problem of ``inp`` restricted to some heads and/or sequences (CPU tensors)."""
    cu = inp["cu_seqlens"].to("cpu").to(torch.int64)
    N = cu.shape[0] - 1
    seqs = list(range(N)) if seqs is None else list(seqs)
    H = inp["q"].shape[1]
    heads = list(range(H)) if heads is None else list(heads)
    dev = inp["q"].device
    hidx = torch.tensor(heads, dtype=torch.int64, device=dev)
    tok = torch.cat([torch.arange(int(cu[n]), int(cu[n + 1])) for n in seqs]) if seqs else torch.zeros(0, dtype=torch.int64)
    tok_d = tok.to(dev)
    out = {}
    for key in ("q", "k", "v", "g_raw", "beta"):
        out[key] = inp[key].index_select(1, hidx).index_select(0, tok_d).to("cpu").contiguous()
    lens = [int(cu[n + 1] - cu[n]) for n in seqs]
    cuts = [0]
    for n in lens:
        cuts.append(cuts[-1] + n)
    out["cu_seqlens"] = torch.tensor(cuts, dtype=torch.int32)
    init = inp.get("init_state")
    out["init_state"] = None if init is None else init[seqs][:, heads].to("cpu").contiguous()
    out["token_index"] = tok
    return out


def oracle_prefill(inp: dict, *, scale, lower_bound, gate_mode, threads=0):
    """FP64 oracle on a (sub-)problem dict as produced by kda_synth / slice_problem."""
    out, fin, _ = oracle.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                                 inp.get("init_state"), scale=scale, lower_bound=lower_bound, gate_mode=gate_mode,
                                 threads=threads)
    return out, fin


def launch_order(seqlens, num_heads, ranked_max=256):
    """(sequence, head) of each launch position of the prefill: head p % H of the sequence
    ranked p // H by length, longest first, ties by index (batches of more than
    ``ranked_max`` sequences keep index order). The windowed tail of kda_prefill_ex is the
    last ``chains % SMs`` positions."""
    N = len(seqlens)
    ranked = list(range(N))
    if 1 < N <= ranked_max:
        ranked.sort(key=lambda n: (-seqlens[n], n))
    return [(ranked[p // num_heads], p % num_heads) for p in range(N * num_heads)]
