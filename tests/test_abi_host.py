"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, exports
every entry point include/kda.h declares, and rejects bad arguments before any CUDA call.

Pointer arguments here are plain integers that are never dereferenced: every case
below fails validation on the host, which happens before the library touches the
device.
"""
import ctypes
import os
import re

import pytest
import torch

import kda_recurrent_gb300 as K
from kda_recurrent_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return K.load()


def declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)))


def test_header_declares_the_bound_entry_points():
    assert declared_entry_points() == sorted(K.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_abi_version_and_status_strings(lib):
    assert lib.kda_abi_version() >> 16 == 1
    for code in (0, -1, -2, -3, -4, -5, -6, 99):
        assert isinstance(K.kda_status_string(code), str) and K.kda_status_string(code)
    assert K.kda_status_string(K.KDA_ERR_MISALIGNED) == "misaligned pointer"


A16 = 0x10000  # a 16-byte-aligned fake address (never dereferenced)


def prefill_call(lib, **over):
    args = dict(q=A16, k=A16, v=A16, g=A16, beta=A16, cu=A16, init=None, out=A16, fin=None, N=1, T=32, H=2,
                scale=0.1, lb=-5.0, mode=0)
    args.update(over)
    return lib.kda_prefill(args["q"], args["k"], args["v"], args["g"], args["beta"], args["cu"], args["init"],
                           args["out"], args["fin"], args["N"], args["T"], args["H"], args["scale"], args["lb"],
                           args["mode"], None)


def decode_call(lib, **over):
    args = dict(q=A16, k=A16, v=A16, g=A16, beta=A16, slots=A16, pool=A16, S=16, dt=0, out=A16, R=4, H=2,
                scale=0.1, lb=-5.0, mode=0)
    args.update(over)
    return lib.kda_decode(args["q"], args["k"], args["v"], args["g"], args["beta"], args["slots"], args["pool"],
                          args["S"], args["dt"], args["out"], args["R"], args["H"], args["scale"], args["lb"],
                          args["mode"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(H=0), K.KDA_ERR_INVALID_ARG),
    (dict(N=-1), K.KDA_ERR_INVALID_ARG),
    (dict(T=-5), K.KDA_ERR_INVALID_ARG),
    (dict(mode=3), K.KDA_ERR_INVALID_ARG),
    (dict(lb=1.0), K.KDA_ERR_INVALID_ARG),
    (dict(lb=float("nan")), K.KDA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), K.KDA_ERR_INVALID_ARG),
    (dict(q=None), K.KDA_ERR_INVALID_ARG),
    (dict(out=None), K.KDA_ERR_INVALID_ARG),
    (dict(cu=None), K.KDA_ERR_INVALID_ARG),
    (dict(N=0, T=5), K.KDA_ERR_INVALID_ARG),
    (dict(q=A16 + 8), K.KDA_ERR_MISALIGNED),
    (dict(out=A16 + 2), K.KDA_ERR_MISALIGNED),
    (dict(fin=A16 + 4), K.KDA_ERR_MISALIGNED),
    (dict(beta=A16 + 2), K.KDA_ERR_MISALIGNED),
    (dict(N=0, T=0), K.KDA_OK),
    (dict(T=0, fin=None), K.KDA_OK),
])
def test_prefill_rejects_bad_arguments_on_host(lib, over, expect):
    assert prefill_call(lib, **over) == expect


def test_prefill_ex_rejects_misaligned_workspace_on_host(lib):
    r = lib.kda_prefill_ex(A16, A16, A16, A16, A16, A16, None, A16, None, 1, 32, 2, 0.1, -5.0, 0, None, None, 0, 0,
                           A16 + 8, 1 << 20, None)
    assert r == K.KDA_ERR_MISALIGNED


@pytest.mark.parametrize("every,ck,offs,rows,expect", [(48, A16, A16, 4, K.KDA_ERR_INVALID_ARG),
                                                        (-32, A16, A16, 4, K.KDA_ERR_INVALID_ARG),
                                                        (64, None, A16, 4, K.KDA_ERR_INVALID_ARG),
                                                        (64, A16, None, 4, K.KDA_ERR_INVALID_ARG),
                                                        (64, A16, A16, 0, K.KDA_ERR_INVALID_ARG),
                                                        (64, A16 + 4, A16, 4, K.KDA_ERR_MISALIGNED)])
def test_prefill_ex_checkpoint_arguments_on_host(lib, every, ck, offs, rows, expect):
    r = lib.kda_prefill_ex(A16, A16, A16, A16, A16, A16, None, A16, None, 1, 32, 2, 0.1, -5.0, 0, ck, offs, rows, every,
                           None, 0, None)
    assert r == expect


@pytest.mark.parametrize("over,expect", [
    (dict(H=0), K.KDA_ERR_INVALID_ARG),
    (dict(R=-1), K.KDA_ERR_INVALID_ARG),
    (dict(S=0), K.KDA_ERR_INVALID_ARG),
    (dict(dt=2), K.KDA_ERR_INVALID_ARG),
    (dict(mode=-1), K.KDA_ERR_INVALID_ARG),
    (dict(lb=0.5), K.KDA_ERR_INVALID_ARG),
    (dict(pool=None), K.KDA_ERR_INVALID_ARG),
    (dict(slots=None), K.KDA_ERR_INVALID_ARG),
    (dict(pool=A16 + 4), K.KDA_ERR_MISALIGNED),
    (dict(v=A16 + 1), K.KDA_ERR_MISALIGNED),
    (dict(slots=A16 + 2), K.KDA_ERR_MISALIGNED),
    (dict(R=0), K.KDA_OK),
])
def test_decode_rejects_bad_arguments_on_host(lib, over, expect):
    assert decode_call(lib, **over) == expect


@pytest.mark.parametrize("flags,eps,expect", [(4, 0.0, K.KDA_ERR_INVALID_ARG), (1, -1.0, K.KDA_ERR_INVALID_ARG),
                                              (1, float("nan"), K.KDA_ERR_INVALID_ARG), (2, -1.0, K.KDA_OK),
                                              (3, 1e-6, K.KDA_OK)])
def test_decode_ex_flag_validation_on_host(lib, flags, eps, expect):
    # rows = 0 makes valid calls a no-op that never touches the device
    r = lib.kda_decode_ex(A16, A16, A16, A16, A16, A16, A16, 16, 0, A16, 0, 1, 2, 0.1, -5.0, 0, flags, eps, None)
    assert r == expect


@pytest.mark.parametrize("tokens,expect", [(0, K.KDA_ERR_INVALID_ARG), (-2, K.KDA_ERR_INVALID_ARG),
                                           (17, K.KDA_ERR_UNSUPPORTED), (16, K.KDA_OK), (1, K.KDA_OK)])
def test_decode_tokens_per_row_validation_on_host(lib, tokens, expect):
    r = lib.kda_decode_ex(A16, A16, A16, A16, A16, A16, A16, 16, 0, A16, 0, tokens, 2, 0.1, -5.0, 0, 0, 0.0, None)
    assert r == expect


def test_binding_checks_dtypes_and_shapes_before_calling(lib):
    q = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    beta = torch.zeros(4, 2)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(TypeError):
        K.kda_prefill(q.float(), q, q, q, beta, cu, None, q, None, 0.1)
    with pytest.raises(ValueError):
        K.kda_prefill(q, q, q, q, beta[:3], cu, None, q, None, 0.1)
    with pytest.raises(TypeError):
        K.kda_decode(q, q, q, q, beta, torch.zeros(4, dtype=torch.int64), torch.zeros(8, 2, 128, 128), q, 0.1)
    with pytest.raises(ValueError, match="CUDA device"):  # host tensors never reach the library
        K.kda_prefill(q, q, q, q, beta, cu, None, q, None, 0.1)


def test_product_path_has_no_fallback(monkeypatch, tmp_path):
    """Without the built library the binding raises; nothing else computes."""
    monkeypatch.setattr(kbuild, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(K, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        K.load()


def flags(chains, wins):
    """Bytes of the per-window map flags after the state slots (one int32 per window, 256-byte padded)."""
    return (chains * wins * 4 + 255) // 256 * 256


def test_window_plan_on_host(lib):
    """kda_prefill_workspace_size with an explicit SM count is host arithmetic only."""
    slot = 128 * 128 * 4  # one FP32 state; a chain with W windows keeps 3 W - 5 of them
    size = K.kda_prefill_workspace_size
    assert size(1, 8192, 8, sm_count=152) == 8 * 55 * slot + flags(8, 20)    # 8 chains x 20 windows
    assert size(1, 512, 8, sm_count=152) == 8 * 7 * slot + flags(8, 4)      # 16 chunks: 4 windows of 4
    assert size(16, 25729, 32, sm_count=152) == 0                           # 512 chains fill the GPU
    assert size(8, 131072, 96, sm_count=152) == 8 * 55 * slot + flags(8, 20)  # 5 full waves + 8 chains
    assert size(2, 8192, 76, sm_count=152) == 0                             # exactly one full wave
    assert size(1, 8192, 204, sm_count=152) == 0                            # 52-chain tail: > a third
    assert size(1, 8192, 202, sm_count=152) == 50 * 7 * slot + flags(50, 4)  # 50-chain tail, 4 windows
    assert size(1, 64, 1, sm_count=152) == 0                               # 2 chunks: no windows
    # a small GPU: W = min(SMs / tail + 1, chunks / 4) windows for a tail of at most SMs / 3
    assert size(1, 1024, 1, sm_count=8) == 1 * 19 * slot + flags(1, 8)      # W = 8
    assert size(3, 3000, 1, sm_count=8) == 0                               # tail 3 > 8 / 3
    assert size(10, 64000, 1, sm_count=8) == 2 * 10 * slot + flags(2, 5)    # 8 + 2 chains, W = 5
    assert K.kda_prefill_workspace_size(1, 352, 2, sm_count=152) == 0                 # 11 chunks: W would be 2
    assert K.kda_prefill_workspace_size(0, 0, 1, sm_count=152) == 0
    with pytest.raises(K.KdaError):
        K.kda_prefill_workspace_size(1, 100, 0, sm_count=152)
    with pytest.raises(K.KdaError):
        K.kda_prefill_workspace_size(1, 100, 1, sm_count=-1)


def test_noalloc_scratch_bound_on_host(lib):
    """Every window plan needs at most 3 SMs - 2 FP32 states (and under 1 KiB of map flags), so
    the fixed 32 MiB array of kda_prefill_noalloc holds every plan on GPUs of up to 171 SMs
    (host arithmetic only)."""
    slot = 128 * 128 * 4
    for sms in (8, 76, 148, 152, 160, 171):
        worst = 0
        for tail in range(1, sms // 3 + 1):
            # `tail` chains left over past full waves, each long enough for sms / tail + 1 windows
            seqs = sms + tail
            toks = seqs * (sms // tail + 1) * 4 * 32
            worst = max(worst, K.kda_prefill_workspace_size(seqs, toks, 1, sm_count=sms))
        assert worst == (3 * sms - 2) * slot + flags(1, sms + 1), sms  # reached by a tail of one chain
        assert worst <= K.KDA_NOALLOC_SCRATCH_BYTES
    assert (3 * 172 - 2) * slot > K.KDA_NOALLOC_SCRATCH_BYTES
