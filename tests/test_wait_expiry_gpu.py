"""Failure detection on the GPU without a fault: every device-side wait of the library is
bounded, and a CTA whose wait runs out records KDA_ERR_DEVICE_TIMEOUT, waits (bounded) for
its own copies and tensor-core work in flight, frees its tensor memory and returns.

None of the product library's waits ever runs out (its limit is 2 s), so this test builds a
separate copy of the same sources -- never the product library -- with a 1 ms limit and one
hand-off withheld at compile time: in the prefill the solve warps never release chunk 3 to
the state warps; in the streaming decode the producer never fills the fourth item of each
CTA. The waits for those hand-offs give up by design; nothing faults or hangs. The test
checks, through the C ABI, that the calls return, that the test library's status word
reports the timeout, and that the product library, called next in the same process, still
passes parity against the oracle: the aborted CTAs left the context usable and released
their tensor memory.
"""
import ctypes
import os
import time

import pytest
import torch

import kda_recurrent_gb300 as K
import kda_synth as S
from helpers import assert_out_close, assert_state_close, oracle_prefill
from kda_recurrent_gb300 import build as kbuild

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALE = S.DEFAULT_SCALE
WITHHELD = 3  # chunk (prefill) / local item (decode) whose hand-off the test build drops
TEST_LIB = os.path.join(kbuild.BUILD_DIR, "wait_limit_test", "libkda_gb300_wait_limit_test.so")


@pytest.fixture(scope="module")
def tlib():
    path = kbuild.build(extra_flags=["-DKDA_WAIT_LIMIT_NS=1000000ull", f"-DKDA_TEST_WITHHOLD_HANDOFF={WITHHELD}"],
                        lib_path=TEST_LIB)
    assert os.path.abspath(path) != os.path.abspath(kbuild.LIB_PATH)
    return K.bind(ctypes.CDLL(path))


def p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def status(lib):
    detail = ctypes.c_int32(0)
    return lib.kda_device_status(stream(), ctypes.byref(detail)), detail.value


def prefill_raw(lib, inp, out, fin, workspace=None, lower_bound=-5.0):
    T, H, _ = inp["q"].shape
    N = inp["cu_seqlens"].shape[0] - 1
    ws_bytes = 0 if workspace is None else workspace.numel()
    return lib.kda_prefill_ex(p(inp["q"]), p(inp["k"]), p(inp["v"]), p(inp["g_raw"]), p(inp["beta"]),
                              p(inp["cu_seqlens"]), p(inp["init_state"]), p(out), p(fin), N, T, H, SCALE, lower_bound,
                              0, None, None, 0, 0, p(workspace), ws_bytes, stream())


def timed_sync():
    t0 = time.monotonic()
    torch.cuda.synchronize()
    return time.monotonic() - t0


def test_prefill_wait_expiry_is_reported_and_the_context_stays_usable(tlib):
    assert status(tlib)[0] == K.KDA_OK
    # a chain too short to reach the withheld hand-off runs normally in the test build
    inp = S.prefill_inputs([96], 2, seed=51, init_std=0.02, device=DEV)
    out, fin = torch.empty_like(inp["q"]), torch.empty_like(inp["init_state"])
    assert prefill_raw(tlib, inp, out, fin) == K.KDA_OK
    assert status(tlib)[0] == K.KDA_OK
    ref_out, ref_fin = oracle_prefill({k: v.cpu() for k, v in inp.items()}, scale=SCALE, lower_bound=-5.0,
                                      gate_mode="lower_bound")
    assert_out_close(out.cpu(), ref_out)
    assert_state_close(fin.cpu(), ref_fin)

    # 16 chunks per chain on the sequential schedule: every CTA gives up at chunk 3
    inp = S.prefill_inputs([512, 300], 2, seed=52, init_std=0.02, device=DEV)
    out, fin = torch.zeros_like(inp["q"]), torch.zeros_like(inp["init_state"])
    assert prefill_raw(tlib, inp, out, fin) == K.KDA_OK
    assert timed_sync() < 20.0
    st, detail = status(tlib)
    assert st == K.KDA_ERR_DEVICE_TIMEOUT, (st, detail)
    assert 0 <= detail < 4  # the CTA (chain) that recorded it first

    # the window schedule (window 0, window pass, carry, output pass): each window CTA of at
    # least 4 chunks gives up the same way
    inp = S.prefill_inputs([3000], 2, seed=53, init_std=0.02, device=DEV)
    n = tlib.kda_prefill_workspace_size(1, 3000, 2, 0)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    out, fin = torch.zeros_like(inp["q"]), torch.zeros_like(inp["init_state"])
    assert prefill_raw(tlib, inp, out, fin, workspace=ws) == K.KDA_OK
    assert timed_sync() < 20.0
    assert status(tlib)[0] == K.KDA_ERR_DEVICE_TIMEOUT
    assert status(tlib)[0] == K.KDA_OK  # read and cleared

    # the product library, next in the same process: unaffected, and parity holds
    inp = S.prefill_inputs([700, 64], 2, seed=54, init_std=0.02, device=DEV)
    out, fin = K.prefill(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["cu_seqlens"],
                         inp["init_state"], scale=SCALE, lower_bound=-5.0,
                         workspace=K.prefill_workspace(2, 764, 2, DEV))
    assert K.kda_device_status()[0] == K.KDA_OK
    ref_out, ref_fin = oracle_prefill({k: v.cpu() for k, v in inp.items()}, scale=SCALE, lower_bound=-5.0,
                                      gate_mode="lower_bound")
    assert_out_close(out.cpu(), ref_out)
    assert_state_close(fin.cpu(), ref_fin)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decode_wait_expiry_is_reported_and_the_context_stays_usable(tlib, state_dtype):
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    H = 8
    rows = 6 * sms // H + 8  # at least 6 (row, head) items per CTA: the streaming schedule
    pool = S.state_pool(rows + 16, H, state_dtype, std=0.02, seed=55, device=DEV)
    d = S.decode_inputs(rows, H, seed=55, device=DEV)
    slots = S.slot_indices(rows, rows + 16, seed=55, device=DEV)
    out = torch.zeros_like(d["q"])
    sdt = K.STATE_DTYPES[state_dtype]
    assert status(tlib)[0] == K.KDA_OK
    st = tlib.kda_decode(p(d["q"]), p(d["k"]), p(d["v"]), p(d["g_raw"]), p(d["beta"]), p(slots), p(pool),
                         pool.shape[0], sdt, p(out), rows, H, SCALE, -5.0, 0, stream())
    assert st == K.KDA_OK
    assert timed_sync() < 20.0
    assert status(tlib)[0] == K.KDA_ERR_DEVICE_TIMEOUT

    # the product library on the same pool afterwards: parity against the oracle
    pool = S.state_pool(rows + 16, H, state_dtype, std=0.02, seed=56, device=DEV)
    gathered = pool[slots.long()].double().cpu()
    o = K.decode(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], slots, pool, scale=SCALE, lower_bound=-5.0)
    assert K.kda_device_status()[0] == K.KDA_OK
    ro, rs, _ = oracle.decode(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], gathered, scale=SCALE,
                              lower_bound=-5.0)
    assert_out_close(o.cpu(), ro)
    assert_state_close(pool[slots.long()].cpu(), rs)
