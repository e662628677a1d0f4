"""Debug-build checks on the GPU, in place of a memory checker (compute-sanitizer is not
available here): a build of the same sources with KDA_DEBUG_CHECKS compares every decode row's
slot with the earlier rows' and records a repeated slot as KDA_ERR_DEVICE_INPUT, with the later
row as its detail. The product library never runs that check; this test builds its own copy,
in a folder of its own, and calls it through the C ABI.
"""
import ctypes
import os

import pytest
import torch

import kda_recurrent_gb300 as K
import kda_synth as S
from kda_recurrent_gb300 import build as kbuild

pytestmark = pytest.mark.gpu
DEV = "cuda"
DEBUG_LIB = os.path.join(kbuild.BUILD_DIR, "debug_checks", "libkda_gb300_debug_checks.so")


@pytest.fixture(scope="module")
def dlib():
    path = kbuild.build(extra_flags=["-DKDA_DEBUG_CHECKS"], lib_path=DEBUG_LIB)
    return K.bind(ctypes.CDLL(path))


def p(t):
    return ctypes.c_void_p(t.data_ptr())


def decode_status(lib, rows, slots, state_dtype="f32", H=8):
    pool = S.state_pool(64 if rows < 64 else 2 * rows, H, state_dtype, std=0.02, seed=61, device=DEV)
    d = S.decode_inputs(rows, H, seed=61, device=DEV)
    out = torch.empty_like(d["q"])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.kda_decode(p(d["q"]), p(d["k"]), p(d["v"]), p(d["g_raw"]), p(d["beta"]), p(slots), p(pool),
                        pool.shape[0], K.STATE_DTYPES[state_dtype], p(out), rows, H, S.DEFAULT_SCALE, -5.0, 0, stream)
    assert st == K.KDA_OK
    detail = ctypes.c_int32(0)
    code = lib.kda_device_status(stream, ctypes.byref(detail))
    assert torch.isfinite(out.float()).all()
    return code, detail.value


@pytest.mark.parametrize("rows", [6, 40, 1200])  # register kernel (16- and 64-column blocks); streaming
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_repeated_slot_is_reported_by_the_debug_build(dlib, rows, state_dtype):
    slots = torch.arange(rows, dtype=torch.int32, device=DEV)
    assert decode_status(dlib, rows, slots, state_dtype) == (K.KDA_OK, 0)
    dup = rows - 2
    slots[dup] = slots[1]
    assert decode_status(dlib, rows, slots, state_dtype) == (K.KDA_ERR_DEVICE_INPUT, dup)


def test_repeated_padding_rows_are_not_duplicates(dlib):
    slots = torch.tensor([-1, 3, -1, 5, -7, 0], dtype=torch.int32, device=DEV)
    assert decode_status(dlib, 6, slots) == (K.KDA_OK, 0)
