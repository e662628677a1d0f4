"""GB300 (sm_103a) Kimi Delta Attention hot path: Python binding of the C ABI in ``include/kda.h``.

Every step of the computation runs in the CUDA library ``_build/libkda_gb300.so``;
this module only marshals arguments (dtype / shape / device checks, raw pointers,
the current CUDA stream). If the library is missing it raises -- there is no other
implementation behind these calls.

Low-level calls mirror the C names and take caller-owned torch tensors:
    kda_prefill(q, k, v, g_raw, beta, cu_seqlens, init_state, out, final_state, scale,
                lower_bound, gate_mode, stream=None)
    kda_decode(q, k, v, g_raw, beta, slot_idx, state_pool, out, scale, lower_bound,
               gate_mode, stream=None)
    kda_prefill_ex(..., workspace=None, stream=None), kda_prefill_workspace_size(N, T, H, sm_count=0)
    kda_status_string(status), kda_device_status(stream=None)
Convenience wrappers ``prefill`` / ``decode`` allocate the outputs.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_MISALIGNED = -3
KDA_ERR_CUDA = -4
KDA_ERR_DEVICE_TIMEOUT = -5
KDA_ERR_DEVICE_INPUT = -6

GATE_MODES = {"lower_bound": 0, "softplus": 1, "log_decay": 2}
STATE_DTYPES = {"f32": 0, "bf16": 1}
HEAD_DIM = 128
CHUNK = 32

EXPORTED_SYMBOLS = ("kda_prefill", "kda_prefill_ex", "kda_prefill_workspace_size", "kda_prefill_noalloc", "kda_decode",
                    "kda_decode_ex", "kda_status_string", "kda_device_status", "kda_abi_version")
KDA_NOALLOC_SCRATCH_BYTES = 32 << 20  # fixed scratch array of kda_prefill_noalloc
KDA_DECODE_L2NORM_QK = 1
KDA_DECODE_BETA_LOGITS = 2
KDA_DECODE_MAX_TOKENS = 16

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {kda_status_string(status)} ({status})")
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Load the CUDA library (building it first only if asked). Raises if it is absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(f"KDA CUDA library not built: {path} (run kda_recurrent_gb300.build.build())")
                _build.build()
            _lib = bind(ctypes.CDLL(path))
    return _lib


def bind(lib):
    """Declares the argument and result types of every C entry point on a loaded library
    handle (the product library, or a test build of the same sources)."""
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.kda_prefill.restype = ctypes.c_int
    lib.kda_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, f32, f32, i32, vp]
    lib.kda_prefill_ex.restype = ctypes.c_int
    lib.kda_prefill_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, f32, f32, i32, vp, vp,
                                   i64, i32, vp, i64, vp]
    lib.kda_prefill_workspace_size.restype = ctypes.c_int64
    lib.kda_prefill_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.kda_prefill_noalloc.restype = ctypes.c_int
    lib.kda_prefill_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, f32, f32, i32, vp]
    lib.kda_decode.restype = ctypes.c_int
    lib.kda_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, vp, i32, i32, f32, f32, i32, vp]
    lib.kda_decode_ex.restype = ctypes.c_int
    lib.kda_decode_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, vp, i32, i32, i32, f32, f32, i32, i32,
                                  f32, vp]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_device_status.restype = ctypes.c_int
    lib.kda_device_status.argtypes = [vp, ctypes.POINTER(i32)]
    lib.kda_abi_version.restype = ctypes.c_int
    lib.kda_abi_version.argtypes = []
    return lib


def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def _mode(gate_mode) -> int:
    return GATE_MODES[gate_mode] if isinstance(gate_mode, str) else int(gate_mode)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, shape, device):
    import torch
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    del torch


def _require_cuda(device):
    """Host tensors never reach the library: its kernels would read them as device addresses."""
    if device.type != "cuda":
        raise ValueError(f"tensors must be on a CUDA device, got {device}")


def kda_prefill(q, k, v, g_raw, beta, cu_seqlens, init_state, out, final_state, scale, lower_bound=0.0,
                gate_mode="lower_bound", stream=None):
    """Varlen chunk-32 prefill into caller-owned ``out`` / ``final_state`` (see include/kda.h)."""
    import torch
    T, H, d = q.shape
    N = cu_seqlens.shape[0] - 1
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g_raw", g_raw), ("out", out)):
        _check(t, name, torch.bfloat16, (T, H, d), dev)
    _check(beta, "beta", torch.float32, (T, H), dev)
    _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
    for name, t in (("init_state", init_state), ("final_state", final_state)):
        if t is not None:
            _check(t, name, torch.float32, (N, H, d, d), dev)
    _require_cuda(dev)
    with torch.cuda.device(dev):  # the library plans for, and launches on, the current device
        st = load().kda_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta), _ptr(cu_seqlens),
                                _ptr(init_state), _ptr(out), _ptr(final_state), N, T, H, float(scale),
                                float(lower_bound), _mode(gate_mode), _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill")


def kda_prefill_workspace_size(num_seqs, total_tokens, num_heads, sm_count=0) -> int:
    """Workspace bytes kda_prefill_ex uses for this shape (0: none); sm_count 0 asks the current device."""
    n = load().kda_prefill_workspace_size(int(num_seqs), int(total_tokens), int(num_heads), int(sm_count))
    if n < 0:
        raise KdaError(int(n), "kda_prefill_workspace_size")
    return int(n)


def kda_prefill_ex(q, k, v, g_raw, beta, cu_seqlens, init_state, out, final_state, scale, lower_bound=0.0,
                   gate_mode="lower_bound", workspace=None, stream=None, checkpoints=None, ckpt_offsets=None,
                   ckpt_every=0):
    """kda_prefill with a caller-owned device workspace (a uint8 tensor, or None) and optional
    intermediate states every ``ckpt_every`` tokens into ``checkpoints`` [rows, H, 128, 128] at
    rows ``ckpt_offsets[n] + j``."""
    import torch
    T, H, d = q.shape
    N = cu_seqlens.shape[0] - 1
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g_raw", g_raw), ("out", out)):
        _check(t, name, torch.bfloat16, (T, H, d), dev)
    _check(beta, "beta", torch.float32, (T, H), dev)
    _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
    for name, t in (("init_state", init_state), ("final_state", final_state)):
        if t is not None:
            _check(t, name, torch.float32, (N, H, d, d), dev)
    if ckpt_every:
        _check(ckpt_offsets, "ckpt_offsets", torch.int32, (N,), dev)
        _check(checkpoints, "checkpoints", torch.float32, (checkpoints.shape[0], H, d, d), dev)
    nbytes = 0
    if workspace is not None:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace: must be a contiguous tensor on the inputs' device")
        nbytes = workspace.numel() * workspace.element_size()
    _require_cuda(dev)
    with torch.cuda.device(dev):  # the window plan follows the current device's SM count
        st = load().kda_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta), _ptr(cu_seqlens),
                                   _ptr(init_state), _ptr(out), _ptr(final_state), N, T, H, float(scale),
                                   float(lower_bound), _mode(gate_mode), _ptr(checkpoints if ckpt_every else None),
                                   _ptr(ckpt_offsets if ckpt_every else None),
                                   int(checkpoints.shape[0]) if ckpt_every else 0, int(ckpt_every),
                                   _ptr(workspace), nbytes, _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_ex")


def kda_prefill_noalloc(q, k, v, g_raw, beta, cu_seqlens, init_state, out, final_state, scale, lower_bound=0.0,
                        gate_mode="lower_bound", stream=None):
    """The window-scheduled prefill without a caller workspace, for callers that cannot allocate
    device memory: the library's own fixed 32 MiB scratch array stands in for it. Calls share
    that array, so calls that overlap on the GPU must be serialised (see include/kda.h)."""
    import torch
    T, H, d = q.shape
    N = cu_seqlens.shape[0] - 1
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g_raw", g_raw), ("out", out)):
        _check(t, name, torch.bfloat16, (T, H, d), dev)
    _check(beta, "beta", torch.float32, (T, H), dev)
    _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
    for name, t in (("init_state", init_state), ("final_state", final_state)):
        if t is not None:
            _check(t, name, torch.float32, (N, H, d, d), dev)
    _require_cuda(dev)
    with torch.cuda.device(dev):  # the scratch array and the plan are those of the current device
        st = load().kda_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta), _ptr(cu_seqlens),
                                        _ptr(init_state), _ptr(out), _ptr(final_state), N, T, H, float(scale),
                                        float(lower_bound), _mode(gate_mode), _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_noalloc")


def prefill_workspace(num_seqs, total_tokens, num_heads, device):
    """A uint8 device tensor sized for kda_prefill_ex on `device` (None when no workspace is used)."""
    import torch
    with torch.cuda.device(device):
        n = kda_prefill_workspace_size(num_seqs, total_tokens, num_heads)
    return torch.empty(n, dtype=torch.uint8, device=device) if n > 0 else None


def kda_decode(q, k, v, g_raw, beta, slot_idx, state_pool, out, scale, lower_bound=0.0,
               gate_mode="lower_bound", stream=None):
    """T = 1 decode of ``rows`` tokens against ``state_pool`` (updated in place)."""
    _decode_call("kda_decode", q, k, v, g_raw, beta, slot_idx, state_pool, out, scale, lower_bound, gate_mode, 0,
                 0.0, stream)


def kda_decode_ex(q, k, v, g_raw, beta, slot_idx, state_pool, out, scale, lower_bound=0.0,
                  gate_mode="lower_bound", flags=0, norm_eps=0.0, stream=None):
    """Decode with T tokens per row (q, k, v, g_raw, out [R, T, H, 128]; beta [R, T, H]; 3-D
    tensors mean T = 1) and the input options KDA_DECODE_L2NORM_QK (with ``norm_eps``) and
    KDA_DECODE_BETA_LOGITS."""
    _decode_call("kda_decode_ex", q, k, v, g_raw, beta, slot_idx, state_pool, out, scale, lower_bound, gate_mode,
                 flags, norm_eps, stream)


def _decode_call(name, q, k, v, g_raw, beta, slot_idx, state_pool, out, scale, lower_bound, gate_mode, flags,
                 norm_eps, stream):
    import torch
    if q.dim() == 3:
        R, H, d = q.shape
        T = 1
        tok_shape, beta_shape = (R, H, d), (R, H)
    else:
        R, T, H, d = q.shape
        tok_shape, beta_shape = (R, T, H, d), (R, T, H)
        if name == "kda_decode":
            raise ValueError("kda_decode takes one token per row; use kda_decode_ex")
    dev = q.device
    for nm, t in (("q", q), ("k", k), ("v", v), ("g_raw", g_raw), ("out", out)):
        _check(t, nm, torch.bfloat16, tok_shape, dev)
    _check(beta, "beta", torch.float32, beta_shape, dev)
    _check(slot_idx, "slot_idx", torch.int32, (R,), dev)
    if state_pool.dtype == torch.float32:
        sdt = STATE_DTYPES["f32"]
    elif state_pool.dtype == torch.bfloat16:
        sdt = STATE_DTYPES["bf16"]
    else:
        raise TypeError("state_pool must be float32 or bfloat16")
    _check(state_pool, "state_pool", state_pool.dtype, (state_pool.shape[0], H, d, d), dev)
    lib = load()
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta), _ptr(slot_idx), _ptr(state_pool),
            int(state_pool.shape[0]), sdt, _ptr(out), R)
    tail = (float(scale), float(lower_bound), _mode(gate_mode))
    _require_cuda(dev)
    with torch.cuda.device(dev):  # the schedule follows the current device's SM count
        if name == "kda_decode":
            st = lib.kda_decode(*head, H, *tail, _stream_handle(stream, dev))
        else:
            st = lib.kda_decode_ex(*head, T, H, *tail, int(flags), float(norm_eps), _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, name)


def kda_device_status(stream=None):
    """(status, detail): reads and clears the device status word (synchronises the stream)."""
    import torch
    detail = ctypes.c_int32(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    st = load().kda_device_status(_stream_handle(stream, dev), ctypes.byref(detail))
    return st, detail.value


def prefill(q, k, v, g_raw, beta, cu_seqlens, init_state=None, *, scale, lower_bound=0.0,
            gate_mode="lower_bound", want_final=True, workspace=None, stream=None):
    """Allocates ``out`` (and ``final_state``) and runs ``kda_prefill`` (``kda_prefill_ex`` when a
    workspace is given); returns (out, final_state)."""
    import torch
    T, H, d = q.shape
    N = cu_seqlens.shape[0] - 1
    out = torch.empty_like(q)
    final = torch.empty(N, H, d, d, dtype=torch.float32, device=q.device) if want_final else None
    if workspace is None:
        kda_prefill(q, k, v, g_raw, beta, cu_seqlens, init_state, out, final, scale, lower_bound, gate_mode, stream)
    else:
        kda_prefill_ex(q, k, v, g_raw, beta, cu_seqlens, init_state, out, final, scale, lower_bound, gate_mode,
                       workspace, stream)
    return out, final


def decode(q, k, v, g_raw, beta, slot_idx, state_pool, *, scale, lower_bound=0.0, gate_mode="lower_bound",
           flags=0, norm_eps=0.0, stream=None):
    """Allocates ``out`` and runs ``kda_decode`` / ``kda_decode_ex`` (pool updated in place); returns out."""
    import torch
    out = torch.empty_like(q)
    if flags:
        kda_decode_ex(q, k, v, g_raw, beta, slot_idx, state_pool, out, scale, lower_bound, gate_mode, flags, norm_eps,
                      stream)
    else:
        kda_decode(q, k, v, g_raw, beta, slot_idx, state_pool, out, scale, lower_bound, gate_mode, stream)
    del torch
    return out
