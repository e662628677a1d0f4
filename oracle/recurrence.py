"""ctypes front end of the FP64 token recurrence in ``kda_oracle.c``.

TEST INFRASTRUCTURE (see the package docstring).

The recurrence (Kimi Delta Attention, the gated delta rule with per-channel decay;
"FlashInfer PR #4262: CAKE KDA Prefill Highlights" section 2 gives its chunked
form, whose token-level definition this is):

    S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
    o_t = scale * S_t^T q_t

Inputs may be torch tensors (any dtype, any device) or numpy arrays; they are
widened exactly to float64 before the C code sees them. Results are float64
numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")

GATE_MODES = {"lower_bound": 0, "softplus": 1, "log_decay": 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` with gcc (-O2, no fast-math) into ``oracle/_build``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-pthread",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            lib.oracle_kda_prefill.restype = ctypes.c_int
            lib.oracle_kda_prefill.argtypes = [dp, dp, dp, dp, dp, ip, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_int32, ctypes.c_int32, dp, ctypes.c_double,
                                               ctypes.c_double, ctypes.c_int32, ip, ctypes.c_int32,
                                               dp, dp, ctypes.c_int32]
            lib.oracle_kda_decode.restype = ctypes.c_int
            lib.oracle_kda_decode.argtypes = [dp, dp, dp, dp, dp, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, dp, ctypes.c_double, ctypes.c_double,
                                              ctypes.c_int32, dp, ctypes.c_int32]
            lib.oracle_kda_decode_ex.restype = ctypes.c_int
            lib.oracle_kda_decode_ex.argtypes = [dp, dp, dp, dp, dp, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32, dp, ctypes.c_double, ctypes.c_double,
                                                 ctypes.c_int32, ctypes.c_double, ctypes.c_int32, dp,
                                                 ctypes.c_int32]
            lib.oracle_kda_gate.restype = ctypes.c_double
            lib.oracle_kda_gate.argtypes = [ctypes.c_double, ctypes.c_int32, ctypes.c_double]
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen on its own side, then hand over
        x = x.detach().to("cpu").double().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _mode(gate_mode) -> int:
    return GATE_MODES[gate_mode] if isinstance(gate_mode, str) else int(gate_mode)


def oracle_threads(threads: int = 0) -> int:
    """Threads the oracle uses for ``threads`` (0 = every online core)."""
    return threads if threads > 0 else (os.cpu_count() or 1)


def prefill(q, k, v, g_raw, beta, cu_seqlens, init_state=None, *, scale, lower_bound=0.0,
            gate_mode="lower_bound", chains=None, want_final=True, threads=0, out=None):
    """Varlen prefill by the token recurrence, in FP64.

    Shapes: q, k, g_raw [T, H, dk]; v [T, H, dv]; beta [T, H]; cu_seqlens [N+1];
    init_state [N, H, dk, dv] or None (zeros). Returns (out [T, H, dv],
    final_state [N, H, dk, dv] or None, threads_used). ``chains`` optionally lists
    chain ids n*H + h to evaluate; rows of other chains stay as in ``out``
    (NaN-filled when ``out`` is not given).
    """
    q, k, v, a, b = (_f64(t) for t in (q, k, v, g_raw, beta))
    cu = _i32(cu_seqlens)
    T, H, dk = q.shape
    dv = v.shape[2]
    N = cu.shape[0] - 1
    assert k.shape == (T, H, dk) and a.shape == (T, H, dk) and v.shape[:2] == (T, H)
    assert b.shape == (T, H) and int(cu[-1]) == T and int(cu[0]) == 0
    s0 = _f64(init_state)
    if s0 is not None:
        assert s0.shape == (N, H, dk, dv)
    if out is None:
        out = np.full((T, H, dv), np.nan, dtype=np.float64)
    fin = np.zeros((N, H, dk, dv), dtype=np.float64) if want_final else None
    ch = None if chains is None else _i32(chains)
    lib = _load()
    rc = lib.oracle_kda_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(cu, ctypes.c_int32),
                                N, H, dk, dv, _ptr(s0), float(scale), float(lower_bound),
                                _mode(gate_mode), _ptr(ch, ctypes.c_int32),
                                0 if ch is None else int(ch.shape[0]), _ptr(out), _ptr(fin),
                                int(threads))
    if rc < 0:
        raise RuntimeError(f"oracle_kda_prefill failed with {rc}")
    return out, fin, rc


def decode(q, k, v, g_raw, beta, state, *, scale, lower_bound=0.0, gate_mode="lower_bound",
           norm_eps=None, beta_logits=False, threads=0):
    """T = 1 decode on gathered states, in FP64.

    Shapes: q, k, g_raw [R, H, dk]; v [R, H, dv]; beta [R, H]; state [R, H, dk, dv]
    (the pool rows already gathered by slot). Returns (out [R, H, dv],
    new_state [R, H, dk, dv], threads_used); the input ``state`` is not modified.
    ``norm_eps`` (not None) first L2-normalises q and k as x / sqrt(sum x^2 + eps);
    ``beta_logits`` reads beta as logits and applies the logistic function (the two input
    options of the decode ABI in FlashInfer PR #5551 / #5573).
    """
    q, k, v, a, b = (_f64(t) for t in (q, k, v, g_raw, beta))
    R, H, dk = q.shape
    dv = v.shape[2]
    st = np.array(_f64(state), dtype=np.float64, copy=True)
    assert st.shape == (R, H, dk, dv)
    out = np.zeros((R, H, dv), dtype=np.float64)
    lib = _load()
    rc = lib.oracle_kda_decode_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), R * H, dk, dv, _ptr(st),
                                  float(scale), float(lower_bound), _mode(gate_mode),
                                  -1.0 if norm_eps is None else float(norm_eps), int(bool(beta_logits)),
                                  _ptr(out), int(threads))
    if rc < 0:
        raise RuntimeError(f"oracle_kda_decode failed with {rc}")
    return out, st, rc


def gate(a: float, gate_mode="lower_bound", lower_bound=0.0) -> float:
    """The per-channel log decay g the C oracle uses for raw gate value ``a``."""
    return _load().oracle_kda_gate(float(a), _mode(gate_mode), float(lower_bound))
