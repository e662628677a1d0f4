"""KDA oracle: slow, plainly correct FP64 CPU implementations of the KDA hot path.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. It shares no code with the
CUDA path (``kda_recurrent_gb300``) and does not import it.

Contents
  * ``prefill`` / ``decode`` -- the token-by-token recurrence in FP64 (plain C,
    ``kda_oracle.c``, one POSIX thread per core over independent chains).
  * ``brute`` -- explicit transition-matrix expansion for T <= 8 (numpy).
  * ``chunked`` -- the chunk-32 closed form of "FlashInfer PR #4262: CAKE KDA
    Prefill Highlights" section 2 in FP64 (numpy), with the fixed exponent anchor
    of its section 1 and a range checker for that anchor.

Pins (tests/test_oracle_pins.py) tie the recurrence to closed forms, invariants,
library routines and the brute-force expansion; each function's docstring names
the passage it follows.
"""
from .recurrence import decode, gate, prefill, oracle_threads  # noqa: F401
from . import brute, chunked  # noqa: F401
