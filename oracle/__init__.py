"""CPU oracle of the GPT-2 training step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call, link
or execute anything under ``oracle/``: only ``tests/``, the smoke check
(``__graft_entry__.smoke``) and the CPU-baseline leg of ``bench.py`` use it.

The oracle is a plain, slow, obviously correct restatement of the step in
float64 PyTorch CPU ops (matmul is the only library primitive used as a step),
with hand-derived backward formulas.  It shares no code with the CUDA library:
the two meet only through the seeded inputs of the ``synthetic`` module.

Parity status of each function (what pins it, besides itself) is listed in the
docstring of :mod:`oracle.gpt2`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "init_rng.c")
_LIB = os.path.join(_HERE, "liboracle_init.so")
_handle = None


def build(force: bool = False) -> str:
    """Compile the oracle's C initialiser (plain gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def init_lib():
    global _handle
    if _handle is None:
        lib = ctypes.CDLL(build())
        lib.oracle_sm64.restype = ctypes.c_uint64
        lib.oracle_sm64.argtypes = [ctypes.c_uint64]
        lib.oracle_draw.restype = ctypes.c_uint64
        lib.oracle_draw.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        lib.oracle_normal_fill.restype = None
        lib.oracle_normal_fill.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                           ctypes.c_void_p]
        _handle = lib
    return _handle
