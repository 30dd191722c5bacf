"""Builds and loads the oracle's C word loop (``copy_oracle.c``).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Plain gcc, no CUDA:
the oracle must not depend on anything the GPU path builds.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "copy_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libcopy_oracle.so")
_lock = threading.Lock()
_handle = None


def build(force: bool = False) -> str:
    """Compile copy_oracle.c into a shared object; returns its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-shared", "-fPIC",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def load():
    global _handle
    with _lock:
        if _handle is None:
            _handle = ctypes.CDLL(build())
        return _handle
