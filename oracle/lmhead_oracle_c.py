"""ctypes binding and build step of the C float64 oracle (lmhead_oracle_c.c).

TEST INFRASTRUCTURE ONLY: used by ``tests/``, ``__graft_entry__`` (which
builds it) and ``bench.py``'s CPU baseline and reference arm.  The product
never loads it.

``score_rows`` has the interface of ``lmhead_oracle.score_rows``: every row
handed in is a kept row; it returns (logprob, entropy, lse, dh or None,
dW or None) in float64.
"""

from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lmhead_oracle_c.c")
LIBDIR = os.path.join(HERE, "_build")
LIB = os.path.join(LIBDIR, "liblmhead_oracle_c.so")
_lib = None


def build(force: bool = False) -> str:
    """Compiles the oracle with the host C compiler (-O2, OpenMP) if stale."""
    os.makedirs(LIBDIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler for the oracle")
    tmp = LIB + ".tmp"
    r = subprocess.run([cc, "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-o", tmp, SRC,
                        "-lm"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the C oracle failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        handle = ctypes.CDLL(LIB)
        d = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        handle.lmhead_oracle_score_rows.restype = ctypes.c_int
        handle.lmhead_oracle_score_rows.argtypes = [d, d, ctypes.POINTER(i64), d, d, i64, i64,
                                                    i64, d, d, d, d, d]
        handle.lmhead_oracle_threads.restype = ctypes.c_int
        handle.lmhead_oracle_threads.argtypes = []
        _lib = handle
    return _lib


def threads() -> int:
    """Threads the oracle's parallel loops run on (OMP_NUM_THREADS or all cores)."""
    return int(lib().lmhead_oracle_threads())


def _dp(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def score_rows(h_rows, W, targets_rows, g_lp_rows=None, g_ent_rows=None):
    """Forward (and, given g_lp_rows, backward) of the given kept rows."""
    h = np.ascontiguousarray(h_rows, dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.float64)
    y = np.ascontiguousarray(targets_rows, dtype=np.int64)
    R, H = h.shape
    V = W.shape[0]
    gl = None if g_lp_rows is None else np.ascontiguousarray(g_lp_rows, dtype=np.float64)
    ge = None if (g_lp_rows is None or g_ent_rows is None) else np.ascontiguousarray(
        g_ent_rows, dtype=np.float64)
    lp, ent, lse = np.empty(R), np.empty(R), np.empty(R)
    dh = np.empty((R, H)) if gl is not None else None
    dW = np.empty((V, H)) if gl is not None else None
    code = lib().lmhead_oracle_score_rows(
        _dp(h), _dp(W), y.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _dp(gl), _dp(ge), R, H,
        V, _dp(lp), _dp(ent), _dp(lse), _dp(dh), _dp(dW))
    if code == 1:
        raise ValueError("a target is outside [0, V)")
    if code != 0:
        raise RuntimeError(f"C oracle failed with code {code}")
    return lp, ent, lse, dh, dW
