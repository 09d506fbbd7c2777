"""ORACLE (test infrastructure): fp64 attention and the log-sum-exp merge.

attend_heads() calls the plain C loops in oracle/attention.c.
merge() is GraniKV Eq. 1 (Section 2.3, "Cascade inference"), extended from two
states to any number by applying the same weights e^(lse_i - m) to each state:
    m = max_i lse_i,  O = sum_i e^(lse_i - m) O_i / sum_i e^(lse_i - m),
    lse = m + ln sum_i e^(lse_i - m).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "attention.c")
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(src):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gk_oracle_attend_heads.restype = ctypes.c_int
        lib.gk_oracle_attend_heads.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int64, dp, dp, dp, ctypes.c_double, dp, dp]
        lib.gk_oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads() -> int:
    return _load().gk_oracle_threads()


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def attend_heads(q, k, v, scale=None):
    """q [Hkv*g, d], k/v [Hkv, n, d] (fp64) -> (o [Hkv*g, d], lse [Hkv*g])."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    hkv, n, d = k.shape
    rows = q.shape[0]
    assert q.shape[1] == d and rows % hkv == 0 and v.shape == k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty((rows, d), dtype=np.float64)
    lse = np.empty(rows, dtype=np.float64)
    rc = _load().gk_oracle_attend_heads(hkv, rows // hkv, d, n, _ptr(q), _ptr(k), _ptr(v),
                                        float(scale), _ptr(o), _ptr(lse))
    if rc:
        raise MemoryError("oracle attention could not allocate its score buffer")
    return o, lse


def merge(states):
    """Merge [(o [rows, d], lse [rows]), ...] of disjoint key sets into one state."""
    os_ = np.stack([np.asarray(o, dtype=np.float64) for o, _ in states])
    ls = np.stack([np.asarray(l, dtype=np.float64) for _, l in states])
    m = ls.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(ls), np.exp(ls - m_safe[None, :]), 0.0)
    z = w.sum(axis=0)
    o = np.where(finite[:, None], (w[:, :, None] * os_).sum(axis=0) / np.where(z > 0, z, 1.0)[:, None], 0.0)
    lse = np.where(finite, m_safe + np.log(np.where(z > 0, z, 1.0)), -np.inf)
    return o, lse
