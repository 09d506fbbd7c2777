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
# the same loops built with AddressSanitizer and UndefinedBehaviorSanitizer; a
# process selects it with GK_ORACLE_LIB (and preloads the sanitizer runtimes)
LIB_SAN = os.path.join(_HERE, "liboracle_san.so")
SAN_FLAGS = ["-fsanitize=address", "-fsanitize=undefined", "-fno-omit-frame-pointer",
             "-fno-sanitize-recover=undefined"]
_lib = None


def build(force: bool = False, sanitized: bool = False) -> str:
    src = os.path.join(_HERE, "attention.c")
    out = LIB_SAN if sanitized else LIB_PATH
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        env = dict(os.environ)
        env.pop("LD_PRELOAD", None)
        flags = SAN_FLAGS if sanitized else []
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", *flags, "-o", tmp, src, "-lm"], env=env)
        os.replace(tmp, out)
    return out


def _load():
    global _lib
    if _lib is None:
        path = os.environ.get("GK_ORACLE_LIB")
        if not path:
            path = build()
        lib = ctypes.CDLL(path)
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
