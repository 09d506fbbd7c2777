"""ctypes loader for the device-side input generator (synth/fill.cu)."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .gen import normal_table_bits

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None
_tables = {}


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "fill.cu")
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(src):
        subprocess.check_call([
            "nvcc", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
            "-gencode", "arch=compute_103a,code=sm_103a", "-o", LIB_PATH, src])
    return LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB_PATH)
        lib.synth_fill_normal_bf16.restype = ctypes.c_int
        lib.synth_fill_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                               ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                               ctypes.c_void_p]
        _lib = lib
    return _lib


def _table(device):
    import torch
    key = str(device)
    if key not in _tables:
        t = torch.from_numpy(normal_table_bits().view(np.int16).copy()).to(device)
        _tables[key] = t
    return _tables[key]


def fill_normal(out, key: int, offset: int = 0, log2_scale: int = 0, stream=None) -> None:
    """Fill a contiguous bf16 (or int16) CUDA tensor with stream `key` elements offset.. ."""
    import torch
    assert out.is_cuda and out.is_contiguous() and out.element_size() == 2
    s = stream if stream is not None else torch.cuda.current_stream(out.device)
    rc = _load().synth_fill_normal_bf16(ctypes.c_void_p(out.data_ptr()), out.numel(), key, offset,
                                        log2_scale, ctypes.c_void_p(_table(out.device).data_ptr()),
                                        ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth fill failed with cuda error {rc}")
