"""Compile libgk.so (the C-ABI library) in place for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked with the
static CUDA runtime.  No CMake; a minute or so on a few cores.

build_sanitized() makes libgk_san.so, the same sources with the host code
instrumented by AddressSanitizer and UndefinedBehaviorSanitizer (gcc's
-fsanitize=address,undefined; device code is unchanged).  Python is not
instrumented, so a process that loads it needs libasan preloaded:
sanitizer_env() gives the environment for that, and GK_LIB_PATH selects the
library in the binding.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgk.so")
BUILD_SAN = os.path.join(HERE, "_build_san")
LIB_SAN = os.path.join(HERE, "libgk_san.so")
# one -Xcompiler per option: nvcc splits an -Xcompiler argument at its commas
SAN_FLAGS = [f for o in ("-fsanitize=address", "-fsanitize=undefined", "-fno-omit-frame-pointer",
                         "-fno-sanitize-recover=undefined") for f in ("-Xcompiler", o)]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["host_pool.cpp", "plan.cpp", "kv_write.cu", "gather_attn.cu", "merge.cu", "prefix_tc.cu",
           "prefix_warp.cu", "cascade_split.cu", "static_scratch.cu", "calibrate.cu"]
COMMON = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-lineinfo", "-I" + os.path.join(ROOT, "include")]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _tool_env() -> dict:
    """The compiler's environment: without the sanitizer runtimes a sanitized
    test process preloads (nvcc's own tools are not built for them)."""
    env = dict(os.environ)
    env.pop("LD_PRELOAD", None)
    return env


def _compile(src: str, extra, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [_nvcc(), *COMMON, *ARCH, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd.insert(1, "-x")
        cmd.insert(2, "cu")
    r = subprocess.run(cmd, capture_output=True, text=True, env=_tool_env())
    if r.returncode != 0:
        raise RuntimeError(f"compiling {src} failed:\n{r.stdout}\n{r.stderr}")
    return obj


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "gk.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), "-shared", *ARCH, "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=_tool_env())
    if r.returncode != 0:
        raise RuntimeError(f"linking libgk.so failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def build_sanitized(force: bool = False) -> str:
    """libgk_san.so: host code under AddressSanitizer and UndefinedBehaviorSanitizer."""
    if not force and not _stale(LIB_SAN):
        return LIB_SAN
    os.makedirs(BUILD_SAN, exist_ok=True)
    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, SAN_FLAGS, BUILD_SAN), SOURCES))
    tmp = LIB_SAN + f".tmp{os.getpid()}"
    cmd = [_nvcc(), "-shared", *ARCH, *SAN_FLAGS, "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=_tool_env())
    if r.returncode != 0:
        raise RuntimeError(f"linking libgk_san.so failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_SAN)
    return LIB_SAN


def _gcc_lib(name: str) -> str:
    r = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True, env=_tool_env())
    return r.stdout.strip()


def sanitizer_env(base=None) -> dict:
    """Environment for a Python process that loads libgk_san.so: the sanitizer
    runtimes preloaded (Python itself is not instrumented), leak checks off
    (the interpreter keeps its allocations until exit), CUDA's use of the
    shadow gap allowed, and the first undefined-behaviour report fatal."""
    env = dict(os.environ if base is None else base)
    env["LD_PRELOAD"] = ":".join(p for p in (_gcc_lib("libasan.so"), _gcc_lib("libubsan.so")) if p)
    env["ASAN_OPTIONS"] = "detect_leaks=0:protect_shadow_gap=0:alloc_dealloc_mismatch=0:abort_on_error=0"
    env["UBSAN_OPTIONS"] = "halt_on_error=1:print_stacktrace=1"
    env["GK_LIB_PATH"] = LIB_SAN
    return env


if __name__ == "__main__":
    if "--sanitized" in sys.argv:
        print(build_sanitized(force="--force" in sys.argv))
    else:
        build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
        print(LIB)
