"""The library's host code and the oracle's C loops under AddressSanitizer and
UndefinedBehaviorSanitizer (CPU).

Every C-ABI call takes raw host pointers and counts, so out-of-bounds reads or
writes, use after free and undefined arithmetic in the block manager, the HOT
allocator, the prefix caches and the planner would corrupt a caller's memory
silently.  This test builds libgk_san.so and liboracle_san.so (gcc's
-fsanitize=address,undefined on the host code; the first undefined-behaviour
report is fatal) and runs the host-side test files against them in a child
process that preloads the sanitizer runtimes (Python itself is not
instrumented, so leak checks stay off).  A sanitizer report fails the child
and so this test.
"""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

HOST_TESTS = ["tests/test_abi_host.py", "tests/test_prefix_cache_host.py", "tests/test_partition_host.py",
              "tests/test_oracle_attention.py"]

# In the child: the sanitized builds are the ones loaded, and the ASan runtime is live.
PROBE = """
import ctypes, os, sys
sys.path.insert(0, os.getcwd())
from paged_kv_cache_pool_gb300 import binding
from oracle import attention
assert binding.LIB_PATH.endswith("libgk_san.so"), binding.LIB_PATH
binding.lib()
attention.threads()
maps = open("/proc/self/maps").read()
assert "libgk_san.so" in maps and "liboracle_san.so" in maps and "libasan" in maps
ctypes.CDLL(None).__asan_init
print("sanitized builds loaded")
"""


def _run(args, env):
    r = subprocess.run(args, env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    return r.returncode, (r.stdout[-4000:] + "\n" + r.stderr[-4000:])


def test_host_code_under_address_and_undefined_behaviour_sanitizers():
    from paged_kv_cache_pool_gb300 import build
    from oracle import attention
    build.build()                     # the tests' own fixtures expect the plain build to be current
    build.build_sanitized()
    env = build.sanitizer_env()
    env["GK_ORACLE_LIB"] = attention.build(sanitized=True)
    env["OMP_NUM_THREADS"] = "2"
    rc, out = _run([sys.executable, "-c", PROBE], env)
    assert rc == 0, out
    rc, out = _run([sys.executable, "-m", "pytest", *HOST_TESTS, "-q", "-x", "-p", "no:cacheprovider",
                    "-m", "not gpu"], env)
    assert rc == 0, out
    assert "ERROR: AddressSanitizer" not in out and "runtime error:" not in out, out
