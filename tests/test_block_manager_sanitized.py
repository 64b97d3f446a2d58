"""The native host block manager under AddressSanitizer and
UndefinedBehaviorSanitizer (CPU only).

``tests/block_manager_fuzz.cpp`` drives every allocator entry point of
``include/pa.h`` with random valid and invalid calls and checks, after each,
that free + referenced blocks equal the pool and that each block's refcount
equals its number of holders (the fixed-size, refcounted blocks of "Paged
Attention and KV Cache Fragmentation", section "How PagedAttention maps an
OS concept onto GPU memory").  A memory error, undefined behaviour or a
broken invariant fails the test.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BUILD = os.path.join(ROOT, "paged_kv_cache_228_gb300", "_build")


@pytest.fixture(scope="module")
def fuzz_binary():
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    os.makedirs(BUILD, exist_ok=True)
    exe = os.path.join(BUILD, "block_manager_fuzz")
    cmd = [gxx, "-std=c++17", "-O1", "-g", "-fno-omit-frame-pointer",
           "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
           "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "block_manager_fuzz.cpp"),
           os.path.join(ROOT, "paged_kv_cache_228_gb300", "csrc", "block_manager.cpp"),
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and "sanitize" in r.stderr:
        pytest.skip("sanitizer runtime not available: " + r.stderr.strip().splitlines()[-1])
    assert r.returncode == 0, r.stderr
    return exe


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_block_manager_under_sanitizers(fuzz_binary, seed):
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    r = subprocess.run([fuzz_binary, str(seed), "6000"], capture_output=True, text=True,
                       env=env, timeout=300)
    assert r.returncode == 0, (r.stdout + r.stderr)[-3000:]
    assert r.stdout.startswith("ok")
