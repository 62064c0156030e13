"""The host C++ (the fp64 oracle and the input generator) under AddressSanitizer
and UndefinedBehaviorSanitizer.  compute-sanitizer is not used on the GPU path;
its race and bounds checking is replaced there by tail shapes, bitwise
determinism runs and the oracle comparison.  Host code gets the real thing:
`sanitize_driver.cpp` runs every exported oracle and generator routine on
ragged shapes (V = 1, odd sizes, one or four threads, an out-of-range target,
a keep mask), and any out-of-bounds access, use after free, leak, signed
overflow or misaligned access aborts it with a report."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_oracle_and_generator_under_asan_and_ubsan(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    exe = str(tmp_path / "sanitize_driver")
    cmd = [gxx, "-std=c++17", "-O1", "-g", "-fno-omit-frame-pointer", "-fsanitize=address,undefined",
           "-fno-sanitize-recover=all", "-pthread", os.path.join(ROOT, "tests", "sanitize_driver.cpp"),
           os.path.join(ROOT, "oracle", "oracle.cpp"), os.path.join(ROOT, "gen", "philox_gen.cpp"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and ("asan" in r.stderr or "ubsan" in r.stderr):
        pytest.skip("sanitizer runtime not installed: " + r.stderr[-300:])
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, ASAN_OPTIONS="abort_on_error=1:detect_leaks=1",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    p = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=600)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "sanitize driver: ok" in p.stdout
