"""The oracle's C code under AddressSanitizer and UndefinedBehaviorSanitizer
(CPU, no GPU).

oracle.c is compiled once more with the sanitizers into a temporary library,
and the oracle's whole-step tests (the independent restatement, the layer-range
pins, the 8-bit expert path) run against it in a child process that preloads
the sanitizer runtimes (ORACLE_LIB points the wrapper at that library).  An
out-of-bounds access, a use of freed memory or undefined behaviour in the
oracle fails the child, whatever the numbers.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _runtime(name: str) -> str | None:
    r = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True)
    path = r.stdout.strip()
    return path if r.returncode == 0 and os.path.isabs(path) and os.path.exists(path) else None


def test_oracle_step_tests_clean_under_sanitizers():
    if not shutil.which("gcc"):
        pytest.skip("no gcc")
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not asan or not ubsan:
        pytest.skip("the compiler has no sanitizer runtime")
    d = tempfile.mkdtemp(prefix="orc_san_")
    try:
        lib = os.path.join(d, "liboracle_san.so")
        src = os.path.join(ROOT, "oracle", "oracle.c")
        subprocess.run(["gcc", "-O1", "-g", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                        "-fsanitize=address,undefined", "-fno-omit-frame-pointer",
                        "-fno-sanitize-recover=undefined", "-o", lib, src, "-lm"], check=True)
        log = os.path.join(d, "san")
        env = dict(os.environ, ORACLE_LIB=lib, LD_PRELOAD=f"{asan} {ubsan}", OMP_NUM_THREADS="4",
                   ASAN_OPTIONS=f"detect_leaks=0:log_path={log}", UBSAN_OPTIONS=f"log_path={log}")
        tests = [os.path.join(HERE, t) for t in ("test_oracle_step_restated.py", "test_oracle_fp8.py")]
        r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", *tests],
                           capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
        reports = "".join(open(os.path.join(d, f)).read() for f in sorted(os.listdir(d)) if f.startswith("san"))
        out = r.stdout + r.stderr
        assert r.returncode == 0 and not reports, (reports or out)[-4000:]
    finally:
        shutil.rmtree(d, ignore_errors=True)
