"""The host scheduler (mk_sched.cpp) under AddressSanitizer and
UndefinedBehaviorSanitizer, over random valid configurations (CPU, no GPU).

tests/sched_fuzz.cpp drives validate_config, attention_sms, split_kv and
build_plan with random model shapes, schedule settings, SM counts (1 .. 152),
batches and sequence lengths (0 up to the page-table capacity); a memory error
(std::vector accesses past the size included: libstdc++'s container
annotations are on) or undefined behaviour ends the run with a non-zero
status.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "persistent_moe_decode_gb300", "csrc")


@pytest.fixture(scope="module")
def fuzz_bin():
    cxx = shutil.which("g++")
    if not cxx:
        pytest.skip("no g++")
    d = tempfile.mkdtemp(prefix="sched_fuzz_")
    exe = os.path.join(d, "sched_fuzz")
    cmd = [cxx, "-std=c++17", "-O1", "-g", "-D_GLIBCXX_SANITIZE_VECTOR", "-fsanitize=address,undefined",
           "-fno-omit-frame-pointer",
           "-fno-sanitize-recover=undefined", f"-I{os.path.join(ROOT, 'include')}", f"-I{CSRC}",
           os.path.join(HERE, "sched_fuzz.cpp"), os.path.join(CSRC, "mk_sched.cpp"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        if "sanitize" in r.stderr or "asan" in r.stderr.lower():
            pytest.skip("the compiler has no sanitizer runtime")
        raise AssertionError(r.stderr[-2000:])
    yield exe
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("seed", [1, 2])
def test_scheduler_clean_under_sanitizers(fuzz_bin, seed):
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0", UBSAN_OPTIONS="print_stacktrace=1")
    r = subprocess.run([fuzz_bin, str(seed)], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, (r.stdout[-1000:], r.stderr[-3000:])
    assert "ERROR" not in r.stderr and "runtime error" not in r.stderr, r.stderr[-3000:]
    n_cfg, n_plan = (int(v) for v in r.stdout.split()[1::2])
    assert n_cfg > 1000 and n_plan == n_cfg
