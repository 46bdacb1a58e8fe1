"""The C-ABI library builds, loads and exports what include/mk.h declares (no GPU)."""
from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np
import pytest

from persistent_moe_decode_gb300 import build as B
from persistent_moe_decode_gb300 import mk
from persistent_moe_decode_gb300.configs import A3B, MID, TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return mk.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"\b(mk_[a-z_]+)\s*\(", src))
    return sorted(names)


def test_header_and_binding_agree():
    assert sorted(mk.EXPORTS) == declared_functions()


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror_and_version(lib):
    assert mk.mk_abi_version() == 1
    for code in range(0, -10, -1):
        assert mk.mk_strerror(code) != "unknown error"
    assert mk.mk_strerror(-99) == "unknown error"


def test_struct_layout_matches_header(lib, tmp_path):
    """Every field offset and struct size the C compiler gives the header's
    structs equals the ctypes mirror's."""
    import subprocess
    lines = []
    for st in (mk.mk_config, mk.mk_weights, mk.mk_error):
        lines.append(f'printf("{st.__name__} %zu\\n", sizeof({st.__name__}));')
        for name, _ in st._fields_:
            lines.append(f'printf("{st.__name__}.{name} %zu\\n", offsetof({st.__name__}, {name}));')
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "mk.h"\nint main(void) {\n'
                   + "\n".join(lines) + "\nreturn 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(line.split() for line in out if line)
    for st in (mk.mk_config, mk.mk_weights, mk.mk_error):
        assert int(got[st.__name__]) == C.sizeof(st), st.__name__
        for name, _ in st._fields_:
            assert int(got[f"{st.__name__}.{name}"]) == getattr(st, name).offset, (st.__name__, name)


def test_create_rejects_bad_configs_before_touching_the_device(lib):
    w = mk.mk_weights()
    for bad in (dict(head_dim=96), dict(n_q_heads=5), dict(max_batch=17), dict(page_size=8),
                dict(n_experts=300), dict(kv_split_tokens=100), dict(hidden=1000),
                dict(n_q_heads=64, n_kv_heads=8, head_dim=128), dict(expert_format=2),
                # 8-bit experts: batch 1 only, hidden 2048 or <= 1024, moe_inter % 16
                dict(expert_format=mk.MK_EXPERTS_FP8_E4M3, max_batch=2),
                dict(expert_format=mk.MK_EXPERTS_FP8_E4M3, hidden=1536),
                dict(expert_format=mk.MK_EXPERTS_FP8_E4M3, moe_inter=136),
                # claimed expert tiles: a multiple of 16 rows, or 0 / -1
                dict(moe_claim_rows=24), dict(moe_claim_rows=-2)):
        cfg = mk.make_config(TINY, 1, 8, 16)
        for k, v in bad.items():
            setattr(cfg, k, v)
        h = C.c_void_p()
        rc = lib.mk_create(C.byref(cfg), C.byref(w), C.byref(h))
        assert rc == mk.MK_ERR_BAD_CONFIG, bad


def test_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cfg = mk.make_config(TINY, 1, 8, 16)
    buf = np.zeros(1 << 20, dtype=np.uint8)
    p = buf.ctypes.data + (-buf.ctypes.data) % 16
    L = TINY.n_layers
    arr = (C.c_void_p * L)(*([p] * L))
    pp = C.cast(arr, C.POINTER(C.c_void_p))
    w = mk.mk_weights(embed=p, lm_head=p, final_norm=p, attn_norm=pp, w_qkv=pp, w_o=pp,
                      w_router=pp, w_gate=pp, w_up=pp, w_down=pp, k_pool=pp, v_pool=pp)
    h = C.c_void_p()
    assert lib.mk_create(C.byref(cfg), C.byref(w), C.byref(h)) == mk.MK_ERR_CUDA
    assert not h.value


def test_null_handle_calls_are_rejected(lib):
    assert lib.mk_decode_step(None, None, None) == mk.MK_ERR_BAD_ARG
    assert lib.mk_step_status(None, None) == mk.MK_ERR_BAD_ARG
    assert lib.mk_schedule_step(None, 1, None, None, None, None, None) == mk.MK_ERR_BAD_ARG
    lib.mk_destroy(None)


@pytest.mark.parametrize("dims", [TINY, MID, A3B])
def test_plan_builds_for_the_workload_shapes(lib, dims):
    cfg = mk.make_config(dims, 16, 64, 1024)
    tasks, off, n_bars = mk.mk_plan(cfg, 152, 16)
    assert off[0] == 0 and off[-1] == len(tasks) and np.all(np.diff(off) >= 0)
    assert n_bars > 0
