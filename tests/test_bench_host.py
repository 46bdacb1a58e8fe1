"""Host-side pieces of bench.py, without a GPU.

The CPU baseline inside the measured line must time the oracle on a step
whose pages are all present: after ``advance()`` the next token can land on a
page the batch has not taken yet, and only ``prepare_step()`` takes it.
"""
from __future__ import annotations

import numpy as np
import pytest

import bench
from persistent_moe_decode_gb300.configs import WORKLOADS
from persistent_moe_decode_gb300.synth import DecodeBatch, make_kv_pools, make_model


@pytest.fixture(scope="module")
def tiny_inputs(oracle_lib):
    wl = WORKLOADS["tiny"].with_(context=63)     # the first advance crosses a page boundary
    model = make_model(wl.dims, wl.seed, "cpu")
    batch = DecodeBatch(wl)
    kp, vp = make_kv_pools(wl.dims, batch.num_pages, wl.kv_std, wl.seed, "cpu")
    return wl, model, batch, kp, vp


def test_cpu_sample_after_advance_on_a_page_boundary(tiny_inputs):
    wl, model, batch, kp, vp = tiny_inputs
    batch.advance(np.array([5], dtype=np.int32))
    assert int(batch.seq_lens[0]) == 64
    # the page of position 64 is not taken yet: the oracle refuses the step
    raw = (batch.tokens.copy(), batch.seq_lens.copy(), batch.page_tables.copy())
    with pytest.raises(RuntimeError, match="-2"):
        bench.CpuSample(model, kp, vp, raw, wl, 2).time_token()
    state = bench.snapshot(batch)
    assert state[2][0, 64 // 16] >= 0
    cs = bench.CpuSample(model, kp, vp, state, wl, 2)
    assert cs.time_token() > 0.0
    out = cs.measure(0.0)
    assert out["value"] > 0 and out["cores"] >= 1 and "context 64" in out["sample"]


def test_context_reported_the_same_way_in_both_arms():
    assert bench.context_of(np.array([8197])) == 8197
    assert bench.context_of(np.array([1, 2])) == "ragged"


def test_algorithmic_bytes_count_the_expert_format():
    """Per distinct routed expert: 2 bytes a weight (BF16), or 1 byte a weight
    plus one fp32 scale per row of its gate, up and down matrices (E4M3)."""
    from persistent_moe_decode_gb300.configs import A3B, algorithmic_bytes
    d = A3B
    per_bf16 = 3 * d.moe_inter * d.hidden * 2
    per_fp8 = 3 * d.moe_inter * d.hidden + 4 * (2 * d.moe_inter + d.hidden)
    distinct = [8] * d.n_layers
    keys = [8197]
    b16 = algorithmic_bytes(d, distinct, keys)
    b8 = algorithmic_bytes(d, distinct, keys, "fp8")
    assert b16 - b8 == sum(distinct) * (per_bf16 - per_fp8)
    assert b16 == 6889312256                     # the 8K batch-1 step the benchmark reports (8197 keys)


def test_traffic_key_ignores_comments_but_not_code():
    """The traffic record's key hashes the kernel code without comments and
    blank lines: a documentation edit keeps it, a code edit changes it."""
    import bench
    src = "int a; // count\n/* the\n   block */ int b;\n\n  float c;   \n"
    assert bench.kernel_code(src) == "int a;\n int b;\n  float c;"
    assert bench.kernel_code(src.replace("// count", "// the number of things")) == bench.kernel_code(src)
    assert bench.kernel_code(src.replace("int b;", "int b = 1;")) != bench.kernel_code(src)
