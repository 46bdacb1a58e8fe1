"""Parity of the CUDA decode step with the CPU oracle, through the C ABI.

Both sides get the same seeded weights, KV pools, page tables and tokens.  The
trajectory is teacher-forced by the GPU: each step both consume the GPU's
greedy token; each keeps its own KV cache.  Acceptance per step: logits
max-abs <= 2e-2 and relative L2 <= 1e-2; the expert set of every (layer,
token) equal to the oracle's wherever the oracle's k-th / (k+1)-th router-logit
gap exceeds 1e-3; greedy argmax equal on >= 99% of steps.

The kernel keeps every activation in fp32 (only the appended K/V are BF16, as
the cache is) and is compared with the oracle's plain fp64 definition.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from persistent_moe_decode_gb300 import mk
from persistent_moe_decode_gb300.configs import WORKLOADS
from tests._pair import Pair, check_logits, check_routing, run_trajectory
from tests._util import host_pool

pytestmark = pytest.mark.gpu


def rope_np(qkv_row, dims, pos):
    """RoPE (rotate-half pairs (i, i + d/2)) of the q heads of one row, fp64."""
    d, hq = dims.head_dim, dims.n_q_heads
    q = qkv_row[:hq * d].astype(np.float64).reshape(hq, d)
    i = np.arange(d // 2)
    ang = pos * dims.rope_theta ** (-2.0 * i / d)
    c, s_ = np.cos(ang), np.sin(ang)
    x1, x2 = q[:, :d // 2], q[:, d // 2:]
    return np.concatenate([x1 * c - x2 * s_, x2 * c + x1 * s_], axis=1).reshape(-1)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from persistent_moe_decode_gb300 import build
    build.build()
    oracle.build()


def test_tiny_intermediates_match_layer_by_layer():
    pair = Pair(WORKLOADS["tiny"])
    try:
        gpu, ref, tr = pair.step(trace=True)
        d = pair.wl.dims
        B = pair.wl.batch
        dec = pair.run.dec
        for l in range(d.n_layers + 1):
            h = np.frombuffer(dec.scratch(mk.MK_SCRATCH_H, l), dtype=np.float32).reshape(B, d.hidden)
            np.testing.assert_allclose(h, tr["h_in"][l], atol=1e-4, rtol=1e-3, err_msg=f"h layer {l}")
        for l in range(d.n_layers):
            x = np.frombuffer(dec.scratch(mk.MK_SCRATCH_X, l), dtype=np.float32).reshape(B, d.hidden)
            np.testing.assert_allclose(x, tr["x"][l], atol=1e-4, rtol=1e-4, err_msg=f"x layer {l}")
            qkv = np.frombuffer(dec.scratch(mk.MK_SCRATCH_QKV, l), dtype=np.float32).reshape(B, -1)
            pos = pair.run.batch.seq_lens[:B]
            q = np.stack([rope_np(qkv[b], d, int(pos[b])) for b in range(B)])
            np.testing.assert_allclose(q, tr["q"][l], atol=1e-4, rtol=1e-4, err_msg=f"q layer {l}")
            r = np.frombuffer(dec.scratch(mk.MK_SCRATCH_ROUTER, l), dtype=np.float32).reshape(B, -1)
            np.testing.assert_allclose(r, tr["router"][l], atol=1e-4, rtol=1e-4,
                                       err_msg=f"router layer {l}")
            a = np.frombuffer(dec.scratch(mk.MK_SCRATCH_ATTN, l), dtype=np.float32).reshape(B, -1)
            np.testing.assert_allclose(a, tr["attn"][l], atol=1e-4, rtol=1e-3,
                                       err_msg=f"attn layer {l}")
            o = np.frombuffer(dec.scratch(mk.MK_SCRATCH_OPROJ, l), dtype=np.float32)
            o = o.reshape(B, d.hidden)
            np.testing.assert_allclose(o, tr["attn_proj"][l], atol=1e-4, rtol=1e-3,
                                       err_msg=f"oproj layer {l}")
            y = np.frombuffer(dec.scratch(mk.MK_SCRATCH_MOE, l), dtype=np.float32)
            y = y.reshape(B, d.hidden)
            np.testing.assert_allclose(y, tr["moe"][l], atol=1e-4, rtol=1e-3,
                                       err_msg=f"moe layer {l}")
        check_logits(gpu, ref)
        check_routing(pair, tr)
        # the new K/V landed in the pool at the token's slot, as the oracle wrote it
        P = d.page_size
        pos = int(pair.run.batch.seq_lens[0])
        pg = int(pair.run.batch.page_tables[0, pos // P])
        kp = host_pool(pair.run.k_pool[:, pg])
        np.testing.assert_allclose(oracle.bf16_to_f64(kp[:, :, pos % P]),
                                   oracle.bf16_to_f64(pair.orc.k_pool[:, pg, :, pos % P]), atol=3e-2)
    finally:
        pair.close()


def test_tiny_trajectory():
    pair = Pair(WORKLOADS["tiny"])
    try:
        run_trajectory(pair, WORKLOADS["tiny"].steps)
    finally:
        pair.close()


SCHEDULES = (
    # every SM runs every phase, in each wave order, on all / one / seven SMs
    [dict(n_attn_claimers=10000, wave_order=o, sm_cap=c, n_moe_claimers=5)
     for o in (mk.MK_WAVES_DEFAULT, mk.MK_WAVES_ATTN_FIRST, mk.MK_WAVES_INTERLEAVED)
     for c in (0, 1, 7)]
    # SM roles: one or three attention SMs, the rest on the experts
    + [dict(n_attn_claimers=a, sm_cap=c) for a in (1, 3) for c in (0, 7)]
)


@pytest.mark.parametrize("kw", SCHEDULES, ids=lambda kw: "-".join(f"{k}{v}" for k, v in kw.items()))
def test_tiny_schedules_give_identical_logits(kw):
    """Any wave order, SM count, role split and slice count gives bit-identical
    output for a fixed split-KV chunk: every sum has a fixed order whatever SM
    computes it."""
    wl = WORKLOADS["tiny"]
    from persistent_moe_decode_gb300.runner import StepRunner
    ref_run = StepRunner(wl, device="cuda", kv_split_tokens=64)
    ref_run.step()
    torch.cuda.synchronize()
    ref_run.check_status()
    ref = ref_run.logits.clone()
    ref_run.close()
    run = StepRunner(wl, device="cuda", kv_split_tokens=64, **kw)
    run.step()
    torch.cuda.synchronize()
    run.check_status()
    assert torch.equal(run.logits, ref)
    run.close()


def test_tiny_forced_split_kv_matches_oracle():
    """64-token splits: the step's 65 keys make two items and a real combine."""
    pair = Pair(WORKLOADS["tiny"], kv_split_tokens=64)
    try:
        gpu, ref, tr = pair.step(trace=True)
        check_logits(gpu, ref)
        check_routing(pair, tr)
    finally:
        pair.close()


MID_SCHEDULES = (
    [dict(n_attn_claimers=a) for a in (20, 40, 75)]
    + [dict(n_attn_claimers=10000, wave_order=o) for o in (mk.MK_WAVES_DEFAULT, mk.MK_WAVES_INTERLEAVED)]
    + [dict(n_attn_claimers=3, sm_cap=16), dict(n_attn_claimers=10000, sm_cap=5)]
)


@pytest.mark.parametrize("kw", MID_SCHEDULES, ids=lambda kw: "-".join(f"{k}{v}" for k, v in kw.items()))
def test_mid_schedules_give_identical_logits(kw):
    """Hidden 2048: the one-token P1 and O-proj chunks take the
    split-contraction GEMV and the experts' down projection goes through the
    per-group partials; neither sum order depends on the SM count, the role
    split or the wave order, so the logits are bit-identical."""
    wl = WORKLOADS["mid_8k"]
    from persistent_moe_decode_gb300.runner import StepRunner
    ref_run = StepRunner(wl, device="cuda", kv_split_tokens=256)
    ref_run.step()
    torch.cuda.synchronize()
    ref_run.check_status()
    ref = ref_run.logits.clone()
    ref_run.close()
    run = StepRunner(wl, device="cuda", kv_split_tokens=256, **kw)
    run.step()
    torch.cuda.synchronize()
    run.check_status()
    assert torch.equal(run.logits, ref)
    run.close()


def test_mid_trajectory_and_split_kv():
    wl = WORKLOADS["mid_8k"].with_(steps=4)
    pair = Pair(wl)
    try:
        run_trajectory(pair, wl.steps)
    finally:
        pair.close()


@pytest.mark.parametrize("name", ["tiny_b5", "tiny_b12", "mid_b16", "mid_b4", "a3b4_b3"])
def test_multi_sequence_trajectory_with_churn(name):
    """Several ragged sequences per step (one and two GEMV token passes), one
    sequence retiring and a new one joining every step."""
    wl = WORKLOADS[name]
    pair = Pair(wl)
    try:
        run_trajectory(pair, wl.steps)
    finally:
        pair.close()


def test_fp8_experts_tiny_moe_output_and_trajectory():
    """8-bit routed experts (E4M3 bytes, one fp32 scale per row; CUDA-core rows
    of 256 columns): every layer's MoE output on the first step against the
    oracle's, then the whole teacher-forced trajectory."""
    wl = WORKLOADS["tiny_fp8"]
    pair = Pair(wl)
    try:
        gpu, ref, tr = pair.step(trace=True)
        d = wl.dims
        for l in range(d.n_layers):
            y = np.frombuffer(pair.run.dec.scratch(mk.MK_SCRATCH_MOE, l), dtype=np.float32)
            np.testing.assert_allclose(y.reshape(1, d.hidden), tr["moe"][l], atol=1e-4, rtol=1e-3,
                                       err_msg=f"moe layer {l}")
        check_logits(gpu, ref)
        check_routing(pair, tr)
    finally:
        pair.close()
    pair = Pair(wl)
    try:
        run_trajectory(pair, wl.steps)
    finally:
        pair.close()


def test_fp8_experts_mid_with_forced_split_kv():
    """8-bit experts with 256-token split-KV items (many items, several
    combines per head): two steps of the trajectory."""
    wl = WORKLOADS["mid_fp8"].with_(steps=2)
    pair = Pair(wl, kv_split_tokens=256)
    try:
        run_trajectory(pair, wl.steps)
    finally:
        pair.close()


def test_fp8_experts_mid_trajectory():
    """8-bit experts on the tensor cores (rows of 2048 E4M3 bytes, 16 per
    stage), mid model at 8K context."""
    wl = WORKLOADS["mid_fp8"].with_(steps=4)
    pair = Pair(wl)
    try:
        gpu, ref, tr = pair.step(trace=True)
        for l in range(wl.dims.n_layers):
            y = np.frombuffer(pair.run.dec.scratch(mk.MK_SCRATCH_MOE, l), dtype=np.float32)
            np.testing.assert_allclose(y.reshape(1, -1), tr["moe"][l], atol=1e-4, rtol=1e-3,
                                       err_msg=f"moe layer {l}")
        check_logits(gpu, ref)
        run_trajectory(pair, wl.steps - 1)
    finally:
        pair.close()


@pytest.mark.parametrize("name,steps", [("tiny_dense", 8), ("tiny_dense_b5", 6), ("mid_dense", 4),
                                        ("tiny_dense_fp8", 8)])
def test_dense_ffn_models(name, steps):
    """Dense feed-forward layers as one always-selected expert (E = k = 1):
    batch 1, several sequences with churn, and the mid shape with an
    intermediate size of 4096."""
    wl = WORKLOADS[name].with_(steps=steps)
    pair = Pair(wl)
    try:
        run_trajectory(pair, steps)
    finally:
        pair.close()


@pytest.mark.parametrize("name,rows", [("tiny_b12", 16), ("mid_b16", 64), ("mid_b16", 256), ("a3b4_b3", 128)])
def test_claimed_expert_tiles_give_identical_logits(name, rows):
    """Several tokens: the expert branch claiming tiles of its rows from
    per-layer counters computes every row as the static shares do, so a step
    gives bit-identical logits whichever SM took which tile."""
    wl = WORKLOADS[name]
    from persistent_moe_decode_gb300.runner import StepRunner
    out = []
    for kw in ({"moe_claim_rows": -1}, {"moe_claim_rows": rows}):
        run = StepRunner(wl, device="cuda", **kw)
        run.step()
        torch.cuda.synchronize()
        run.check_status()
        out.append(run.logits.clone())
        run.close()
    assert torch.equal(out[0], out[1])


def test_tiny_b12_intermediates():
    pair = Pair(WORKLOADS["tiny_b12"])
    try:
        gpu, ref, tr = pair.step(trace=True)
        d = pair.wl.dims
        B = pair.wl.batch
        dec = pair.run.dec
        for l in range(d.n_layers):
            x = np.frombuffer(dec.scratch(mk.MK_SCRATCH_X, l), dtype=np.float32).reshape(B, d.hidden)
            np.testing.assert_allclose(x, tr["x"][l], atol=1e-4, rtol=1e-4, err_msg=f"x layer {l}")
            a = np.frombuffer(dec.scratch(mk.MK_SCRATCH_ATTN, l), dtype=np.float32).reshape(B, -1)
            np.testing.assert_allclose(a, tr["attn"][l], atol=1e-4, rtol=1e-3, err_msg=f"attn layer {l}")
            y = np.frombuffer(dec.scratch(mk.MK_SCRATCH_MOE, l), dtype=np.float32).reshape(B, d.hidden)
            np.testing.assert_allclose(y, tr["moe"][l], atol=1e-4, rtol=1e-3, err_msg=f"moe layer {l}")
        check_logits(gpu, ref)
        check_routing(pair, tr)
    finally:
        pair.close()


def test_device_timeout_is_reported_and_recoverable():
    """A wait target that nothing can reach runs out (short limit) and reports
    MK_ERR_TIMEOUT; the context stays usable and the next step is correct."""
    from persistent_moe_decode_gb300.runner import StepRunner
    wl = WORKLOADS["tiny"]
    run = StepRunner(wl, device="cuda", timeout_ms=200)
    try:
        mk.mk_debug_bump_wait(run.dec.h, 1, 1000)
        run.step()
        torch.cuda.synchronize()
        rc, err = run.dec.status()
        assert rc == mk.MK_ERR_TIMEOUT, (rc, err.as_dict())
        mk.mk_debug_bump_wait(run.dec.h, 1, 0)
        run.step()
        torch.cuda.synchronize()
        run.check_status()
        assert torch.isfinite(run.logits).all()
    finally:
        run.close()
