"""Pins of the oracle's 8-bit expert path (CPU, no GPU).

The format is the OCP 8-bit floating point specification's E4M3 with one fp32
scale per output row: weight = scale[row] * e4m3(byte).  The pins hold the
oracle to things other than itself:

* every one of the 256 codes decodes as PyTorch's float8_e4m3fn does (a
  library routine; the encoding has no infinities and two NaN codes);
* the spec's landmarks: 448 is the largest finite value, 2^-9 the smallest
  subnormal, 2^-6 the smallest normal;
* with power-of-two scales every weight s * e4m3(q) is a BF16 value, so the
  8-bit path must give bit for bit what the BF16 path gives on those BF16
  weights: for one matrix-vector product, for one expert block (gate, up,
  down with their own scales) and for a whole decode step.  A swapped scale
  array, a scale indexed by the wrong dimension or a gate / up mix-up breaks
  the equality.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from persistent_moe_decode_gb300.configs import TINY
from persistent_moe_decode_gb300.synth import (DecodeBatch, bf16_bits, make_kv_pools, make_model,
                                               quantize_e4m3_rows)
from persistent_moe_decode_gb300.configs import WORKLOADS
from tests._util import dims_dict, host_pool, host_weights

RNG = np.random.default_rng(11)


def test_all_codes_decode_like_torch_float8_e4m3fn():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.isnan(ours).sum() == 2                       # S.1111.111, both signs
    fin = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[fin], ref[fin])


def test_spec_landmarks():
    assert oracle.e4m3_to_f64(np.array([0x7E]))[0] == 448.0          # largest finite
    assert oracle.e4m3_to_f64(np.array([0xFE]))[0] == -448.0
    assert oracle.e4m3_to_f64(np.array([0x01]))[0] == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_to_f64(np.array([0x08]))[0] == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_to_f64(np.array([0x38]))[0] == 1.0            # exponent field = bias
    assert oracle.e4m3_to_f64(np.array([0x80]))[0] == 0.0 and np.signbit(oracle.e4m3_to_f64(np.array([0x80]))[0])


def _codes(shape, rng):
    """Random finite E4M3 codes (no NaN)."""
    c = rng.integers(0, 256, size=shape, dtype=np.int64)
    c[(c & 0x7F) == 0x7F] = 0x3C
    return c.astype(np.uint8)


def _pow2_scales(shape, rng):
    return (2.0 ** -rng.integers(6, 12, size=shape)).astype(np.float32)


def _bf16_twin(q, s):
    """BF16 bits of s[row] * e4m3(q[row][col]): exact (4 significant bits times a power of two)."""
    w = oracle.e4m3_to_f64(q) * s[..., None].astype(np.float64)
    bits = bf16_bits(torch.tensor(w, dtype=torch.float32).to(torch.bfloat16)).copy()
    assert np.array_equal(oracle.bf16_to_f64(bits), w)
    return bits


def test_matvec_e4m3_equals_bf16_matvec_on_exact_weights():
    q = _codes((37, 96), RNG)
    s = _pow2_scales(37, RNG)
    x = RNG.standard_normal(96)
    np.testing.assert_array_equal(oracle.matvec_e4m3(q, s, x), oracle.matvec(_bf16_twin(q, s), x))


def test_matvec_e4m3_scale_is_per_output_row():
    q = _codes((8, 40), RNG)
    s = _pow2_scales(8, RNG)
    x = RNG.standard_normal(40)
    y = oracle.matvec_e4m3(q, s, x)
    y1 = oracle.matvec_e4m3(q, np.ones(8, dtype=np.float32), x)
    np.testing.assert_array_equal(y, y1 * s.astype(np.float64))


def _exact_fp8_model(seed=5):
    """A tiny model whose experts are given as E4M3 codes with power-of-two
    row scales, plus the BF16 model holding exactly those weights."""
    rng = np.random.default_rng(seed)
    m = make_model(TINY, seed=seed)
    L, E, I, H = TINY.n_layers, TINY.n_experts, TINY.moe_inter, TINY.hidden
    fp8 = {"q_gate": _codes((L, E, I, H), rng), "q_up": _codes((L, E, I, H), rng),
           "q_down": _codes((L, E, H, I), rng), "s_gate": _pow2_scales((L, E, I), rng),
           "s_up": _pow2_scales((L, E, I), rng), "s_down": _pow2_scales((L, E, H), rng)}
    # keep the expert outputs in a sensible range: codes up to 448 times 2^-6..2^-11
    w = host_weights(m)
    w["w_gate"] = _bf16_twin(fp8["q_gate"], fp8["s_gate"])
    w["w_up"] = _bf16_twin(fp8["q_up"], fp8["s_up"])
    w["w_down"] = _bf16_twin(fp8["q_down"], fp8["s_down"])
    return m, w, fp8


def test_moe_fp8_equals_bf16_on_exact_weights():
    m, w, fp8 = _exact_fp8_model()
    k, v = make_kv_pools(TINY, 8, 1.0, seed=1)
    a = oracle.Oracle(dims_dict(TINY), w, host_pool(k), host_pool(v))
    b = oracle.Oracle(dims_dict(TINY), host_weights(m), host_pool(k), host_pool(v), fp8=fp8)
    x = RNG.standard_normal(TINY.hidden) * 0.1
    for layer in range(TINY.n_layers):
        idx = np.array([6, 1], dtype=np.int32)
        wt = np.array([0.625, 0.375])
        np.testing.assert_array_equal(b.moe(layer, x, idx, wt), a.moe(layer, x, idx, wt))


def test_decode_step_fp8_equals_bf16_on_exact_weights():
    m, w, fp8 = _exact_fp8_model(seed=8)
    wl = WORKLOADS["tiny_fp8"]
    batch = DecodeBatch(wl, seed=3)
    k, v = make_kv_pools(TINY, batch.num_pages, 1.0, seed=3)
    a = oracle.Oracle(dims_dict(TINY), w, host_pool(k), host_pool(v))
    b = oracle.Oracle(dims_dict(TINY), host_weights(m), host_pool(k), host_pool(v), fp8=fp8)
    batch.prepare_step()
    args = (batch.tokens, batch.seq_lens, batch.page_tables)
    la = a.decode_step(*args)
    lb = b.decode_step(*args)
    np.testing.assert_array_equal(lb, la)
    np.testing.assert_array_equal(b.k_pool, a.k_pool)


def test_quantizer_rounds_each_row_to_its_nearest_code():
    """The synthetic inputs' per-row quantiser (not the method's arithmetic):
    every byte is a nearest E4M3 value of w / scale, and the row maximum maps to 448."""
    w = torch.randn(6, 300).to(torch.bfloat16) * 0.02
    q, s = quantize_e4m3_rows(w)
    vals = oracle.e4m3_to_f64(q.numpy())
    t = (w.double() / s.double().unsqueeze(-1)).numpy()
    grid = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    grid = np.unique(grid[~np.isnan(grid)])
    nearest = np.abs(t[..., None] - grid).min(-1)
    np.testing.assert_allclose(np.abs(t - vals), nearest, atol=1e-6 * np.abs(t).max())
    np.testing.assert_allclose(np.abs(vals).max(-1), 448.0)


@pytest.mark.parametrize("name", ["tiny_fp8"])
def test_fp8_workload_model_shapes(name):
    wl = WORKLOADS[name]
    m = make_model(wl.dims, 0, "cpu", wl.expert_format)
    d = wl.dims
    assert m.fp8["q_gate"].shape == (d.n_layers, d.n_experts, d.moe_inter, d.hidden)
    assert m.fp8["q_down"].shape == (d.n_layers, d.n_experts, d.hidden, d.moe_inter)
    assert m.fp8["s_down"].shape == (d.n_layers, d.n_experts, d.hidden)
    assert m.w_gate.numel() == 0
