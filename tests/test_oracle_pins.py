"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against a closed form, an invariant, a
brute-force computation on tiny inputs, or a special case that reduces to a
library routine (torch / numpy), so that a dropped term, a wrong sign, a
wrong index or a transposed operand fails at least one of them.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from persistent_moe_decode_gb300.configs import TINY, ModelDims
from persistent_moe_decode_gb300.synth import make_kv_pools, make_model, bf16_bits
from tests._util import dims_dict, make_oracle

RNG = np.random.default_rng(1234)


def rand_bf16_bits(shape, std=1.0, mean=0.0, seed=0):
    g = torch.Generator().manual_seed(seed)
    t = (torch.randn(shape, generator=g, dtype=torch.float32) * std + mean).to(torch.bfloat16)
    return bf16_bits(t).copy()


# ------------------------------------------------------------------ BF16

def test_bf16_roundtrip_and_ties():
    # exactly representable values survive
    for v in [0.0, 1.0, -2.5, 0.015625, 3.0e38 / 2 ** 100]:
        bits = oracle.to_bf16_bits(np.array([v]))
        assert oracle.bf16_to_f64(bits)[0] == np.float64(np.float32(v)) or v == 3.0e38 / 2 ** 100
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even) -> up
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    # just above a tie rounds up
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7


def test_bf16_matches_torch_rounding():
    x = RNG.standard_normal(4096) * np.exp(RNG.uniform(-20, 20, 4096))
    ours = oracle.to_bf16_bits(x)
    ref = bf16_bits(torch.tensor(x, dtype=torch.float32).to(torch.bfloat16))
    np.testing.assert_array_equal(ours, ref)


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_unit_gain_has_unit_rms():
    h = RNG.standard_normal(256) * 7.0
    ones = bf16_bits(torch.ones(256, dtype=torch.bfloat16)).copy()
    out = oracle.rmsnorm(h, ones, 1e-6)
    assert abs(np.sqrt(np.mean(out ** 2)) - 1.0) < 1e-6


def test_rmsnorm_scale_invariant():
    h = RNG.standard_normal(512)
    g = rand_bf16_bits(512, 0.02, 1.0, seed=3)
    a = oracle.rmsnorm(h, g, 0.0)
    b = oracle.rmsnorm(h * 123.5, g, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=0)


def test_rmsnorm_matches_torch():
    h = RNG.standard_normal(2048)
    g = rand_bf16_bits(2048, 0.02, 1.0, seed=4)
    gw = torch.tensor(oracle.bf16_to_f64(g))
    ref = F.rms_norm(torch.tensor(h), (2048,), weight=gw, eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rmsnorm(h, g, 1e-6), ref, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ RoPE

def test_rope_position_zero_is_identity():
    v = RNG.standard_normal(128)
    np.testing.assert_array_equal(oracle.rope(v, 0, 1e6), v)


def test_rope_d2_closed_form():
    # d = 2: one pair with inverse frequency theta^0 = 1, angle = pos radians
    for pos in [1, 7, 1000]:
        out = oracle.rope([1.0, 0.0], pos, 1e4)
        np.testing.assert_allclose(out, [math.cos(pos), math.sin(pos)], atol=1e-12)
        out = oracle.rope([0.0, 1.0], pos, 1e4)
        np.testing.assert_allclose(out, [-math.sin(pos), math.cos(pos)], atol=1e-12)


def test_rope_pairs_are_i_and_i_plus_half():
    # only coordinate 3 set: rotation must move it into coordinate 3 + d/2 only
    d = 16
    v = np.zeros(d)
    v[3] = 1.0
    out = oracle.rope(v, 5, 100.0)
    ang = 5 * 100.0 ** (-2 * 3 / d)
    expect = np.zeros(d)
    expect[3], expect[3 + d // 2] = math.cos(ang), math.sin(ang)
    np.testing.assert_allclose(out, expect, atol=1e-12)


def test_rope_preserves_norm_and_relative_position():
    d = 128
    q, k = RNG.standard_normal(d), RNG.standard_normal(d)
    for pos in [3, 8191, 262143]:
        assert abs(np.linalg.norm(oracle.rope(q, pos, 1e6)) - np.linalg.norm(q)) < 1e-9
    base = None
    for off in range(10):
        p = int(RNG.integers(0, 100000))
        dot = oracle.rope(q, p + 17, 1e6) @ oracle.rope(k, p, 1e6)
        if base is None:
            base = dot
        assert abs(dot - base) < 1e-8


# ------------------------------------------------------------------ mat-vec

def test_matvec_matches_numpy():
    w = rand_bf16_bits((37, 96), 0.02, seed=5)
    x = RNG.standard_normal((3, 96))
    ref = x @ oracle.bf16_to_f64(w).T
    np.testing.assert_allclose(oracle.matvec(w, x), ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(oracle.matvec(w, x[1]), ref[1], rtol=1e-12, atol=1e-15)


# --------------------------------------------------------- paged attention

def _pools(n_pages, hkv, P, d, seed):
    k = rand_bf16_bits((n_pages, hkv, P, d), 1.0, seed=seed)
    v = rand_bf16_bits((n_pages, hkv, P, d), 1.0, seed=seed + 1)
    return k, v


def _dims(hkv=2, d=64, P=16):
    dd = dims_dict(TINY)
    dd.update(n_kv_heads=hkv, head_dim=d, page_size=P)
    return dd


def _dense(pool, pt, n_keys, g):
    P = pool.shape[2]
    rows = [pool[pt[p // P], g, p % P] for p in range(n_keys)]
    return oracle.bf16_to_f64(np.stack(rows))


@pytest.mark.parametrize("n_keys", [1, 5, 16, 17, 64, 77])
def test_paged_attention_brute_force(n_keys):
    d, P, hkv = 64, 16, 2
    kp, vp = _pools(12, hkv, P, d, seed=10)
    pt = RNG.permutation(12).astype(np.int32)
    q = RNG.standard_normal(d)
    for g in range(hkv):
        K = _dense(kp, pt, n_keys, g)
        V = _dense(vp, pt, n_keys, g)
        s = K @ q / math.sqrt(d)
        p = np.exp(s - s.max())
        p /= p.sum()
        ref = p @ V
        out = oracle.paged_attention(_dims(hkv, d, P), kp, vp, pt, n_keys, g, q)
        np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_paged_attention_matches_sdpa_gqa():
    d, P, hkv, hq, n_keys = 64, 16, 2, 4, 50
    kp, vp = _pools(8, hkv, P, d, seed=20)
    pt = RNG.permutation(8).astype(np.int32)
    q = RNG.standard_normal((hq, d))
    K = np.stack([_dense(kp, pt, n_keys, g) for g in range(hkv)])
    V = np.stack([_dense(vp, pt, n_keys, g) for g in range(hkv)])
    ref = F.scaled_dot_product_attention(torch.tensor(q)[None, :, None, :], torch.tensor(K)[None],
                                         torch.tensor(V)[None], enable_gqa=True)[0, :, 0].numpy()
    for h in range(hq):
        out = oracle.paged_attention(_dims(hkv, d, P), kp, vp, pt, n_keys, h // (hq // hkv), q[h])
        np.testing.assert_allclose(out, ref[h], rtol=1e-10, atol=1e-12)


def test_paged_attention_page_permutation_invariant():
    d, P, hkv, n_keys = 64, 16, 2, 60
    kp, vp = _pools(6, hkv, P, d, seed=30)
    pt = np.arange(6, dtype=np.int32)
    q = RNG.standard_normal(d)
    a = oracle.paged_attention(_dims(hkv, d, P), kp, vp, pt, n_keys, 1, q)
    perm = RNG.permutation(6)
    kp2, vp2 = kp.copy(), vp.copy()
    kp2[perm] = kp
    vp2[perm] = vp
    b = oracle.paged_attention(_dims(hkv, d, P), kp2, vp2, perm[pt].astype(np.int32), n_keys, 1, q)
    np.testing.assert_array_equal(a, b)


def test_paged_attention_special_cases():
    d, P, hkv = 64, 16, 2
    kp, vp = _pools(4, hkv, P, d, seed=40)
    pt = np.array([2, 0, 3, 1], dtype=np.int32)
    q = RNG.standard_normal(d)
    # a single key returns its value row
    out = oracle.paged_attention(_dims(hkv, d, P), kp, vp, pt, 1, 1, q)
    np.testing.assert_allclose(out, oracle.bf16_to_f64(vp[2, 1, 0]), rtol=0, atol=1e-15)
    # q = 0 gives the plain mean of the values
    out = oracle.paged_attention(_dims(hkv, d, P), kp, vp, pt, 40, 0, np.zeros(d))
    np.testing.assert_allclose(out, _dense(vp, pt, 40, 0).mean(0), rtol=1e-12, atol=1e-14)


def test_split_merge_identity_of_the_softmax():
    """Any partition of the keys with the (m, l, o) merge equals one pass.

    This pins the merge rule the CUDA path's split-KV attention relies on
    against the oracle's single-pass attention."""
    d, P, hkv, n_keys = 64, 16, 2, 77
    kp, vp = _pools(6, hkv, P, d, seed=50)
    pt = RNG.permutation(6).astype(np.int32)
    q = RNG.standard_normal(d) * 3
    full = oracle.paged_attention(_dims(hkv, d, P), kp, vp, pt, n_keys, 0, q)
    K, V = _dense(kp, pt, n_keys, 0), _dense(vp, pt, n_keys, 0)
    for bounds in ([0, 77], [0, 16, 77], [0, 1, 30, 31, 64, 77]):
        ms, ls, os_ = [], [], []
        for a, b in zip(bounds[:-1], bounds[1:]):
            s = K[a:b] @ q / math.sqrt(d)
            m = s.max()
            p = np.exp(s - m)
            ms.append(m), ls.append(p.sum()), os_.append(p @ V[a:b])
        M = max(ms)
        num = sum(math.exp(m - M) * o for m, o in zip(ms, os_))
        den = sum(math.exp(m - M) * l for m, l in zip(ms, ls))
        np.testing.assert_allclose(num / den, full, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------- routing

def test_route_matches_full_sort():
    for trial in range(50):
        E, k = int(RNG.choice([8, 64, 128])), int(RNG.integers(1, 9))
        r = RNG.standard_normal(E)
        if trial % 5 == 0:
            r[RNG.integers(0, E, 4)] = r[0]        # plant ties
        idx, w, gap = oracle.route(r, k)
        r32 = r.astype(np.float32)
        order = sorted(range(E), key=lambda e: (-float(r32[e]), e))
        assert list(idx) == order[:k]
        if k < E:
            assert gap == pytest.approx(float(r32[order[k - 1]]) - float(r32[order[k]]), abs=0)
        sel = np.exp(r[idx] - r.max())
        np.testing.assert_allclose(w, sel / sel.sum(), rtol=1e-13)
        assert abs(w.sum() - 1.0) < 1e-14
        assert np.all(np.diff(w) <= 1e-15)


def test_route_k_equal_e_is_full_softmax():
    r = RNG.standard_normal(16) * 4
    idx, w, _ = oracle.route(r, 16)
    p = torch.softmax(torch.tensor(r), 0).numpy()
    np.testing.assert_allclose(w, p[idx], rtol=1e-13)


# -------------------------------------------------------------------- MoE

@pytest.fixture(scope="module")
def tiny_oracle():
    m = make_model(TINY, seed=7)
    k, v = make_kv_pools(TINY, 16, 1.0, seed=7)
    return m, make_oracle(m, k, v)


def _expert(m, l, e, x):
    wg = m.w_gate[l, e].double()
    wu = m.w_up[l, e].double()
    wd = m.w_down[l, e].double()
    xt = torch.tensor(x)
    return (wd @ (F.silu(wg @ xt) * (wu @ xt))).numpy()


def test_moe_equals_dense_masked_sum(tiny_oracle):
    m, orc = tiny_oracle
    E = TINY.n_experts
    x = RNG.standard_normal(TINY.hidden)
    idx = np.array([5, 2], dtype=np.int32)
    w = np.array([0.7, 0.3])
    mask = np.zeros(E)
    mask[idx] = w
    dense = sum(mask[e] * _expert(m, 1, e, x) for e in range(E))
    np.testing.assert_allclose(orc.moe(1, x, idx, w), dense, rtol=1e-10, atol=1e-13)


def test_moe_silu_limits(tiny_oracle):
    m, orc = tiny_oracle
    # x = 0 makes g = u = 0 for every expert: the MoE output is exactly zero
    out = orc.moe(0, np.zeros(TINY.hidden), np.array([1, 3], dtype=np.int32), np.array([0.5, 0.5]))
    assert np.all(out == 0.0)


def test_moe_bf16_hidden_flag_rounds(tiny_oracle):
    m, orc = tiny_oracle
    x = RNG.standard_normal(TINY.hidden)
    idx, w = np.array([4], dtype=np.int32), np.array([1.0])
    a = orc.moe(0, x, idx, w, 0)
    b = orc.moe(0, x, idx, w, oracle.BF16_A)
    assert not np.array_equal(a, b)
    np.testing.assert_allclose(a, b, rtol=0, atol=2e-2 * np.abs(a).max())


# ------------------------------------------------------- whole decode step

def _tiny_setup(seed=11, n_pages=12, ctx=40, batch=1, model_fn=None):
    m = make_model(TINY, seed=seed)
    if model_fn:
        model_fn(m)
    k, v = make_kv_pools(TINY, n_pages, 1.0, seed=seed)
    orc = make_oracle(m, k, v)
    rng = np.random.default_rng(seed)
    pt = np.stack([rng.permutation(n_pages)[:8] for _ in range(batch)]).astype(np.int32)
    if batch > 1:   # disjoint pages per sequence
        perm = rng.permutation(n_pages)
        pt = perm[:batch * 4].reshape(batch, 4).astype(np.int32)
    toks = rng.integers(0, TINY.vocab, size=batch).astype(np.int32)
    lens = np.full(batch, ctx, dtype=np.int32)
    return m, orc, pt, toks, lens


def _lm_of(m, h):
    g = m.final_norm.double()
    x = F.rms_norm(torch.tensor(h), (TINY.hidden,), weight=g, eps=TINY.rms_eps)
    return (m.lm_head.double() @ x).numpy()


def test_step_identity_layers_reduce_to_embed_norm_lmhead():
    """Zero O-proj and zero expert down weights make every layer the identity."""
    def zero(m):
        m.w_o.zero_()
        m.w_down.zero_()
    m, orc, pt, toks, lens = _tiny_setup(model_fn=zero)
    logits = orc.decode_step(toks, lens, pt)
    ref = _lm_of(m, m.embed[toks[0]].double().numpy())
    np.testing.assert_allclose(logits[0], ref, rtol=1e-10, atol=1e-12)


def test_step_uniform_attention_gqa_mapping():
    """Zero keys make attention uniform; per-KV-head constant values expose the
    query-head -> KV-head group mapping and the new token's own value."""
    def prep(m):
        m.w_down.zero_()
        H, d, hq, hkv = TINY.hidden, TINY.head_dim, TINY.n_q_heads, TINY.n_kv_heads
        m.w_qkv[:, hq * d:(hq + hkv) * d].zero_()     # new keys = 0
    m, orc, pt, toks, lens = _tiny_setup(model_fn=prep, ctx=37)
    d, hq, hkv, P = TINY.head_dim, TINY.n_q_heads, TINY.n_kv_heads, TINY.page_size
    v0 = np.stack([np.full(d, 0.5 + g) for g in range(hkv)])
    orc.k_pool[...] = 0
    for g in range(hkv):
        orc.v_pool[:, :, g] = oracle.to_bf16_bits(v0[g])
    logits, tr = orc.decode_step(toks, lens, pt, trace=True)
    C = int(lens[0])
    for l in range(TINY.n_layers):
        x = tr["x"][l, 0]
        vnew = (m.w_qkv[l, (hq + hkv) * d:].double().numpy() @ x).reshape(hkv, d)
        vnew = oracle.bf16_to_f64(oracle.to_bf16_bits(vnew))
        for h in range(hq):
            g = h // (hq // hkv)
            expect = (C * v0[g] + vnew[g]) / (C + 1)
            np.testing.assert_allclose(tr["attn"][l, 0, h * d:(h + 1) * d], expect, rtol=1e-10)
        # residual: h_{l+1} = h_l + W_o attn (MoE is zero)
        ap = m.w_o[l].double().numpy() @ tr["attn"][l, 0]
        np.testing.assert_allclose(tr["h_in"][l + 1, 0], tr["h_in"][l, 0] + ap, rtol=1e-10, atol=1e-12)


def test_step_moe_branch_matches_torch_topk():
    def prep(m):
        m.w_o.zero_()
    m, orc, pt, toks, lens = _tiny_setup(model_fn=prep)
    logits, tr = orc.decode_step(toks, lens, pt, trace=True)
    for l in range(TINY.n_layers):
        x = tr["x"][l, 0]
        r = m.w_router[l].double().numpy() @ x
        np.testing.assert_allclose(tr["router"][l, 0], r, rtol=1e-12)
        val, ind = torch.topk(torch.softmax(torch.tensor(r), 0), TINY.top_k)
        w = (val / val.sum()).numpy()
        assert list(tr["idx"][l, 0]) == list(ind.numpy())
        moe = sum(w[j] * _expert(m, l, int(ind[j]), x) for j in range(TINY.top_k))
        np.testing.assert_allclose(tr["moe"][l, 0], moe, rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(tr["h_in"][l + 1, 0], tr["h_in"][l, 0] + moe, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(logits[0], _lm_of(m, tr["h_in"][-1, 0]), rtol=1e-10, atol=1e-12)


def test_step_writes_rotated_kv_at_its_slot():
    m, orc, pt, toks, lens = _tiny_setup(ctx=21)
    _, tr = orc.decode_step(toks, lens, pt, trace=True)
    d, hq, hkv, P = TINY.head_dim, TINY.n_q_heads, TINY.n_kv_heads, TINY.page_size
    pos = int(lens[0])
    page, slot = pt[0, pos // P], pos % P
    theta = TINY.rope_theta
    for l in range(TINY.n_layers):
        x = tr["x"][l, 0]
        qkv = m.w_qkv[l].double().numpy() @ x
        k = qkv[hq * d:(hq + hkv) * d].reshape(hkv, d)
        v = qkv[(hq + hkv) * d:].reshape(hkv, d)
        # complex form of the rotation: z_i = k_i + j k_{i+d/2}, times e^{j pos theta^(-2i/d)}
        half = d // 2
        z = k[:, :half] + 1j * k[:, half:]
        z = z * np.exp(1j * pos * theta ** (-2.0 * np.arange(half) / d))
        krot = np.concatenate([z.real, z.imag], axis=1)
        np.testing.assert_array_equal(orc.k_pool[l, page, :, slot], oracle.to_bf16_bits(krot))
        np.testing.assert_array_equal(orc.v_pool[l, page, :, slot], oracle.to_bf16_bits(v))
        qrot = qkv[:hq * d].reshape(hq, d)
        zq = (qrot[:, :half] + 1j * qrot[:, half:]) * np.exp(1j * pos * theta ** (-2.0 * np.arange(half) / d))
        np.testing.assert_allclose(tr["q"][l, 0], np.concatenate([zq.real, zq.imag], 1).reshape(-1),
                                   rtol=1e-9, atol=1e-12)


def test_step_batch_rows_independent_and_page_relabel_invariant():
    m, orc, pt, toks, lens = _tiny_setup(batch=2, n_pages=12, ctx=30)
    k0, v0 = orc.k_pool.copy(), orc.v_pool.copy()
    both = orc.decode_step(toks, lens, pt)
    singles = []
    for b in range(2):
        orc.k_pool[...] = k0
        orc.v_pool[...] = v0
        singles.append(orc.decode_step(toks[b:b + 1], lens[b:b + 1], pt[b:b + 1])[0])
    np.testing.assert_array_equal(both, np.stack(singles))
    # relabel physical pages: identical logits
    perm = np.random.default_rng(3).permutation(orc.num_pages)
    orc.k_pool[:, perm] = k0
    orc.v_pool[:, perm] = v0
    relabeled = orc.decode_step(toks, lens, perm[pt].astype(np.int32))
    np.testing.assert_array_equal(relabeled, both)


def test_step_bf16_flags_round_where_stated():
    m, orc, pt, toks, lens = _tiny_setup()
    k0, v0 = orc.k_pool.copy(), orc.v_pool.copy()
    exact = orc.decode_step(toks, lens, pt)
    orc.k_pool[...] = k0
    orc.v_pool[...] = v0
    rounded, tr = orc.decode_step(toks, lens, pt, flags=oracle.ALL_BF16, trace=True)
    for key in ("x", "q", "attn"):
        vals = tr[key].reshape(-1)
        np.testing.assert_array_equal(vals, oracle.bf16_to_f64(oracle.to_bf16_bits(vals)))
    assert not np.array_equal(exact, rounded)
    np.testing.assert_allclose(rounded, exact, atol=2e-2)


def test_step_rejects_bad_pages():
    m, orc, pt, toks, lens = _tiny_setup()
    bad = pt.copy()
    bad[0, 0] = orc.num_pages + 3
    with pytest.raises(RuntimeError):
        orc.decode_step(toks, lens, bad)


# ------------------------------------------------------- dense FFN layers

def test_one_expert_is_the_dense_ffn():
    """With E = k = 1 the routing is exactly (0, 1.0) whatever the logit, and
    the MoE branch is the dense SwiGLU FFN W_d (SiLU(W_g x) * W_u x)."""
    from persistent_moe_decode_gb300.configs import TINY_DENSE
    for logit in (-3.5, 0.0, 7.25):
        idx, w, _ = oracle.route(np.array([logit]), 1)
        assert idx.tolist() == [0] and w.tolist() == [1.0]
    m = make_model(TINY_DENSE, seed=4)
    k, v = make_kv_pools(TINY_DENSE, 8, 1.0, seed=4)
    orc = make_oracle(m, k, v)
    x = RNG.standard_normal(TINY_DENSE.hidden)
    wg, wu, wd = (m.w_gate[1, 0].double(), m.w_up[1, 0].double(), m.w_down[1, 0].double())
    xt = torch.tensor(x)
    dense = (wd @ (F.silu(wg @ xt) * (wu @ xt))).numpy()
    np.testing.assert_allclose(orc.moe(1, x, np.array([0], dtype=np.int32), np.array([1.0])), dense,
                               rtol=1e-10, atol=1e-13)
