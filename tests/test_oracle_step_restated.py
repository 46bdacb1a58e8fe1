"""The oracle's whole decode step and its layer runner, pinned against an
independent fp64 PyTorch restatement of the step, written from the definition
("Inside the megakernel serving engine for North Mini Code": the parallel
transformer layer and the decode graph of §Tasks):

  h = E[token];  per layer  x = RMSNorm(h; g_l),
  [q; k; v] = W_qkv x,  RoPE on q and k at the token's position (here in its
  complex form: pair (i, i + d/2) is the complex number x_i + j x_{i+d/2},
  multiplied by exp(j pos theta^(-2i/d))),  k and v appended to the cache as
  BF16,  attention of every query head over its KV head's keys
  (scaled_dot_product_attention with GQA on the gathered pages),
  a = W_o attn,  router softmax, top-k renormalised,  MoE as a dense
  all-experts computation times a {0, w} mask,  h += a + m;
  logits = W_lm RMSNorm(h; g_f).

Nothing here calls the oracle's arithmetic; the oracle is then compared with
it.  ``orc_run_layers`` (the CPU baseline's body and the full-size layer
checker) is pinned the same way, and against ``orc_decode_step`` bit for bit.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from persistent_moe_decode_gb300.configs import MID, TINY
from persistent_moe_decode_gb300.synth import make_kv_pools, make_model
from tests._util import dims_dict, host_pool, host_weights


def bf16_round(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)


def rope_complex(x: torch.Tensor, pos: int, theta: float) -> torch.Tensor:
    d = x.shape[-1]
    half = d // 2
    z = torch.complex(x[..., :half], x[..., half:])
    ang = pos * theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    z = z * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([z.real, z.imag], dim=-1)


def torch_layers(m, kp, vp, l0, l1, h, lens, pt, force=None):
    """Layers [l0, l1) on the residual h [B, H] (fp64); appends K/V to kp, vp
    (BF16 tensors [L, pages, hkv, P, d]) in place.  Returns the new h.
    ``force`` maps (layer, token) to the experts that token must use (weights
    renormalised over them)."""
    d_ = m.dims
    hq, hkv, d, P, K = d_.n_q_heads, d_.n_kv_heads, d_.head_dim, d_.page_size, d_.top_k
    B = h.shape[0]
    h = h.clone()
    for l in range(l0, l1):
        x = F.rms_norm(h, (d_.hidden,), weight=m.attn_norm[l].double(), eps=d_.rms_eps)
        qkv = x @ m.w_qkv[l].double().T
        q = qkv[:, :hq * d].reshape(B, hq, d)
        k = qkv[:, hq * d:(hq + hkv) * d].reshape(B, hkv, d)
        v = qkv[:, (hq + hkv) * d:].reshape(B, hkv, d)
        att = torch.empty(B, hq * d, dtype=torch.float64)
        for b in range(B):
            pos = int(lens[b])
            qb = rope_complex(q[b], pos, d_.rope_theta)
            kb = rope_complex(k[b], pos, d_.rope_theta)
            page, slot = int(pt[b, pos // P]), pos % P
            kp[l, page, :, slot] = kb.to(torch.float32).to(torch.bfloat16)
            vp[l, page, :, slot] = v[b].to(torch.float32).to(torch.bfloat16)
            n = pos + 1
            rows = torch.tensor([int(pt[b, p // P]) for p in range(n)])
            slots = torch.arange(n) % P
            Kg = kp[l][rows, :, slots].double().permute(1, 0, 2)   # [hkv, n, d]
            Vg = vp[l][rows, :, slots].double().permute(1, 0, 2)
            o = F.scaled_dot_product_attention(qb[:, None, :].unsqueeze(0), Kg.unsqueeze(0),
                                               Vg.unsqueeze(0), enable_gqa=True)
            att[b] = o[0, :, 0, :].reshape(-1)
        a = att @ m.w_o[l].double().T
        r = x @ m.w_router[l].double().T
        p = torch.softmax(r, dim=-1)
        top = torch.topk(p, K, dim=-1)
        mask = torch.zeros_like(p).scatter(1, top.indices, top.values / top.values.sum(1, keepdim=True))
        for (fl, fb), experts in (force or {}).items():
            if fl == l:
                sel = torch.as_tensor(experts)
                mask[fb] = 0.0
                mask[fb, sel] = p[fb, sel] / p[fb, sel].sum()
        g = torch.einsum("eih,bh->bei", m.w_gate[l].double(), x)
        u = torch.einsum("eih,bh->bei", m.w_up[l].double(), x)
        y = torch.einsum("ehi,bei->beh", m.w_down[l].double(), F.silu(g) * u)
        moe = (mask[:, :, None] * y).sum(1)
        h = h + a + moe
    return h


def torch_step(m, kp, vp, tokens, lens, pt, force=None):
    h = m.embed[torch.as_tensor(tokens, dtype=torch.long)].double()
    h = torch_layers(m, kp, vp, 0, m.dims.n_layers, h, lens, pt, force)
    xf = F.rms_norm(h, (m.dims.hidden,), weight=m.final_norm.double(), eps=m.dims.rms_eps)
    return (xf @ m.lm_head.double().T).numpy()


def setup(dims, n_pages, lens, seed=5):
    m = make_model(dims, seed=seed)
    kp, vp = make_kv_pools(dims, n_pages, 1.0, seed=seed)
    rng = np.random.default_rng(seed)
    B = len(lens)
    per = (max(lens) + dims.page_size) // dims.page_size
    perm = rng.permutation(n_pages)[:B * per]
    pt = perm.reshape(B, per).astype(np.int32)
    toks = rng.integers(0, dims.vocab, size=B).astype(np.int32)
    return m, kp, vp, pt, toks, np.asarray(lens, dtype=np.int32)


def new_oracle(m, kp, vp):
    return oracle.Oracle(dims_dict(m.dims), host_weights(m), host_pool(kp), host_pool(vp))


def test_whole_step_matches_the_torch_restatement_on_tiny(oracle_lib):
    """C1 shapes, two ragged sequences (one spans a page boundary)."""
    m, kp, vp, pt, toks, lens = setup(TINY, 24, [47, 16])
    orc = new_oracle(m, kp, vp)
    logits = orc.decode_step(toks, lens, pt)
    kt, vt = kp.clone(), vp.clone()
    ref = torch_step(m, kt, vt, toks, lens, pt)
    np.testing.assert_allclose(logits, ref, rtol=1e-9, atol=1e-11)
    # the K/V both append are identical BF16 values
    np.testing.assert_array_equal(orc.k_pool, host_pool(kt))
    np.testing.assert_array_equal(orc.v_pool, host_pool(vt))


def test_run_layers_matches_the_torch_restatement(oracle_lib):
    m, kp, vp, pt, toks, lens = setup(TINY, 24, [30, 5, 64])
    orc = new_oracle(m, kp, vp)
    h0 = m.embed[torch.as_tensor(toks, dtype=torch.long)].double()
    got = orc.run_layers(0, TINY.n_layers, h0.numpy(), lens, pt)
    ref = torch_layers(m, kp.clone(), vp.clone(), 0, TINY.n_layers, h0, lens, pt).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def _run_layers_equals_decode_step(m, kp, vp, pt, toks, lens):
    d = m.dims
    orc_a = new_oracle(m, kp, vp)
    logits = orc_a.decode_step(toks, lens, pt)
    orc_b = new_oracle(m, kp, vp)
    h0 = oracle.bf16_to_f64(orc_b.w["embed"][toks])
    h = orc_b.run_layers(0, d.n_layers, h0, lens, pt)
    xf = np.stack([oracle.rmsnorm(h[b], orc_b.w["final_norm"], d.rms_eps) for b in range(len(toks))])
    lg = oracle.matvec(orc_b.w["lm_head"], xf).reshape(len(toks), -1)
    np.testing.assert_array_equal(lg, logits)                 # same code path, same order
    np.testing.assert_array_equal(orc_a.k_pool, orc_b.k_pool)
    np.testing.assert_array_equal(orc_a.v_pool, orc_b.v_pool)
    return orc_b, h0, h


def test_run_layers_plus_head_equals_decode_step_on_tiny(oracle_lib):
    m, kp, vp, pt, toks, lens = setup(TINY, 24, [40, 3])
    _run_layers_equals_decode_step(m, kp, vp, pt, toks, lens)


def test_run_layers_plus_head_equals_decode_step_on_two_mid_layers(oracle_lib):
    d2 = dataclasses.replace(MID, n_layers=2)
    m, kp, vp, pt, toks, lens = setup(d2, 24, [100])
    _run_layers_equals_decode_step(m, kp, vp, pt, toks, lens)


def test_run_layers_composes_over_the_layer_range(oracle_lib):
    """[0, 1) then [1, 2) equals [0, 2): the bound and the carried residual."""
    m, kp, vp, pt, toks, lens = setup(TINY, 24, [33, 17])
    h0 = oracle.bf16_to_f64(host_weights(m)["embed"][toks])
    whole = new_oracle(m, kp, vp).run_layers(0, 2, h0, lens, pt)
    orc = new_oracle(m, kp, vp)
    h1 = orc.run_layers(0, 1, h0, lens, pt)
    h2 = orc.run_layers(1, 2, h1, lens, pt)
    np.testing.assert_array_equal(h2, whole)
    assert not np.array_equal(h1, whole) and not np.array_equal(h1, h0)
    # an empty range is the identity; a range past the model is refused
    np.testing.assert_array_equal(orc.run_layers(1, 1, h1, lens, pt), h1)
    with pytest.raises(RuntimeError):
        orc.run_layers(0, 3, h0, lens, pt)


def test_forced_routing_of_its_own_choice_changes_nothing(oracle_lib):
    m, kp, vp, pt, toks, lens = setup(TINY, 24, [40, 9])
    orc = new_oracle(m, kp, vp)
    k0, v0 = orc.k_pool.copy(), orc.v_pool.copy()
    plain, tr = orc.decode_step(toks, lens, pt, trace=True)
    orc.k_pool[...] = k0
    orc.v_pool[...] = v0
    mask = np.ones(tr["idx"].shape[:2], dtype=bool)
    forced = orc.decode_step(toks, lens, pt, force=(tr["idx"], mask))
    np.testing.assert_array_equal(forced, plain)


def test_forced_routing_matches_the_torch_restatement(oracle_lib):
    """Other experts imposed on token 1 at layer 0 and token 0 at layer 1: the
    oracle equals the restatement that imposes the same sets."""
    m, kp, vp, pt, toks, lens = setup(TINY, 24, [40, 9])
    orc = new_oracle(m, kp, vp)
    k0, v0 = orc.k_pool.copy(), orc.v_pool.copy()
    _, tr = orc.decode_step(toks, lens, pt, trace=True)
    orc.k_pool[...] = k0
    orc.v_pool[...] = v0
    idx = tr["idx"].copy()
    mask = np.zeros(idx.shape[:2], dtype=bool)
    force = {}
    for (l, b) in ((0, 1), (1, 0)):
        others = [e for e in range(TINY.n_experts) if e not in idx[l, b]]
        idx[l, b] = others[:TINY.top_k]
        mask[l, b] = True
        force[(l, b)] = others[:TINY.top_k]
    got, tr2 = orc.decode_step(toks, lens, pt, trace=True, force=(idx, mask))
    assert tr2["idx"][0, 1].tolist() == force[(0, 1)]
    ref = torch_step(m, kp.clone(), vp.clone(), toks, lens, pt, force)
    np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-11)
    plain = torch_step(m, kp.clone(), vp.clone(), toks, lens, pt)
    assert np.abs(got - plain).max() > 1e-6       # the imposed experts do change the step
