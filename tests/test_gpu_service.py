"""The decode service (include/mk.h, mk_service_*) over 32 continuous-batching
steps of the batch-16 workload's pattern, against the oracle.

16 slots hold sequences with ragged cached contexts; every step one request
finishes (requests are given staggered lengths) and a new one joins its slot
with 100 cached tokens on fresh random pages, as in the batch-16 workload
("Inside the megakernel serving engine for North Mini Code", §The serving
engine around the kernel).  The service retires, admits, schedules, runs the
step, picks the greedy tokens on the device and feeds them to the next step;
the test only submits requests and reads what happened.  Each step the oracle
runs the same batch (the same sequences, lengths, pages and input tokens,
i.e. teacher-forced by the GPU's tokens) on its own KV cache: logits within
max-abs 2e-2 and relative L2 1e-2, routed sets equal under the gap rule, the
device's greedy token equal to the argmax of the GPU logits, and equal to the
oracle's on >= 99 % of the (step, sequence) pairs.  The model is the
30B/3.3B-active shape cut to 4 layers, so the oracle keeps up.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from persistent_moe_decode_gb300 import mk
from persistent_moe_decode_gb300.configs import A3B
from persistent_moe_decode_gb300.synth import _normal_bf16, make_kv_pools, make_model
from tests._pair import GAP, MAX_ABS, REL_L2, oracle_step_following_ties
from tests._util import dims_dict, host_pool, host_weights

pytestmark = pytest.mark.gpu

STEPS, SLOTS, JOIN, MAXNEW = 32, 16, 100, 16


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from persistent_moe_decode_gb300 import build
    build.build()
    oracle.build()


def test_service_continuous_batching_matches_the_oracle():
    d = dataclasses.replace(A3B, n_layers=4)
    P = d.page_size
    rng = np.random.default_rng(7)
    ctx0 = rng.integers(64, 2048, size=SLOTS)
    max_pages = -(-(int(ctx0.max()) + STEPS + 1) // P) + 1
    n_pages = int(sum(-(-(int(c) + STEPS + 1) // P) for c in ctx0) + (STEPS + 2) * (-(-(JOIN + MAXNEW + 1) // P)))
    model = make_model(d, 3, "cuda")
    kp, vp = make_kv_pools(d, n_pages, 1.0, 3, "cuda")
    orc = oracle.Oracle(dims_dict(d), host_weights(model), host_pool(kp), host_pool(vp))
    dec = mk.Decoder(model, kp, vp, max_batch=SLOTS, max_pages_per_seq=max_pages)
    logits = torch.empty(SLOTS, d.vocab, dtype=torch.float32, device="cuda")
    svc = mk.mk_service_create(dec.h, logits.data_ptr())
    free = list(rng.permutation(n_pages)[::-1])
    pages_of, first_tok = {}, {}

    def submit(cached, max_new, fresh):
        npg = -(-(cached + max_new) // P)
        pg = [int(free.pop()) for _ in range(npg)]
        if fresh:     # a new synthetic prefix for the joining sequence, on both sides
            idx = torch.as_tensor(pg, dtype=torch.long, device="cuda")
            for l in range(d.n_layers):
                shape = (len(pg), d.n_kv_heads, P, d.head_dim)
                kp[l, idx] = _normal_bf16(shape, int(rng.integers(1 << 62)), "cuda", 1.0)
                vp[l, idx] = _normal_bf16(shape, int(rng.integers(1 << 62)), "cuda", 1.0)
                orc.k_pool[l, pg] = host_pool(kp[l, idx])
                orc.v_pool[l, pg] = host_pool(vp[l, idx])
        tok = int(rng.integers(0, d.vocab))
        rid = mk.mk_service_submit(svc, np.array(pg, dtype=np.int32), cached, tok, max_new)
        pages_of[rid], first_tok[rid] = pg, tok
        return rid

    try:
        ids0 = [submit(int(ctx0[k]), k + 1, False) for k in range(SLOTS)]   # one finishes per step
        agree = pairs = compared = 0
        greedy = {}
        for step in range(STEPS):
            mk.mk_service_run(svc, 1)
            mk.mk_service_wait(svc)
            ids, lens, toks = mk.mk_service_batch(svc, SLOTS)
            B = len(ids)
            assert B == SLOTS, (step, B)
            gpu = logits[:B].double().cpu().numpy()
            pt = np.full((B, max_pages), -1, dtype=np.int32)
            for i, rid in enumerate(ids):
                pt[i, :len(pages_of[rid])] = pages_of[rid]
            idx, _ = mk.mk_get_routing(dec.h, d.n_layers, B, d.top_k)
            ref, tr, _ = oracle_step_following_ties(orc, toks, lens, pt, idx)
            err = np.abs(gpu - ref).max()
            rel = np.linalg.norm(gpu - ref) / np.linalg.norm(ref)
            assert err <= MAX_ABS and rel <= REL_L2, f"step {step}: max-abs {err:.3e} rel-L2 {rel:.3e}"
            ok = tr["gap"] > GAP
            for l in range(d.n_layers):
                for i in range(B):
                    if ok[l, i]:
                        assert set(idx[l, i]) == set(tr["idx"][l, i]), (step, l, i)
            compared += int(ok.sum())
            for i, rid in enumerate(ids):
                greedy.setdefault(rid, []).append(int(np.argmax(gpu[i])))
                agree += int(np.argmax(gpu[i]) == np.argmax(ref[i]))
                pairs += 1
                # the input token is the first token or the previous greedy token
                k = len(greedy[rid]) - 1
                assert toks[i] == (first_tok[rid] if k == 0 else greedy[rid][k - 1]), (step, i)
            # retired requests give back their pages; one new request joins
            for rid in list(pages_of):
                tokens, done = mk.mk_service_result(svc, rid)
                assert tokens.tolist() == greedy.get(rid, [])[:len(tokens)], rid
                if done:
                    assert len(tokens) == len(greedy[rid])
                    free.extend(pages_of.pop(rid))
            submit(JOIN, MAXNEW, True)
        assert agree >= 0.99 * pairs, f"greedy tokens agreed on {agree}/{pairs}"
        assert compared > 0
        # the first requests finished in order, one per step
        for k, rid in enumerate(ids0):
            tokens, done = mk.mk_service_result(svc, rid)
            assert done and len(tokens) == k + 1
    finally:
        mk.mk_service_destroy(svc)
        dec.close()
