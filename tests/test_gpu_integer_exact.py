"""The integer results of a step, bit for bit: the per-expert grouping of the
routing, the pages the attention gathered and the cache slot of every new
K/V, each against a restatement of its rule ("Inside the megakernel serving
engine for North Mini Code", §Tasks: the route finalize / gather of the MoE
tiles and the paged KV cache):

  grouping   the routed experts of a layer in ascending order; the first
             grouped slot of each = the entries of the experts before it;
             within an expert its entries b * top_k + j in ascending token
             order;
  gather     logical page p of sequence b read from physical page
             page_table[b][p], for p < ceil((seq_len + 1) / 16), nothing else;
  new slot   page_table[b][pos / 16] * 16 + pos % 16 at pos = seq_len.

The routing itself is compared with the oracle's (sets, gap rule) by the
trajectory tests; here the grouping is checked against the GPU's own top-k,
which it must follow exactly.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from persistent_moe_decode_gb300 import mk
from persistent_moe_decode_gb300.configs import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from persistent_moe_decode_gb300 import build
    build.build()


def restated_groups(idx_l, K):
    """(n_act, act, off, ent) of one layer from its [B][K] routing."""
    B = idx_l.shape[0]
    act = sorted(set(int(e) for e in idx_l.reshape(-1)))
    ent, off = [], []
    for e in act:
        off.append(len(ent))
        ent += [b * K + j for b in range(B) for j in range(K) if idx_l[b, j] == e]
    off.append(len(ent))
    return len(act), act, off, ent


@pytest.mark.parametrize("name,steps", [("tiny", 2), ("mid_8k", 1), ("tiny_b12", 3), ("mid_b16", 2)])
def test_grouping_gather_and_slots_are_exact(name, steps):
    from persistent_moe_decode_gb300.runner import StepRunner
    wl = WORKLOADS[name]
    d = wl.dims
    run = StepRunner(wl, device="cuda", trace_records=64)
    try:
        for s in range(steps):
            b = run.batch
            b.prepare_step()
            lens, pt = b.seq_lens.copy(), b.page_tables.copy()
            run.step()
            torch.cuda.synchronize()
            run.check_status()
            B, K, L, MP = wl.batch, d.top_k, d.n_layers, b.max_pages
            idx, _ = run.dec.routing()
            groups = mk.mk_read_debug(run.dec.h, mk.MK_DEBUG_ROUTE_GROUPS).reshape(L, -1)
            for l in range(L):
                n, act, off, ent = restated_groups(idx[l], K)
                g = groups[l]
                assert g[0] == n, (l, g[0], n)
                assert g[1:1 + n].tolist() == act and np.all(g[1 + n:1 + 128] == -1)
                assert g[129:129 + n + 1].tolist() == off
                assert g[258:258 + len(ent)].tolist() == ent and np.all(g[258 + len(ent):] == -1)
            pages = mk.mk_read_debug(run.dec.h, mk.MK_DEBUG_PAGE_GATHER).reshape(B, MP)
            for i in range(B):
                npg = -(-(int(lens[i]) + 1) // d.page_size)
                assert pages[i, :npg].tolist() == pt[i, :npg].tolist(), i
                assert np.all(pages[i, npg:] == -1)
            slots = mk.mk_read_debug(run.dec.h, mk.MK_DEBUG_NEW_SLOT)
            want = [int(pt[i, lens[i] // d.page_size]) * d.page_size + int(lens[i]) % d.page_size for i in range(B)]
            assert slots.tolist() == want
            run.advance(run.greedy())
    finally:
        run.close()
