"""The host scheduler's task lists equal, word for word, an independent
restatement of its rules ("Inside the megakernel serving engine for North
Mini Code", §The task scheduler: named waves per layer in one order, each SM
an equal share of every wave).  The rules, as stated in the scheduler's
documentation:

  roles      with n_attn < n_sm SMs on the attention branch, SM s is one of
             them when floor((s + 1) na / n) > floor(s na / n); attention SMs
             run P1, ATTN, COMBINE, OUT per layer; the others P1, ROUTE, UP,
             DOWN, OUT (one token: P1, ROUTE, UP, OUT, DOWN); without roles
             every SM runs the seven waves in the configured order.
  P1         router rows in runs of max(8, ceil(E / candidates)) rounded up
             to 8, to the expert-branch SMs in index order; W_qkv rows split
             over the SMs without router rows, in proportion to their even
             share of all P1 rows, in whole groups of 8 rows.
  COMBINE    (sequence, query head) units, an even share per combining SM.
  OUT        O-proj rows in groups of 8, shares weighted 4 : 1 toward the
             attention SMs with one token, even otherwise.
  UP, DOWN   "slice s of n" over the expert-branch SMs (UP: n = its size, or
             n_moe_claimers without roles); one token: DOWN takes an even
             share of the hidden rows.
  FINAL      LM-head rows in groups of 8, an even share per SM, the last SM
             also the vocabulary's tail.
"""
from __future__ import annotations

import numpy as np
import pytest

from persistent_moe_decode_gb300 import mk
from persistent_moe_decode_gb300.configs import A3B, MID, TINY

OP_P1, OP_ROUTE, OP_ATTN, OP_UP, OP_COMBINE, OP_OUT, OP_FINAL, OP_DOWN = 1, 2, 3, 4, 5, 6, 7, 8


@pytest.fixture(scope="module", autouse=True)
def built():
    from persistent_moe_decode_gb300 import build
    build.build()


def even(total, n, s):
    return total * s // n, total * (s + 1) // n


def restated_plan(dims, cfg, n_sm, batch, na):
    E, H, V, L = dims.n_experts, dims.hidden, dims.vocab, dims.n_layers
    qrows = (dims.n_q_heads + 2 * dims.n_kv_heads) * dims.head_dim
    roles = na < n_sm

    def attn_sm(s):
        return na >= n_sm or ((s + 1) * na // n_sm) > (s * na // n_sm)

    before = [s * na // n_sm for s in range(n_sm + 1)]
    n_moe_up = (n_sm - na) if roles else (cfg.n_moe_claimers if 0 < cfg.n_moe_claimers < n_sm else n_sm)
    n_comb = na if roles else n_sm
    n_down = (n_sm - na) if roles else n_sm
    # router rows
    cand = n_sm - na if roles else n_sm
    per = -(-max(8, -(-E // cand)) // 8) * 8
    rtr = [(0, 0)] * n_sm
    nxt = 0
    for s in range(n_sm):
        if nxt >= E:
            break
        if roles and attn_sm(s):
            continue
        rtr[s] = (nxt, min(E, nxt + per))
        nxt = rtr[s][1]
    # W_qkv rows: weights = even share of E + qrows, router SMs excluded (unless all are)
    tot = E + qrows
    w = [0 if rtr[s][1] > rtr[s][0] else (even(tot, n_sm, s)[1] - even(tot, n_sm, s)[0]) for s in range(n_sm)]
    if sum(w) == 0:
        w = [even(tot, n_sm, s)[1] - even(tot, n_sm, s)[0] for s in range(n_sm)]
    cw = np.concatenate([[0], np.cumsum(w)])
    g = 8 if qrows % 8 == 0 else 1
    qkv = [(g * ((qrows // g) * int(cw[s]) // int(cw[-1])), g * ((qrows // g) * int(cw[s + 1]) // int(cw[-1])))
           for s in range(n_sm)]
    # O-proj rows
    wo = [4 if (roles and batch == 1 and attn_sm(s)) else 1 for s in range(n_sm)]
    co = np.concatenate([[0], np.cumsum(wo)])
    og = 8 if H % 8 == 0 else 1
    orow = [(og * ((H // og) * int(co[s]) // int(co[-1])), og * ((H // og) * int(co[s + 1]) // int(co[-1])))
            for s in range(n_sm)]
    orders = {mk.MK_WAVES_DEFAULT: [OP_P1, OP_ROUTE, OP_ATTN, OP_UP, OP_COMBINE, OP_DOWN, OP_OUT],
              mk.MK_WAVES_ATTN_FIRST: [OP_P1, OP_ROUTE, OP_ATTN, OP_COMBINE, OP_UP, OP_DOWN, OP_OUT],
              mk.MK_WAVES_INTERLEAVED: [OP_P1, OP_ROUTE, OP_UP, OP_ATTN, OP_DOWN, OP_COMBINE, OP_OUT]}
    lists = []
    for s in range(n_sm):
        if not roles:
            ops = orders[cfg.wave_order]
        elif attn_sm(s):
            ops = [OP_P1, OP_ATTN, OP_COMBINE, OP_OUT]
        else:
            ops = [OP_P1, OP_ROUTE, OP_UP, OP_OUT, OP_DOWN] if batch == 1 else [OP_P1, OP_ROUTE, OP_UP, OP_DOWN, OP_OUT]
        rank = s - before[s] if roles else s
        rows = []
        for l in range(L):
            for op in ops:
                d = [0] * 32
                d[0], d[1] = op, l
                if op == OP_P1:
                    d[2], d[3] = rtr[s]
                    d[6], d[7] = qkv[s]
                elif op == OP_COMBINE:
                    d[2], d[3] = even(batch * dims.n_q_heads, n_comb, before[s] if roles else s)
                elif op == OP_OUT:
                    d[2], d[3] = orow[s]
                elif op == OP_UP:
                    d[2], d[3] = (rank if rank < n_moe_up else -1), n_moe_up
                elif op == OP_DOWN:
                    if batch == 1:
                        d[2], d[3] = even(H, n_down, rank)
                    else:
                        d[2], d[3] = (rank if rank < n_down else -1), n_down
                rows.append(d)
        lo, hi = even(V // 8, n_sm, s)
        d = [0] * 32
        d[0], d[1], d[2], d[3] = OP_FINAL, L, 8 * lo, V if s == n_sm - 1 else 8 * hi
        rows.append(d)
        for k, d in enumerate(rows):
            d[4] = k
        lists.append(np.array(rows, dtype=np.int32))
    targets = {"n_comb_sms": n_comb, "n_up_sms": n_moe_up if not roles else n_sm - na, "n_down_sms": n_down,
               "n_rtr_sms": sum(1 for s in range(n_sm) if rtr[s][1] > rtr[s][0])}
    if not roles:
        targets["n_up_sms"] = n_sm
    return lists, targets


CASES = [(dims, n_sm, batch, na, order, moe)
         for dims in (TINY, MID, A3B)
         for n_sm, na in ((152, 0), (152, 17), (152, 10000), (7, 2), (7, 10000), (2, 1), (1, 10000))
         for batch in (1, 16)
         for order, moe in (((0, 0),) if na < 10000 else ((0, 0), (1, 0), (2, 5)))]


@pytest.mark.parametrize("dims,n_sm,batch,na,order,moe", CASES,
                         ids=lambda v: f"H{v.hidden}" if hasattr(v, "hidden") else str(v))
def test_task_lists_equal_the_restated_rules(dims, n_sm, batch, na, order, moe):
    cfg = mk.make_config(dims, 16, 4096, 1 << 20, n_attn_claimers=na, wave_order=order, n_moe_claimers=moe)
    rng = np.random.default_rng(n_sm + batch)
    lens = rng.integers(1, 9000, size=batch).astype(np.int32)
    plan = mk.mk_plan_step(cfg, n_sm, batch, lens)
    n_attn = plan["n_attn"]
    if na == 0:
        assert 1 <= n_attn <= n_sm - 1
    lists, targets = restated_plan(dims, cfg, n_sm, batch, n_attn)
    off = plan["task_off"]
    for s in range(n_sm):
        got = plan["tasks"][off[s]:off[s + 1]]
        assert got.shape == lists[s].shape, (s, got.shape, lists[s].shape)
        diff = np.argwhere(got != lists[s])
        assert diff.size == 0, f"SM {s}: first differing (task, word) {diff[0].tolist()}: " \
                               f"{got[diff[0][0]].tolist()[:8]} vs {lists[s][diff[0][0]].tolist()[:8]}"
    for k, v in targets.items():
        assert plan[k] == v, (k, plan[k], v)


def restated_split(dims, n_sm, na, lens):
    """Balanced split-KV items: the concatenated pages of all sequences (keys
    = cached length + the new token) cut into na equal runs, one per attention
    SM, each run cut again at sequence boundaries."""
    P = dims.page_size
    pages = [-(-(int(n) + 1) // P) for n in lens]
    first = np.concatenate([[0], np.cumsum(pages)])
    T = int(first[-1])
    items, off = [], []
    for s in range(n_sm):
        off.append(len(items))
        is_attn = na >= n_sm or ((s + 1) * na // n_sm) > (s * na // n_sm)
        if not is_attn:
            continue
        r = s * na // n_sm
        g0, g1 = T * r // na, T * (r + 1) // na
        for b in range(len(lens)):
            p0, p1 = max(g0, first[b]) - first[b], min(g1, first[b + 1]) - first[b]
            if p1 > p0:
                items.append([b, int(p0) * P, min(int(lens[b]) + 1, int(p1) * P)])
    off.append(len(items))
    return items, off


@pytest.mark.parametrize("batch", [1, 5, 16])
@pytest.mark.parametrize("n_sm", [152, 7])
@pytest.mark.parametrize("fp8", [False, True])
def test_attention_split_and_items_equal_the_restated_rules(n_sm, batch, fp8):
    """(The attention-branch size is a float expression: the restatement
    computes it in the same double precision as the host.)"""
    dims = A3B
    if fp8 and batch > 1:
        pytest.skip("8-bit experts are a batch-1 format")
    cfg = mk.make_config(dims, 1 if fp8 else 16, 4096, 1 << 20,
                         expert_format=mk.MK_EXPERTS_FP8_E4M3 if fp8 else mk.MK_EXPERTS_BF16)
    rng = np.random.default_rng(batch * 7 + n_sm)
    lens = rng.integers(1, 40000, size=batch).astype(np.int32)
    plan = mk.mk_plan_step(cfg, n_sm, batch, lens)
    # attention SMs: KV bytes weighted by 1.6 (8192 / mean context)^0.22 / batch^0.45
    # against the routed experts' bytes
    keys = float(np.sum(lens.astype(np.float64) + 1))
    w = 1.6 * (8192.0 / (keys / batch)) ** 0.22 / batch ** 0.45
    kv = w * keys * 2 * dims.n_kv_heads * dims.head_dim * 2
    # 2 bytes a weight; 8-bit experts weighted as 1.5
    moe = min(dims.n_experts, batch * dims.top_k) * 3.0 * dims.moe_inter * dims.hidden * (1.5 if fp8 else 2)
    q = 4 if n_sm >= 64 else 1                    # in steps of 4 SMs on a large GPU
    ideal = n_sm * kv / (kv + moe)
    if batch > 1:                                 # at least 16 % of the SMs (23 % from 8 tokens)
        ideal = max(ideal, (0.23 if batch >= 8 else 0.16) * n_sm)
    na = max(1, min(n_sm - 1, q * int(ideal / q + 0.5)))
    assert plan["n_attn"] == na
    items, off = restated_split(dims, n_sm, na, lens)
    got = plan["items"]
    assert len(got) == len(items)
    np.testing.assert_array_equal(got[:, [0, 3, 4]], np.array(items, dtype=np.int32).reshape(-1, 3))
    np.testing.assert_array_equal(plan["item_off"], off)
    # per item: split index, split count, first item of the sequence, position
    for k, it in enumerate(got):
        b = it[0]
        mine = [i for i in range(len(items)) if items[i][0] == b]
        assert it[1] == mine.index(k) and it[2] == len(mine) and it[5] == mine[0] and it[6] == lens[b]
        assert plan["meta"][b].tolist() == [mine[0], len(mine)]
    # the items of a sequence cover its keys exactly once
    for b in range(batch):
        spans = sorted((int(it[3]), int(it[4])) for it in got if it[0] == b)
        assert spans[0][0] == 0 and spans[-1][1] == lens[b] + 1
        assert all(a[1] == c[0] for a, c in zip(spans, spans[1:]))
