"""Host task lists: every wave's work is covered exactly once, whatever the SM
count, role split or batch (CPU only; the scheduler is host code).

The descriptor words and opcodes are the layout contract with the kernel:
word 0 the opcode, word 1 the layer, words 2-3 the op's range, words 6-7 the
W_qkv rows of a P1 task.
"""
from __future__ import annotations

import numpy as np
import pytest

from persistent_moe_decode_gb300 import mk
from persistent_moe_decode_gb300.configs import A3B, MID, TINY

OP_P1, OP_ROUTE, OP_ATTN, OP_UP, OP_COMBINE, OP_OUT, OP_FINAL, OP_DOWN = 1, 2, 3, 4, 5, 6, 7, 8
F_OP, F_LAYER, F_A0, F_A1, F_B0, F_B1 = 0, 1, 2, 3, 6, 7


@pytest.fixture(scope="module", autouse=True)
def built():
    from persistent_moe_decode_gb300 import build
    build.build()


def covered_once(ranges, total):
    """The half-open ranges tile [0, total) without overlap."""
    hits = np.zeros(total, dtype=np.int64)
    for lo, hi in ranges:
        assert 0 <= lo <= hi <= total, (lo, hi, total)
        hits[lo:hi] += 1
    return bool(np.all(hits == 1))


CASES = [(dims, n_sm, n_attn, batch)
         for dims in (TINY, MID, A3B)
         for n_sm, n_attn in ((152, 0), (152, 28), (152, 40), (152, 10000), (7, 3), (7, 10000), (1, 1))
         for batch in (1, 16)]


@pytest.mark.parametrize("dims,n_sm,n_attn,batch", CASES,
                         ids=lambda v: str(v) if not hasattr(v, "hidden") else f"H{v.hidden}")
def test_every_wave_is_covered_once_per_layer(dims, n_sm, n_attn, batch):
    cfg = mk.make_config(dims, 16, 64, 1024)
    cfg.n_attn_claimers = n_attn
    tasks, off, _ = mk.mk_plan(cfg, n_sm, batch)
    assert off[0] == 0 and off[-1] == len(tasks) and np.all(np.diff(off) >= 0)
    E = dims.n_experts
    Q = (dims.n_q_heads + 2 * dims.n_kv_heads) * dims.head_dim
    H = dims.hidden
    for layer in (0, dims.n_layers - 1):
        t = tasks[tasks[:, F_LAYER] == layer]
        p1 = t[t[:, F_OP] == OP_P1]
        assert len(p1) == n_sm
        assert covered_once(p1[:, [F_A0, F_A1]], E), "router rows"
        assert covered_once(p1[:, [F_B0, F_B1]], Q), "W_qkv rows"
        out = t[t[:, F_OP] == OP_OUT]
        assert len(out) == n_sm and covered_once(out[:, [F_A0, F_A1]], H), "O-proj rows"
        down = t[t[:, F_OP] == OP_DOWN]
        if batch == 1:
            assert covered_once(down[:, [F_A0, F_A1]], H), "DOWN rows"
        else:   # slices of the routed experts' rows, resolved on the device
            n_down = int(down[0, F_A1])
            assert sorted(down[down[:, F_A0] >= 0, F_A0].tolist()) == list(range(n_down)), "DOWN slices"
        comb = t[t[:, F_OP] == OP_COMBINE]
        assert covered_once(comb[:, [F_A0, F_A1]], batch * dims.n_q_heads), "combine units"
        up = t[t[:, F_OP] == OP_UP]
        n_up = int(up[0, F_A1])
        assert sorted(up[up[:, F_A0] >= 0, F_A0].tolist()) == list(range(n_up)), "UP slices"
    final = tasks[tasks[:, F_OP] == OP_FINAL]
    assert len(final) == n_sm and covered_once(final[:, [F_A0, F_A1]], dims.vocab)


@pytest.mark.parametrize("dims", [MID, A3B], ids=["mid", "a3b"])
def test_router_rows_are_few_per_sm_and_on_expert_sms(dims):
    cfg = mk.make_config(dims, 1, 64, 1024)
    cfg.n_attn_claimers = 28
    tasks, off, _ = mk.mk_plan(cfg, 152, 1)
    sm_of = np.repeat(np.arange(152), np.diff(off))
    first = tasks[:, F_LAYER] == 0
    attn_sms = set(sm_of[first & (tasks[:, F_OP] == OP_ATTN)].tolist())
    p1 = tasks[first & (tasks[:, F_OP] == OP_P1)]
    p1_sm = sm_of[first & (tasks[:, F_OP] == OP_P1)]
    n_router = p1[:, F_A1] - p1[:, F_A0]
    assert n_router.max() <= 8
    assert not attn_sms & set(p1_sm[n_router > 0].tolist())
    # an SM with router rows takes no W_qkv rows (its router chunk finishes early)
    assert np.all((p1[:, F_B1] - p1[:, F_B0])[n_router > 0] == 0)


@pytest.mark.parametrize("batch", [1, 16])
def test_expert_branch_orders_down_and_out(batch):
    """Several tokens: an expert SM's DOWN precedes its OUT (OUT's per-token
    expert sums wait for every DOWN task).  One token: OUT comes first (its
    O-proj rows need only the attention; nothing on the SM waits for the
    partial sums)."""
    cfg = mk.make_config(A3B, 16, 64, 1024)
    cfg.n_attn_claimers = 40
    tasks, off, _ = mk.mk_plan(cfg, 152, batch)
    checked = 0
    for s in range(152):
        t = tasks[off[s]:off[s + 1]]
        layer0 = t[t[:, F_LAYER] == 0]
        ops = layer0[:, F_OP].tolist()
        if OP_UP not in ops:
            continue   # attention SM
        i_down, i_out = ops.index(OP_DOWN), ops.index(OP_OUT)
        assert (i_out < i_down) if batch == 1 else (i_down < i_out), (s, ops)
        checked += 1
    assert checked == 152 - 40


def test_one_token_oproj_rows_favour_the_attention_branch():
    """One token: an attention SM's O-proj share is about four times an expert
    SM's (it is idle after its COMBINE); several tokens: even shares."""
    cfg = mk.make_config(A3B, 16, 64, 1024)
    cfg.n_attn_claimers = 40
    for batch, ratio in ((1, 4.0), (16, 1.0)):
        tasks, off, _ = mk.mk_plan(cfg, 152, batch)
        sm_of = np.repeat(np.arange(152), np.diff(off))
        first = tasks[:, F_LAYER] == 0
        attn_sms = set(sm_of[first & (tasks[:, F_OP] == OP_ATTN)].tolist())
        out = tasks[first & (tasks[:, F_OP] == OP_OUT)]
        out_sm = sm_of[first & (tasks[:, F_OP] == OP_OUT)]
        rows = out[:, F_A1] - out[:, F_A0]
        a = np.mean([r for r, s in zip(rows, out_sm) if s in attn_sms])
        e = np.mean([r for r, s in zip(rows, out_sm) if s not in attn_sms])
        assert abs(a / e - ratio) < 0.25 * ratio, (batch, a, e)
