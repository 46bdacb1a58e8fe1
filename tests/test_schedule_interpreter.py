"""The host plan's counter accounting and freedom from deadlock, checked by
running the task lists through the host interpreter (tests/_schedule_sim.py)
with the kernel's wait / arrive semantics, random interleavings and random
routing ("Inside the megakernel serving engine for North Mini Code", §What we
learned: a wrong barrier count hangs or corrupts the step; §The task
scheduler: any wave order must be free of circular waits).

For every wave order and role split, SM counts 1, 2, 7 and 152, batch 1 and
16: the step ends; every counter ends exactly at the target the kernel waits
for; the device-resolved expert shares, or the expert tiles claimed from the
per-layer counters (several tokens), tile their ranges exactly once.  A
target raised by one (the bump word the kernel's time-out test uses, or any
SM count the kernel takes as a target) leaves a wait stuck, which the
interpreter reports.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

from persistent_moe_decode_gb300 import mk
from persistent_moe_decode_gb300.configs import A3B, TINY
from tests._schedule_sim import Deadlock, StepSim, F_BUMP, F_LAYER, F_OP, OP_P1


@pytest.fixture(scope="module", autouse=True)
def built():
    from persistent_moe_decode_gb300 import build
    build.build()


A3B2 = dataclasses.replace(A3B, n_layers=2)
SCHEDULES = ([("waves", o) for o in (mk.MK_WAVES_DEFAULT, mk.MK_WAVES_ATTN_FIRST, mk.MK_WAVES_INTERLEAVED)]
             + [("roles", 0), ("roles", 1)])


def make_step(dims, n_sm, batch, sched, seed):
    rng = np.random.default_rng(seed)
    cfg = mk.make_config(dims, 16, 4096, 1 << 20)
    kind, v = sched
    if kind == "waves":
        cfg.n_attn_claimers = 100000
        cfg.wave_order = v
    else:
        cfg.n_attn_claimers = v                  # 0: chosen per step from the bytes
    if batch == 1:
        lens = np.array([8192 if dims.hidden > 256 else 100], dtype=np.int32)
    else:
        lens = rng.integers(1, 3000, size=batch).astype(np.int32)
    plan = mk.mk_plan_step(cfg, n_sm, batch, lens)
    routing = [np.stack([rng.choice(dims.n_experts, dims.top_k, replace=False) for _ in range(batch)])
               for _ in range(dims.n_layers)]
    return plan, routing, lens


def tiles_once(ranges, total):
    hits = np.zeros(total, dtype=np.int64)
    for lo, hi in ranges:
        assert 0 <= lo <= hi <= total, (lo, hi, total)
        hits[lo:hi] += 1
    return bool(np.all(hits == 1))


def check_step(dims, n_sm, batch, plan, routing, seed, claim_rows=0):
    sim = StepSim(dims, plan, batch, routing, n_sm, claim_rows)
    ctr = sim.run(seed=seed)
    one = batch == 1
    L = dims.n_layers
    meta = plan["meta"]
    for l in range(L):
        want = {("p1", l): n_sm, ("rtr", l): plan["n_rtr_sms"], ("up", l): plan["n_up_sms"],
                ("comb", l): plan["n_comb_sms"],
                ("out", l): n_sm + (plan["n_down_sms"] if one else 0),
                ("down", l): 0 if one else plan["n_down_sms"]}
        for b in range(batch):
            want[("items", l, b)] = int(meta[b][1])
        for k, v in want.items():
            assert ctr.get(k, 0) == v, f"counter {k}: {ctr.get(k, 0)} arrivals, target {v}"
        n_act = len(set(routing[l].reshape(-1).tolist()))
        if one:
            assert tiles_once(sim.coverage["up"][l], n_act * (dims.moe_inter // 8)), "UP groups"
            assert tiles_once(sim.coverage["down"][l], dims.hidden), "DOWN rows"
        else:
            assert tiles_once(sim.coverage["up"][l], n_act * dims.moe_inter), "UP pairs"
            assert tiles_once(sim.coverage["down"][l], n_act * dims.hidden), "DOWN rows"
    assert set(k for k in ctr) <= set(want) | {k for k in ctr if k[1] < L}
    return sim


CASES = [(dims, n_sm, batch, sched)
         for dims in (TINY, A3B2) for n_sm in (1, 2, 7, 152) for batch in (1, 16) for sched in SCHEDULES
         if not (sched[0] == "roles" and n_sm == 1)]


@pytest.mark.parametrize("dims,n_sm,batch,sched", CASES,
                         ids=lambda v: f"H{v.hidden}" if hasattr(v, "hidden") else str(v))
def test_step_ends_with_every_counter_at_its_target(dims, n_sm, batch, sched):
    plan, routing, _ = make_step(dims, n_sm, batch, sched, seed=n_sm * 31 + batch)
    for seed in (0, 1):
        check_step(dims, n_sm, batch, plan, routing, seed)


CLAIM_CASES = [(dims, n_sm, sched, rows) for dims in (TINY, A3B2) for n_sm in (2, 7, 152)
               for sched in (("roles", 0), ("waves", mk.MK_WAVES_DEFAULT)) for rows in (16, 128)]


@pytest.mark.parametrize("dims,n_sm,sched,rows", CLAIM_CASES,
                         ids=lambda v: f"H{v.hidden}" if hasattr(v, "hidden") else str(v))
def test_claimed_expert_tiles_end_with_every_counter_at_its_target(dims, n_sm, sched, rows):
    """Several tokens with the expert tiles claimed from per-layer counters in
    the order the random interleaving gives: every tile is taken exactly once
    and every UP / DOWN counter still ends at its target (one arrival per
    expert-branch SM, whatever it claimed)."""
    plan, routing, _ = make_step(dims, n_sm, 16, sched, seed=n_sm * 7 + rows)
    for seed in (0, 1, 2):
        check_step(dims, n_sm, 16, plan, routing, seed, claim_rows=rows)


@pytest.mark.parametrize("batch", [1, 16])
@pytest.mark.parametrize("dims", [TINY, A3B2], ids=lambda d: f"H{d.hidden}")
def test_a_raised_target_is_reported_as_a_stuck_wait(dims, batch):
    n_sm = 7
    plan, routing, _ = make_step(dims, n_sm, batch, ("roles", 0), seed=5)
    # the bump word of a P1 task (the kernel's own time-out test)
    bumped = dict(plan)
    bumped["tasks"] = plan["tasks"].copy()
    sel = (bumped["tasks"][:, F_OP] == OP_P1) & (bumped["tasks"][:, F_LAYER] == 1)
    bumped["tasks"][sel, F_BUMP] = 1
    with pytest.raises(Deadlock, match="out"):
        StepSim(dims, bumped, batch, routing, n_sm).run(seed=0)
    # every SM count the kernel takes as a counter target, one too high
    for key in ("n_rtr_sms", "n_up_sms", "n_comb_sms") + (() if batch == 1 else ("n_down_sms",)):
        wrong = dict(plan)
        wrong[key] = plan[key] + 1
        with pytest.raises(Deadlock):
            StepSim(dims, wrong, batch, routing, n_sm).run(seed=0)
    # a split count one too high (a sequence's split-KV items)
    wrong = dict(plan)
    wrong["meta"] = plan["meta"].copy()
    wrong["meta"][0, 1] += 1
    with pytest.raises(Deadlock, match="items"):
        StepSim(dims, wrong, batch, routing, n_sm).run(seed=0)


def test_a_wave_order_with_a_circular_wait_is_reported():
    """COMBINE before ATTN on a single SM waits for items only that SM's later
    ATTN task produces: the interpreter must report it."""
    from tests._schedule_sim import OP_ATTN, OP_COMBINE
    plan, routing, _ = make_step(TINY, 1, 1, ("waves", mk.MK_WAVES_DEFAULT), seed=3)
    t = plan["tasks"].copy()
    ia = np.where((t[:, F_OP] == OP_ATTN) & (t[:, F_LAYER] == 0))[0][0]
    ic = np.where((t[:, F_OP] == OP_COMBINE) & (t[:, F_LAYER] == 0))[0][0]
    t[[ia, ic]] = t[[ic, ia]]
    with pytest.raises(Deadlock, match="items"):
        StepSim(TINY, {**plan, "tasks": t}, 1, routing, 1).run(seed=0)
