"""The per-layer timeline summary (timeline.summarize) on a synthetic trace
whose medians, layer length, final phase and idle shares are known (CPU)."""
from __future__ import annotations

import numpy as np

from persistent_moe_decode_gb300.timeline import summarize

L = 8
BASE_NS = 6_500_000_000      # the low word is above 2^31: negative as the int32 the device stores


def _rec(op, layer, sm, t0_us, t1_us, hand_us=None):
    r = np.zeros(16, dtype=np.int64)
    t0 = BASE_NS + int(t0_us * 1000)
    r[0], r[1], r[7] = op, layer, sm
    r[3], r[4] = t0 & 0xffffffff, t0 >> 32
    r[6] = int((t1_us - t0_us) * 1000)
    if hand_us is not None:
        r[13] = int((hand_us - t0_us) * 1000)
    return r


def _trace():
    recs = []
    for l in range(L):
        b = 100.0 * l
        # SM 0, attention branch: P1, ATTN, COMBINE, OUT (ends 10 us before the layer does)
        recs += [_rec(1, l, 0, b, b + 10, hand_us=b - 5), _rec(3, l, 0, b + 10, b + 60),
                 _rec(5, l, 0, b + 60, b + 70), _rec(6, l, 0, b + 70, b + 90)]
        # SM 1, expert branch: P1, ROUTE, UP, DOWN, OUT (its OUT ends the layer)
        recs += [_rec(1, l, 1, b, b + 10), _rec(2, l, 1, b + 10, b + 15), _rec(4, l, 1, b + 15, b + 60),
                 _rec(8, l, 1, b + 60, b + 80), _rec(6, l, 1, b + 80, b + 100)]
    recs += [_rec(7, L, 0, 800, 850), _rec(7, L, 1, 800, 850)]
    tr = np.stack(recs)
    return tr.astype(np.uint32).view(np.int32)        # the device's int32 words


def test_summary_of_a_known_trace():
    out = summarize(_trace())
    lines = out.splitlines()
    assert lines[0].startswith("layers 1..6: median layer 100.0 us")
    assert "attention SMs (1)" in out and "expert SMs (1)" in out
    # phases unique to one branch (P1 and OUT appear in both tables)
    row = {ln.split()[0]: [float(v) for v in ln.split()[1:]] for ln in lines
           if ln.split() and ln.split()[0] in ("ATTN", "COMBINE", "ROUTE", "UP", "DOWN")}
    # the first table is the attention branch: P1 handed 5 us early, starts at 0, ends at 10
    attn_p1 = next(ln for ln in lines if ln.strip().startswith("P1"))
    hand, start, ready, st0, std, end, mx = (float(v) for v in attn_p1.split()[1:])
    assert (hand, start, end, mx) == (-5.0, 0.0, 10.0, 10.0)
    assert row["ATTN"][1] == 10.0 and row["ATTN"][5] == 60.0
    assert row["DOWN"][1] == 60.0 and row["DOWN"][5] == 80.0
    assert "final phase (LM head): 50.0 us" in out
    # SM 0 is idle 10 us a layer: 80 of 850 us; SM 1 never
    assert "idle share per SM (outside any task): median 4.7 %, max 9.4 %" in out
    assert lines[-1] == "step 850.0 us"
