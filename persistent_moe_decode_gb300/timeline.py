"""Per-layer task timeline of the persistent decode step.

    python -m persistent_moe_decode_gb300.timeline --workload a3b_8k [--steps 4] [--out t.npy]

Runs a few decode steps with the task timeline kept (``config.trace_records``:
the kernel instances that record it carry the clock reads; the timed
instances do not), then prints for the last step:

* per branch (attention SMs, expert SMs) and phase, medians over the middle
  layers of when the tasks were handed over, started, had their inputs, got
  their first stage, consumed their last stage and ended, in microseconds
  after the end of the previous layer (its last OUT task);
* the median layer length and the final (LM-head) phase;
* the idle share: per SM, the fraction of the step spent outside any task
  (waiting for a task's hand-over), as median and maximum over the SMs.

The timeline instances run slower than the timed ones (about 5 %): the
shares and orderings are what it is for, not absolute times.
"""
from __future__ import annotations

import argparse

import numpy as np

NAMES = {1: "P1", 2: "ROUTE", 3: "ATTN", 4: "UP", 5: "COMBINE", 6: "OUT", 7: "FINAL", 8: "DOWN"}


def capture(workload: str, steps: int, records: int = 4096):
    import torch

    from .configs import WORKLOADS
    from .runner import StepRunner
    run = StepRunner(WORKLOADS[workload], device="cuda", trace_records=records)
    try:
        for _ in range(steps):
            run.step()
            torch.cuda.synchronize()
            run.check_status()
            run.advance(run.greedy())
        return run.dec.trace()
    finally:
        run.close()


def summarize(tr: np.ndarray) -> str:
    tr = tr.astype(np.int64)
    tr = tr[tr[:, 0] >= 0]
    t0 = (tr[:, 3] & 0xffffffff) | (tr[:, 4] << 32)
    base = t0.min()
    start = (t0 - base) / 1e3
    ready = start + tr[:, 5] / 1e3
    end = start + tr[:, 6] / 1e3
    st0 = start + tr[:, 8] / 1e3
    std = start + tr[:, 9] / 1e3
    hand = start + tr[:, 13] / 1e3
    op, lay, sm = tr[:, 0], tr[:, 1], tr[:, 7]
    L = int(lay[op != 7].max()) + 1
    attn_sms = set(sm[op == 3].tolist())
    is_attn = np.array([s in attn_sms for s in sm])
    lo, hi = max(1, L // 8), max(2, L - L // 8)
    out = []
    layer_len = [end[(op == 6) & (lay == l)].max() - end[(op == 6) & (lay == l - 1)].max() for l in range(lo, hi)]
    out.append(f"layers {lo}..{hi - 1}: median layer {np.median(layer_len):.1f} us "
               f"(min {np.min(layer_len):.1f}, max {np.max(layer_len):.1f})")
    for branch, bm in (("attention SMs", is_attn), ("expert SMs", ~is_attn)):
        if not bm.any():
            continue
        out.append(f"{branch} ({len(set(sm[bm].tolist()))}), us after the previous layer's end:")
        out.append("  phase       hand  start  ready    st0    stD    end  max-end")
        for o, name in NAMES.items():
            if o == 7:
                continue
            rows = []
            for l in range(lo, hi):
                ref = end[(op == 6) & (lay == l - 1)].max()
                m = (op == o) & (lay == l) & bm
                if m.any():
                    rows.append([np.median(a[m]) - ref for a in (hand, start, ready, st0, std, end)]
                                + [end[m].max() - ref])
            if rows:
                a = np.median(np.array(rows), axis=0)
                out.append(f"  {name:9s} " + " ".join(f"{x:6.1f}" for x in a))
    fin = op == 7
    if fin.any():
        ref = end[(op == 6) & (lay == L - 1)].max()
        out.append(f"final phase (LM head): {end[fin].max() - ref:.1f} us")
    idle = []
    for s in np.unique(sm):
        m = sm == s
        span = end[m].max() - start[m].min()
        busy = (end[m] - start[m]).sum()
        idle.append(1.0 - busy / span if span > 0 else 0.0)
    out.append(f"idle share per SM (outside any task): median {np.median(idle) * 100:.1f} %, "
               f"max {np.max(idle) * 100:.1f} %")
    out.append(f"step {end.max() - start.min():.1f} us")
    return "\n".join(out)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="a3b_8k")
    ap.add_argument("--steps", type=int, default=4)
    ap.add_argument("--out", default=None)
    args = ap.parse_args()
    tr = capture(args.workload, args.steps)
    if args.out:
        np.save(args.out, tr)
    print(summarize(tr))


if __name__ == "__main__":
    main()
