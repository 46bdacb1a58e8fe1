"""GPU runner and CPU oracle side by side over the same seeded inputs, and the
acceptance checks of a decode trajectory.

The trajectory is teacher-forced by the GPU: each step both sides consume the
GPU's greedy token; each keeps its own KV cache.  Acceptance per step: logits
max-abs <= 2e-2 and relative L2 <= 1e-2; the expert set of every (layer,
token) equal to the oracle's wherever the oracle's k-th / (k+1)-th router-logit
gap exceeds 1e-3; greedy argmax equal on >= 99% of steps.  The kernel keeps
every activation in fp32 (only the appended K/V are BF16, as the cache is) and
is compared with the oracle's plain fp64 definition (no rounding flags).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tests._util import dims_dict, host_pool, host_weights

MAX_ABS, REL_L2, GAP = 2e-2, 1e-2, 1e-3


def oracle_flags(batch: int) -> int:
    return 0


class Pair:
    """GPU runner + oracle over the same inputs."""

    def __init__(self, wl, **cfg_kw):
        from persistent_moe_decode_gb300.runner import StepRunner
        self.wl = wl
        self.run = StepRunner(wl, device="cuda", **cfg_kw)
        self.orc = oracle.Oracle(dims_dict(wl.dims), host_weights(self.run.model),
                                 host_pool(self.run.k_pool), host_pool(self.run.v_pool))

    def step(self, trace=False):
        b = self.run.batch
        b.prepare_step()
        tokens, lens, pt = b.tokens.copy(), b.seq_lens.copy(), b.page_tables.copy()
        self.run.step()
        torch.cuda.synchronize()
        self.run.check_status()
        gpu = self.run.logits.double().cpu().numpy()
        out = self.orc.decode_step(tokens, lens, pt, flags=oracle_flags(self.wl.batch), trace=trace)
        ref, tr = (out if trace else (out, None))
        return gpu, ref, tr

    def advance(self, tokens):
        ch = self.run.advance(tokens)
        if ch is not None:        # mirror the refilled pages into the oracle's pools
            slot, pages = ch
            idx = torch.as_tensor(pages, dtype=torch.long, device=self.run.k_pool.device)
            self.orc.k_pool[:, pages] = host_pool(self.run.k_pool[:, idx])
            self.orc.v_pool[:, pages] = host_pool(self.run.v_pool[:, idx])

    def close(self):
        self.run.close()


def check_logits(gpu, ref, where=""):
    err = np.abs(gpu - ref).max()
    rel = np.linalg.norm(gpu - ref) / np.linalg.norm(ref)
    assert np.all(np.isfinite(gpu)), f"{where}: non-finite logits"
    assert err <= MAX_ABS and rel <= REL_L2, f"{where}: max-abs {err:.3e} rel-L2 {rel:.3e}"
    return err, rel


def check_routing(pair, tr):
    idx, _ = pair.run.dec.routing()
    ok = tr["gap"] > GAP
    for l in range(idx.shape[0]):
        for b in range(idx.shape[1]):
            if ok[l, b]:
                assert set(idx[l, b]) == set(tr["idx"][l, b]), (l, b, idx[l, b], tr["idx"][l, b])
    return int((~ok).sum())


def run_trajectory(pair, steps, trace_every=1, on_step=None):
    """Teacher-forced trajectory; returns (routing checks exempted by the gap
    rule, routing sets compared, steps whose greedy tokens all agreed)."""
    agree, exempt, compared = 0, 0, 0
    for s in range(steps):
        gpu, ref, tr = pair.step(trace=(s % trace_every == 0))
        check_logits(gpu, ref, f"step {s}")
        if tr is not None:
            ex = check_routing(pair, tr)
            exempt += ex
            compared += tr["gap"].size - ex
            if on_step is not None:
                on_step(s, gpu, ref, tr)
        g_tok, r_tok = gpu.argmax(1), ref.argmax(1)
        agree += int((g_tok == r_tok).all())
        pair.advance(g_tok.astype(np.int32))
    assert agree >= 0.99 * steps, f"argmax agreed on {agree}/{steps} steps"
    return exempt, compared, agree


