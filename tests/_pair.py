"""GPU runner and CPU oracle side by side over the same seeded inputs, and the
acceptance checks of a decode trajectory.

The trajectory is teacher-forced by the GPU: each step both sides consume the
GPU's greedy token; each keeps its own KV cache.  Acceptance per step: logits
max-abs <= 2e-2 and relative L2 <= 1e-2; the expert set of every (layer,
token) equal to the oracle's wherever the oracle's k-th / (k+1)-th router-logit
gap exceeds 1e-3; greedy argmax equal on >= 99% of the (step, sequence)
pairs.  The kernel keeps
every activation in fp32 (only the appended K/V are BF16, as the cache is) and
is compared with the oracle's plain fp64 definition (no rounding flags).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tests._util import dims_dict, host_fp8, host_pool, host_weights

MAX_ABS, REL_L2, GAP = 2e-2, 1e-2, 1e-3


def oracle_flags(batch: int) -> int:
    return 0


def oracle_step_following_ties(orc, tokens, lens, pt, gpu_idx, flags=0):
    """The oracle's step.  Where the GPU decided a near tie the other way (the
    oracle's k-th / (k+1)-th router gap <= GAP, within what fp32 rounding can
    swap, and the routed sets differ), the step is run again with the GPU's
    experts imposed there (orc_decode_step_forced), so that everything after
    the tie is compared like for like; repeated while new such ties appear.
    Returns (logits, trace, number of imposed (layer, token) choices)."""
    ref, tr = orc.decode_step(tokens, lens, pt, flags=flags, trace=True)
    L, B = tr["gap"].shape
    mask = np.zeros((L, B), dtype=bool)
    for _ in range(16):
        differ = np.array([[set(gpu_idx[l, b].tolist()) != set(tr["idx"][l, b].tolist()) for b in range(B)]
                           for l in range(L)])
        tie = differ & (tr["gap"] <= GAP) & ~mask
        if not tie.any():
            break
        mask |= tie
        ref, tr = orc.decode_step(tokens, lens, pt, flags=flags, trace=True, force=(gpu_idx, mask))
    return ref, tr, int(mask.sum())


class Pair:
    """GPU runner + oracle over the same inputs."""

    def __init__(self, wl, **cfg_kw):
        from persistent_moe_decode_gb300.runner import StepRunner
        self.wl = wl
        self.run = StepRunner(wl, device="cuda", **cfg_kw)
        self.orc = oracle.Oracle(dims_dict(wl.dims), host_weights(self.run.model),
                                 host_pool(self.run.k_pool), host_pool(self.run.v_pool),
                                 fp8=host_fp8(self.run.model))

    def step(self, trace=False):
        b = self.run.batch
        b.prepare_step()
        tokens, lens, pt = b.tokens.copy(), b.seq_lens.copy(), b.page_tables.copy()
        self.run.step()
        torch.cuda.synchronize()
        self.run.check_status()
        gpu = self.run.logits.double().cpu().numpy()
        gidx, _ = self.run.dec.routing()
        ref, tr, forced = oracle_step_following_ties(self.orc, tokens, lens, pt, gidx,
                                                     oracle_flags(self.wl.batch))
        self.forced = getattr(self, "forced", 0) + forced
        return gpu, ref, (tr if trace else None)

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


def diagnose(pair, gpu, ref, tr):
    """Per sequence: logits max-abs, the smallest oracle router gap over the
    layers, and the layers whose routed sets differ."""
    idx, _ = pair.run.dec.routing()
    out = []
    for b in range(gpu.shape[0]):
        bad = [l for l in range(idx.shape[0]) if set(idx[l, b]) != set(tr["idx"][l, b])] if tr else []
        gap = float(tr["gap"][:, b].min()) if tr else float("nan")
        out.append(f"seq {b}: max-abs {np.abs(gpu[b] - ref[b]).max():.2e} min-gap {gap:.2e} sets differ at {bad}")
    return "\n".join(out)


def run_trajectory(pair, steps, trace_every=1, on_step=None):
    """Teacher-forced trajectory; returns (routing checks exempted by the gap
    rule, routing sets compared, (step, sequence) pairs whose greedy tokens
    agreed).  Near
    ties the GPU decided the other way are imposed on the oracle
    (oracle_step_following_ties; counted in pair.forced)."""
    agree, exempt, compared, pairs = 0, 0, 0, 0
    misses = []
    for s in range(steps):
        gpu, ref, tr = pair.step(trace=(s % trace_every == 0))
        try:
            err, rel = check_logits(gpu, ref, f"step {s}")
        except AssertionError as e:
            raise AssertionError(f"{e}\n{diagnose(pair, gpu, ref, tr)}") from None
        pair.worst = max(getattr(pair, "worst", (0.0, 0.0)), (float(err), float(rel)))
        if tr is not None:
            ex = check_routing(pair, tr)
            exempt += ex
            compared += tr["gap"].size - ex
            if on_step is not None:
                on_step(s, gpu, ref, tr)
        g_tok, r_tok = gpu.argmax(1), ref.argmax(1)
        agree += int((g_tok == r_tok).sum())
        pairs += len(g_tok)
        for b in np.nonzero(g_tok != r_tok)[0]:
            top = np.sort(ref[b])[-2:]
            misses.append(f"step {s} seq {b}: oracle top-2 gap {top[1] - top[0]:.2e}")
        pair.advance(g_tok.astype(np.int32))
    # the greedy token of every (step, sequence) pair: equal on >= 99 % of them
    assert agree >= 0.99 * pairs, f"argmax agreed on {agree}/{pairs} (step, sequence) pairs: {misses}"
    return exempt, compared, agree


