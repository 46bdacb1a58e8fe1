"""Drives a synthetic decode workload through the C ABI (no arithmetic here).

``StepRunner`` owns the device weights and KV pools of one workload, the
host-side batch bookkeeping (page tables, lengths, churn) and one decoder
handle; ``step()`` schedules and launches one decode step.
"""
from __future__ import annotations

import numpy as np
import torch

from .configs import Workload
from .mk import Decoder
from .synth import DecodeBatch, make_kv_pools, make_model, refill_pages


class StepRunner:
    def __init__(self, wl: Workload, device="cuda", seed: int | None = None, model=None,
                 **cfg_kw):
        self.wl = wl
        self.dims = wl.dims
        self.seed = wl.seed if seed is None else seed
        self.device = torch.device(device)
        self.model = model if model is not None else make_model(wl.dims, self.seed, self.device,
                                                                 wl.expert_format)
        self.batch = DecodeBatch(wl, self.seed)
        self.k_pool, self.v_pool = make_kv_pools(wl.dims, self.batch.num_pages, wl.kv_std,
                                                 self.seed, self.device)
        self.dec = Decoder(self.model, self.k_pool, self.v_pool, max_batch=wl.batch,
                           max_pages_per_seq=self.batch.max_pages, **cfg_kw)
        self.logits = torch.empty(wl.batch, wl.dims.vocab, dtype=torch.float32, device=self.device)
        self.step_index = 0

    def schedule(self, stream=None):
        b = self.batch
        b.prepare_step()
        self.dec.schedule(b.tokens, b.page_tables, b.seq_lens, seq_ids=b.seq_ids, stream=stream)

    def launch(self, stream=None):
        self.dec.decode(self.logits, stream)

    def step(self, stream=None):
        self.schedule(stream)
        self.launch(stream)

    def check_status(self):
        rc, err = self.dec.status()
        if rc != 0:
            raise RuntimeError(f"device step failed: {rc} {err.as_dict()}")

    def greedy(self) -> np.ndarray:
        return self.logits.argmax(dim=1).to(torch.int32).cpu().numpy()

    def advance(self, next_tokens, refill: bool = True) -> tuple[int, list[int]] | None:
        """Append the step's token; with churn, retire one sequence and admit one.

        ``refill`` draws fresh K/V for the joining sequence's pages (input
        synthesis).  Without it the pages keep the random K/V they already hold
        (a retired sequence's), which is as good a synthetic prefix and keeps
        the random-number kernels out of a timed loop."""
        self.batch.advance(next_tokens)
        self.step_index += 1
        if self.wl.churn:
            slot, pages = self.batch.churn()
            if refill:
                refill_pages(self.k_pool, self.v_pool, pages, self.wl.kv_std, self.seed, self.step_index)
            return slot, pages
        return None

    def close(self):
        self.dec.close()
