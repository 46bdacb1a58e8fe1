"""Seeded synthetic inputs for the decode step: weights, paged KV cache, batches.

This is the only module shared by the CUDA path and the CPU oracle.  It draws
random numbers and manages page bookkeeping; it holds none of the decode
step's arithmetic.

Recipe (the workloads of the pages' own synthetic benchmark, "Inside the
megakernel serving engine for North Mini Code", §Performance: decode against a
synthetic KV cache with random weights):

* every weight matrix: BF16 of N(0, 0.02^2), one generator per (tensor, layer)
  so any subset of layers reproduces the same values;
* RMSNorm gains: BF16 of 1 + 0.02 * N(0, 1) (an all-0.02 gain would make
  activations vanish; the offset keeps a wrong gain index visible);
* KV pools: BF16 of N(0, kv_std^2) in 16-token pages, physical pages taken from
  a seeded random permutation of the pool;
* tokens: uniform over the vocabulary;
* 8-bit experts (``expert_format="fp8"``): the same BF16 expert matrices,
  quantised per output row to the OCP E4M3 encoding with scale
  max|row| / 448 (fp32; 448 is E4M3's largest finite value): byte =
  E4M3(w / scale), round to nearest even.  Both implementations take the
  bytes and scales as their inputs.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass

import numpy as np
import torch

from .configs import ModelDims, Workload

WEIGHT_STD = 0.02

_TENSOR_IDS = {"embed": 1, "lm_head": 2, "final_norm": 3, "attn_norm": 4, "w_qkv": 5,
               "w_o": 6, "w_router": 7, "w_gate": 8, "w_up": 9, "w_down": 10,
               "k_pool": 11, "v_pool": 12, "kv_refill": 13}


def _seed_for(seed: int, name: str, layer: int = -1, extra: int = 0) -> int:
    h = hashlib.sha256(f"{seed}/{_TENSOR_IDS[name]}/{layer}/{extra}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _normal_bf16(shape, seed: int, device, std: float, mean: float = 0.0,
                 chunk_elems: int = 1 << 27) -> torch.Tensor:
    """BF16 tensor of N(mean, std^2) from one seeded generator, built in chunks."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        tmp = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        if mean != 0.0:
            tmp.add_(mean)
        flat[s:e].copy_(tmp)
        del tmp
    return out


@dataclass
class SynthModel:
    """Weights of the parallel-layer MoE model, each stacked over layers.

    Layouts (row-major, BF16):
      embed, lm_head [V, H]; final_norm [H]; attn_norm [L, H];
      w_qkv [L, (hq + 2 hkv) d, H]  rows: all q heads, then k heads, then v heads;
      w_o [L, H, hq d]; w_router [L, E, H];
      w_gate, w_up [L, E, I, H]; w_down [L, E, H, I].
    """
    dims: ModelDims
    embed: torch.Tensor
    lm_head: torch.Tensor
    final_norm: torch.Tensor
    attn_norm: torch.Tensor
    w_qkv: torch.Tensor
    w_o: torch.Tensor
    w_router: torch.Tensor
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor
    # 8-bit experts: q_gate, q_up [L, E, I, H] and q_down [L, E, H, I] uint8
    # (E4M3 codes), s_gate, s_up [L, E, I] and s_down [L, E, H] fp32; the BF16
    # w_gate / w_up / w_down are then empty ([L, 0])
    fp8: dict | None = None

    NAMES = ("embed", "lm_head", "final_norm", "attn_norm", "w_qkv", "w_o",
             "w_router", "w_gate", "w_up", "w_down")
    FP8_NAMES = ("q_gate", "q_up", "q_down", "s_gate", "s_up", "s_down")

    def to(self, device) -> "SynthModel":
        kw = {n: getattr(self, n).to(device) for n in self.NAMES}
        f8 = None if self.fp8 is None else {n: t.to(device) for n, t in self.fp8.items()}
        return SynthModel(self.dims, **kw, fp8=f8)

    def nbytes(self) -> int:
        n = sum(getattr(self, n).numel() * 2 for n in self.NAMES)
        if self.fp8 is not None:
            n += sum(t.numel() * t.element_size() for t in self.fp8.values())
        return n


E4M3_MAX = 448.0


def quantize_e4m3_rows(w: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """Per-row E4M3 quantisation of a [..., rows, cols] BF16 tensor: (codes
    uint8 [..., rows, cols], scales fp32 [..., rows]), scale = max|row| / 448."""
    wf = w.float()
    amax = wf.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (wf / scale.unsqueeze(-1)).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), scale


def make_model(dims: ModelDims, seed: int = 0, device="cpu", expert_format: str = "bf16") -> SynthModel:
    L, H, E, I = dims.n_layers, dims.hidden, dims.n_experts, dims.moe_inter
    V = dims.vocab
    qd = dims.n_q_heads * dims.head_dim

    def stack(name, shape, std=WEIGHT_STD, mean=0.0):
        out = torch.empty((L,) + shape, dtype=torch.bfloat16, device=device)
        for l in range(L):
            out[l] = _normal_bf16(shape, _seed_for(seed, name, l), device, std, mean)
        return out

    fp8 = None
    if expert_format == "fp8":
        fp8 = {}
        for name, shape in (("w_gate", (E, I, H)), ("w_up", (E, I, H)), ("w_down", (E, H, I))):
            q = torch.empty((L,) + shape, dtype=torch.uint8, device=device)
            sc = torch.empty((L,) + shape[:2], dtype=torch.float32, device=device)
            for l in range(L):
                q[l], sc[l] = quantize_e4m3_rows(_normal_bf16(shape, _seed_for(seed, name, l), device,
                                                              WEIGHT_STD))
            fp8["q" + name[1:]] = q
            fp8["s" + name[1:]] = sc
        empty = torch.empty((L, 0), dtype=torch.bfloat16, device=device)
        return SynthModel(
            dims=dims,
            embed=_normal_bf16((V, H), _seed_for(seed, "embed"), device, WEIGHT_STD),
            lm_head=_normal_bf16((V, H), _seed_for(seed, "lm_head"), device, WEIGHT_STD),
            final_norm=_normal_bf16((H,), _seed_for(seed, "final_norm"), device, WEIGHT_STD, 1.0),
            attn_norm=stack("attn_norm", (H,), WEIGHT_STD, 1.0),
            w_qkv=stack("w_qkv", (dims.qkv_rows, H)),
            w_o=stack("w_o", (H, qd)),
            w_router=stack("w_router", (E, H)),
            w_gate=empty, w_up=empty, w_down=empty, fp8=fp8)
    if expert_format != "bf16":
        raise ValueError(f"unknown expert format {expert_format!r}")

    return SynthModel(
        dims=dims,
        embed=_normal_bf16((V, H), _seed_for(seed, "embed"), device, WEIGHT_STD),
        lm_head=_normal_bf16((V, H), _seed_for(seed, "lm_head"), device, WEIGHT_STD),
        final_norm=_normal_bf16((H,), _seed_for(seed, "final_norm"), device, WEIGHT_STD, 1.0),
        attn_norm=stack("attn_norm", (H,), WEIGHT_STD, 1.0),
        w_qkv=stack("w_qkv", (dims.qkv_rows, H)),
        w_o=stack("w_o", (H, qd)),
        w_router=stack("w_router", (E, H)),
        w_gate=stack("w_gate", (E, I, H)),
        w_up=stack("w_up", (E, I, H)),
        w_down=stack("w_down", (E, H, I)),
    )


def make_kv_pools(dims: ModelDims, num_pages: int, kv_std: float, seed: int = 0,
                  device="cpu"):
    """K and V pools, each [L, num_pages, hkv, P, d] BF16 of N(0, kv_std^2)."""
    shape = (num_pages, dims.n_kv_heads, dims.page_size, dims.head_dim)
    L = dims.n_layers
    k = torch.empty((L,) + shape, dtype=torch.bfloat16, device=device)
    v = torch.empty((L,) + shape, dtype=torch.bfloat16, device=device)
    for l in range(L):
        k[l] = _normal_bf16(shape, _seed_for(seed, "k_pool", l), device, kv_std)
        v[l] = _normal_bf16(shape, _seed_for(seed, "v_pool", l), device, kv_std)
    return k, v


class DecodeBatch:
    """Host-side batch state: cached lengths, page tables, next tokens.

    Pages come from a seeded random permutation of the pool, so a sequence's
    logical pages are scattered over physical pages.  A page is taken when a
    sequence's next position crosses into it.  With churn, one live slot is
    retired each step (its pages return to the free list) and a new sequence
    joins in its place with ``join_context`` cached tokens.
    """

    def __init__(self, wl: Workload, seed: int | None = None):
        self.wl = wl
        self.dims = wl.dims
        self.rng = np.random.default_rng(wl.seed if seed is None else seed)
        B, P = wl.batch, wl.dims.page_size
        if wl.ragged:
            lo, hi = wl.ragged
            ctx = self.rng.integers(lo, hi + 1, size=B)
        else:
            ctx = np.full(B, wl.context)
        self.seq_lens = ctx.astype(np.int32)
        self.max_pages = math.ceil((wl.max_context + wl.steps + 1) / P)
        need = sum(math.ceil((int(c) + wl.steps + 1) / P) for c in ctx)
        if wl.churn:
            need += wl.steps * math.ceil((wl.join_context + wl.steps + 1) / P)
        self.num_pages = int(need)
        perm = self.rng.permutation(self.num_pages).astype(np.int32)
        self.free = list(perm[::-1])   # pop() from the end = next of the permutation
        self.page_tables = np.full((B, self.max_pages), -1, dtype=np.int32)
        self.n_pages = np.zeros(B, dtype=np.int32)
        for b in range(B):
            self._grow(b, int(self.seq_lens[b]) + 1)
        self.tokens = self.rng.integers(0, wl.dims.vocab, size=B).astype(np.int32)
        self.seq_ids = np.arange(B, dtype=np.int32)
        self.next_seq_id = B

    def _grow(self, b: int, n_tokens: int) -> list[int]:
        P = self.dims.page_size
        want = math.ceil(n_tokens / P)
        added = []
        while self.n_pages[b] < want:
            pg = int(self.free.pop())
            self.page_tables[b, self.n_pages[b]] = pg
            self.n_pages[b] += 1
            added.append(pg)
        return added

    def prepare_step(self) -> None:
        """Make sure every sequence owns the page that its new token lands in."""
        for b in range(self.wl.batch):
            self._grow(b, int(self.seq_lens[b]) + 1)

    def advance(self, next_tokens) -> None:
        self.seq_lens += 1
        self.tokens = np.asarray(next_tokens, dtype=np.int32).copy()

    def churn(self) -> tuple[int, list[int]]:
        """Retire one live slot and admit a new sequence there.

        Returns (slot, new physical pages); the caller refills those pages with
        fresh random K/V so the joining sequence sees a new synthetic prefix.
        """
        B, P = self.wl.batch, self.dims.page_size
        slot = int(self.rng.integers(0, B))
        for i in range(int(self.n_pages[slot])):
            self.free.append(int(self.page_tables[slot, i]))
        # keep the free list in random order
        self.rng.shuffle(self.free)
        self.page_tables[slot, :] = -1
        self.n_pages[slot] = 0
        self.seq_lens[slot] = self.wl.join_context
        added = self._grow(slot, self.wl.join_context + 1)
        self.tokens[slot] = int(self.rng.integers(0, self.dims.vocab))
        self.seq_ids[slot] = self.next_seq_id
        self.next_seq_id += 1
        return slot, added


def refill_pages(k_pool: torch.Tensor, v_pool: torch.Tensor, pages, kv_std: float,
                 seed: int, step: int) -> None:
    """Overwrite the given physical pages of every layer with fresh N(0, kv_std^2)."""
    if not pages:
        return
    dims_shape = k_pool.shape[2:]
    idx = torch.as_tensor(list(pages), dtype=torch.long, device=k_pool.device)
    for l in range(k_pool.shape[0]):
        shape = (len(pages),) + tuple(dims_shape)
        k_pool[l, idx] = _normal_bf16(shape, _seed_for(seed, "kv_refill", l, 2 * step), k_pool.device, kv_std)
        v_pool[l, idx] = _normal_bf16(shape, _seed_for(seed, "kv_refill", l, 2 * step + 1), v_pool.device, kv_std)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 view of a contiguous CPU BF16 tensor (no copy)."""
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
