"""Glue between the seeded input generators and the two implementations.

Tests build inputs with ``persistent_moe_decode_gb300.synth`` and hand the
same values to the CPU oracle (host uint16 views) and to the CUDA path
(device tensors through the C-ABI binding).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from persistent_moe_decode_gb300.configs import ModelDims
from persistent_moe_decode_gb300.synth import SynthModel, bf16_bits


def dims_dict(d: ModelDims, n_layers: int | None = None) -> dict:
    out = dataclasses.asdict(d)
    if n_layers is not None:
        out["n_layers"] = n_layers
    return out


def host_weights(model: SynthModel) -> dict:
    """uint16 views of a CPU copy of every weight (copies device tensors)."""
    out = {}
    for n in SynthModel.NAMES:
        t = getattr(model, n)
        if t.device.type != "cpu":
            t = t.cpu()
        out[n] = bf16_bits(t.contiguous())
    return out


def host_pool(t: torch.Tensor) -> np.ndarray:
    if t.device.type != "cpu":
        t = t.cpu()
    return bf16_bits(t.contiguous()).copy()


def host_fp8(model: SynthModel) -> dict | None:
    """Host numpy copies of the 8-bit experts (codes uint8, scales float32), or None."""
    if model.fp8 is None:
        return None
    return {n: t.cpu().contiguous().numpy() for n, t in model.fp8.items()}


def make_oracle(model: SynthModel, k_pool: torch.Tensor, v_pool: torch.Tensor):
    import oracle
    return oracle.Oracle(dims_dict(model.dims), host_weights(model), host_pool(k_pool),
                         host_pool(v_pool), fp8=host_fp8(model))
