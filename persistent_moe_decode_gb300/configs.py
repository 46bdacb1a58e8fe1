"""Model shapes and decode workloads for the persistent MoE decode step.

The model is the parallel-layer MoE transformer described in "Inside the
megakernel serving engine for North Mini Code" (§Where the speedup comes from,
parallel transformer layers; §Tasks, the decode graph): every layer runs
attention and the MoE feed-forward from the same normalised input and joins
both with a residual add + RMSNorm.  Five workloads cover it, from a tiny
two-layer model to the 30B-total / 3.3B-active shape at batch 1, batch 16 and
256K context.  This module holds shapes only: no arithmetic of the method.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class ModelDims:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_experts: int
    top_k: int
    moe_inter: int
    vocab: int
    rope_theta: float
    rms_eps: float = 1e-6
    page_size: int = 16

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def group(self) -> int:
        """Query heads that share one KV head (GQA group size)."""
        return self.n_q_heads // self.n_kv_heads

    def layer_dense_bytes(self) -> int:
        """BF16 bytes of one layer's dense weights: W_qkv, W_o, router, norm."""
        H = self.hidden
        return 2 * (self.qkv_rows * H + H * self.n_q_heads * self.head_dim
                    + self.n_experts * H + H)

    def expert_bytes(self, expert_format: str = "bf16") -> int:
        """Bytes of one expert's gate, up and down matrices: BF16, or E4M3
        bytes plus one fp32 scale per row (2 I + H rows)."""
        if expert_format == "fp8":
            return 3 * self.moe_inter * self.hidden + 4 * (2 * self.moe_inter + self.hidden)
        return 2 * 3 * self.moe_inter * self.hidden

    def kv_bytes_per_token(self) -> int:
        """BF16 K+V bytes one cached token costs across all layers."""
        return self.n_layers * 2 * self.n_kv_heads * self.head_dim * 2

    def total_weight_bytes(self) -> int:
        return (self.n_layers * (self.layer_dense_bytes()
                                 + self.n_experts * self.expert_bytes())
                + 2 * 2 * self.vocab * self.hidden + 2 * self.hidden)


@dataclass(frozen=True)
class Workload:
    """One decode workload: a model, a batch, the cached contexts, a step count."""
    name: str
    dims: ModelDims
    batch: int
    context: int                  # cached tokens per sequence before step 0 (batch-1 cases)
    steps: int
    kv_std: float = 1.0
    ragged: tuple[int, int] | None = None   # (lo, hi) uniform context draw for continuous batching
    churn: bool = False           # one sequence finishes and one joins each step
    join_context: int = 1024
    seed: int = 0
    extra: dict = field(default_factory=dict)
    expert_format: str = "bf16"   # "bf16", or "fp8": routed experts in E4M3 + per-row scales

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def max_context(self) -> int:
        hi = self.ragged[1] if self.ragged else self.context
        return max(hi, self.join_context if self.churn else 0)


TINY = ModelDims(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                 n_experts=8, top_k=2, moe_inter=128, vocab=1024, rope_theta=1e4)
MID = ModelDims(n_layers=8, hidden=2048, n_q_heads=16, n_kv_heads=4, head_dim=128,
                n_experts=64, top_k=8, moe_inter=768, vocab=32768, rope_theta=1e4)
A3B = ModelDims(n_layers=48, hidden=2048, n_q_heads=32, n_kv_heads=4, head_dim=128,
                n_experts=128, top_k=8, moe_inter=768, vocab=151936, rope_theta=1e6)

# dense feed-forward layers: one expert that every token selects (E = k = 1;
# a softmax over one router logit is exactly 1, so the layer's MoE branch is
# the dense SwiGLU FFN W_d (SiLU(W_g x) * W_u x))
TINY_DENSE = replace(TINY, n_experts=1, top_k=1, moe_inter=512)
MID_DENSE = replace(MID, n_experts=1, top_k=1, moe_inter=4096)

WORKLOADS = {
    # tiny parallel-layer MoE, batch 1, 64 cached tokens, 8 greedy steps
    "tiny": Workload("tiny", TINY, batch=1, context=64, steps=8),
    # mid MoE, batch 1, 8K cached tokens, 32 steps
    "mid_8k": Workload("mid_8k", MID, batch=1, context=8192, steps=32),
    # 30B-total / 3.3B-active, batch 1, 8K cached tokens, 128 steps
    "a3b_8k": Workload("a3b_8k", A3B, batch=1, context=8192, steps=128),
    # same model, continuous batching: 16 ragged contexts U[1K, 32K], churn 1/step
    "a3b_b16": Workload("a3b_b16", A3B, batch=16, context=0, steps=128,
                        ragged=(1024, 32768), churn=True, join_context=1024),
    # same model, batch 1 at 256K cached tokens, 32 steps
    "a3b_256k": Workload("a3b_256k", A3B, batch=1, context=262144, steps=32),
    # the same model at batch 2 and 4, 8K context each (the schedule ablation)
    "a3b_8k_b2": Workload("a3b_8k_b2", A3B, batch=2, context=8192, steps=128),
    "a3b_8k_b4": Workload("a3b_8k_b4", A3B, batch=4, context=8192, steps=128),
    # small multi-sequence cases for the parity tests: ragged contexts with
    # churn, one token pass (5 sequences) and two passes (12, 16 sequences)
    "tiny_b5": Workload("tiny_b5", TINY, batch=5, context=0, steps=6, ragged=(10, 300),
                        churn=True, join_context=40),
    "tiny_b12": Workload("tiny_b12", TINY, batch=12, context=0, steps=6, ragged=(1, 200),
                         churn=True, join_context=17),
    "mid_b16": Workload("mid_b16", MID, batch=16, context=0, steps=3, ragged=(64, 2048),
                        churn=True, join_context=100),
    # few sequences (the tensor-core GEMVs of dense rows with up to 8 / 4 tokens):
    # the mid model at batch 4, the 30B/3.3B shape cut to 4 layers at batch 3
    "mid_b4": Workload("mid_b4", MID, batch=4, context=0, steps=3, ragged=(64, 2048),
                       churn=True, join_context=100),
    "a3b4_b3": Workload("a3b4_b3", replace(A3B, n_layers=4), batch=3, context=0, steps=3,
                        ragged=(200, 1500), churn=True, join_context=100),
    # 8-bit (E4M3) routed experts with per-row scales, batch 1: the tiny and
    # mid models for parity, the 30B/3.3B shape at 8K for throughput
    "tiny_fp8": Workload("tiny_fp8", TINY, batch=1, context=64, steps=8, expert_format="fp8"),
    "mid_fp8": Workload("mid_fp8", MID, batch=1, context=8192, steps=32, expert_format="fp8"),
    "a3b_8k_fp8": Workload("a3b_8k_fp8", A3B, batch=1, context=8192, steps=128, expert_format="fp8"),
    # attention-heavy several-token case on the mid model (16 sequences at
    # 4K-16K, churn): about 4 GB on the device, for full profiler captures
    "mid_b16_16k": Workload("mid_b16_16k", MID, batch=16, context=0, steps=8, ragged=(4096, 16384),
                            churn=True, join_context=2048),
    # dense-FFN models (one always-selected expert): tiny at batch 1 and 5 with
    # churn, mid (intermediate 4096) at 8K
    "tiny_dense": Workload("tiny_dense", TINY_DENSE, batch=1, context=64, steps=8),
    "tiny_dense_b5": Workload("tiny_dense_b5", TINY_DENSE, batch=5, context=0, steps=6, ragged=(10, 300),
                              churn=True, join_context=40),
    "mid_dense": Workload("mid_dense", MID_DENSE, batch=1, context=8192, steps=32),
    # a dense FFN model whose one expert is 8-bit
    "tiny_dense_fp8": Workload("tiny_dense_fp8", TINY_DENSE, batch=1, context=64, steps=8, expert_format="fp8"),
}


def algorithmic_bytes(dims: ModelDims, n_distinct_experts_per_layer, keys_per_seq,
                      expert_format: str = "bf16") -> int:
    """Bytes one decode step must move (the Speed-of-Light numerator).

    Dense weights of every layer, the distinct routed experts of every layer,
    every cached K/V a sequence attends to (including its new token) and the
    LM head.  The embedding table (B rows read) and activations are excluded.
    ``n_distinct_experts_per_layer`` is a list of per-layer counts.
    """
    dense = dims.n_layers * dims.layer_dense_bytes() + 2 * dims.hidden
    experts = sum(int(n) for n in n_distinct_experts_per_layer) * dims.expert_bytes(expert_format)
    per_tok = dims.n_layers * 2 * dims.n_kv_heads * dims.head_dim * 2
    kv = sum(int(n) for n in keys_per_seq) * per_tok
    lm = 2 * dims.vocab * dims.hidden
    return dense + experts + kv + lm
