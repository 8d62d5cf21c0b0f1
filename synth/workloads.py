"""Synthetic workloads of the shard step: unit shapes, virtual-rank counts and input recipes.

Shapes are architecture shapes only (no weights, no data): the parameter
tensors of each model in module-definition order, which is the order a
flattening wrapper concatenates them in. Every input tensor is a seeded
`synth` stream; nothing here does any of the shard step's arithmetic.

Streams: gradient of virtual rank r at optimizer step t is
``normal(..., kind=GRAD, rank=r, step=t)``; master/m/v use step 0 and are
indexed by the element's position in the unit's flat parameter vector.

Distributions: every "N(0, s)" below is the generator's Irwin-Hall
approximation of a normal (the centred sum of twelve uniforms, scaled to
variance s^2, so its support ends at +-6s), truncated toward zero onto the
target format's grid; "|N(0, s)|" is its absolute value and "U(-a, a)" one
53-bit uniform draw, truncated likewise.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable

from . import BF16, FP16, FP32, GRAD, MASTER, MOM1, MOM2, PARAM16, Spec, normal, uniform


def tiny_mlp_numels() -> list[int]:
    """Two-layer MLP: W1 [256,128], b1 [128], W2 [512,256], b2 [256] (164,224 params)."""
    return [256 * 128, 128, 512 * 256, 256]


def gpt2_small_numels() -> list[int]:
    """GPT-2 small (12 layers, d=768, vocab 50257, context 1024, tied head): 124,439,808 params."""
    d, v, ctx, ff = 768, 50257, 1024, 3072
    out = [v * d, ctx * d]
    for _ in range(12):
        out += [d, d,                      # ln_1 weight, bias
                d * 3 * d, 3 * d,          # attn.c_attn weight, bias
                d * d, d,                  # attn.c_proj weight, bias
                d, d,                      # ln_2 weight, bias
                d * ff, ff,                # mlp.c_fc weight, bias
                ff * d, d]                 # mlp.c_proj weight, bias
    out += [d, d]                          # ln_f weight, bias
    return out


def llama3_8b_numels() -> list[int]:
    """Llama-3-8B (32 layers, d=4096, ffn 14336, 32 q / 8 kv heads of 128, vocab 128256, untied head)."""
    d, ff, v, kv = 4096, 14336, 128256, 8 * 128
    out = [v * d]
    for _ in range(32):
        out += [d, d * d, kv * d, kv * d, d * d, d, ff * d, ff * d, d * ff]
    out += [d, v * d]
    return out


def llama70b_layer_numels() -> list[int]:
    """One Llama-70B decoder layer (d=8192, ffn 28672, 64 q / 8 kv heads of 128): 855,654,400 params."""
    d, ff, kv = 8192, 28672, 8 * 128
    return [d, d * d, kv * d, kv * d, d * d, d, ff * d, ff * d, d * ff]


@dataclass
class Workload:
    name: str
    numels: list[int]
    n_ranks: int
    gdtype: int                                  # gradient / parameter 16-bit format
    grad: Callable[[int, int], Spec]             # (rank, step) -> spec
    master: Spec
    m: Spec | None                               # None: zeros
    v: Spec | None
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    first_step: int = 1
    warmup_steps: int = 0
    steps: int = 1
    shards: list[int] = field(default_factory=lambda: [0])   # shards that are stepped
    unshard: bool = False
    reshard: bool = False
    per_rank_full: bool = True                   # rank gradient buffers hold the full unit (else one shard)
    param16: Callable[[int], Spec] | None = None  # 16-bit params of shards that are not stepped

    @property
    def P(self) -> int:
        return sum(self.numels)

    def hp(self, step: int) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay, step=step)


def tiny_mlp(seed: int = 0) -> Workload:
    """Tiny MLP flat unit, N=4, all 4 shards stepped for 3 steps, then unshard."""
    return Workload("tiny-mlp-164k-N4", tiny_mlp_numels(), 4, BF16,
                    grad=lambda r, t: normal(1e-3, BF16, GRAD, r, t, seed),
                    master=normal(0.02, FP32, MASTER, seed=seed), m=None, v=None,
                    steps=3, shards=[0, 1, 2, 3], unshard=True)


def gpt2_small(seed: int = 0) -> Workload:
    """GPT-2 small, N=8: rank-0 shard, m/v from 5 warm-up steps, 10 steps, then the full unshard."""
    return Workload("gpt2-small-124M-N8-rank0", gpt2_small_numels(), 8, BF16,
                    grad=lambda r, t: normal(1e-3, BF16, GRAD, r, t, seed),
                    master=normal(0.02, FP32, MASTER, seed=seed), m=None, v=None,
                    warmup_steps=5, steps=10, shards=[0], unshard=True,
                    param16=lambda k: normal(0.02, BF16, PARAM16, k, 0, seed))


def llama3_8b_shard(seed: int = 0) -> Workload:
    """Llama-3-8B, N=8, one 1/8 shard (rank 0): bf16 grads N(0,1e-4) with 1% of entries x100.

    The other seven shards' bf16 parameters (for the unshard into the flat unit) are seeded
    N(0, 0.02) streams of their own."""
    return Workload("llama3-8b-shard0-N8", llama3_8b_numels(), 8, BF16,
                    grad=lambda r, t: normal(1e-4, BF16, GRAD, r, t, seed, outlier_every=100, outlier_mult=100.0),
                    master=normal(0.02, FP32, MASTER, seed=seed), m=None, v=None,
                    steps=1, shards=[0], per_rank_full=False,
                    param16=lambda k: normal(0.02, BF16, PARAM16, k, 0, seed))


def llama70b_layer(seed: int = 0) -> Workload:
    """Llama-70B decoder layer, N=64, all shards, fp16 grads U(-6e-5, 6e-5), unshard + reshard."""
    return Workload("llama70b-layer-N64-fp16", llama70b_layer_numels(), 64, FP16,
                    grad=lambda r, t: uniform(6e-5, FP16, GRAD, r, t, seed),
                    master=normal(0.02, FP32, MASTER, seed=seed), m=None, v=None,
                    steps=1, shards=list(range(64)), unshard=True, reshard=True)


SWEEP_SIZES = [4099, (1 << 20) + 7, 1 << 26, (1 << 28) + 3, 1 << 30]
SWEEP_RANKS = [2, 8, 64]


def sweep(n: int, n_ranks: int, seed: int = 0) -> Workload:
    """Single flat fp32 shard of n elements (shard 0 of a unit of N*n), N virtual ranks, at step 1000."""
    return Workload(f"sweep-n{n}-N{n_ranks}", [n * n_ranks], n_ranks, BF16,
                    grad=lambda r, t: normal(1e-3, BF16, GRAD, r, t, seed),
                    master=normal(0.02, FP32, MASTER, seed=seed),
                    m=normal(1e-4, FP32, MOM1, seed=seed),
                    v=normal(1e-8, FP32, MOM2, seed=seed, absolute=True),
                    lr=3e-4, weight_decay=0.1, first_step=1000, steps=1, shards=[0],
                    per_rank_full=False)
