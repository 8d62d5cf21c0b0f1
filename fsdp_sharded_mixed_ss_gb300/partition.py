"""One shard per GPU: the real-rank form of the shard step.

Page: "FSDP: Fully Sharded Data Parallel Training at Scale" -- how FSDP shards a
layer (rank k owns elements [floor(kP/N), floor((k+1)P/N)) of the unit's flat
parameter vector, and the gradients, master copy and Adam moments at the same
positions) and the FSDP unit communication cycle (backward ends with a
reduce-scatter of the gradients, every rank steps its own shard with no
communication, and the next forward starts with an all-gather of the 16-bit
parameters).

On one GPU the library runs the N ranks as virtual ranks whose gradient
buffers all sit in local HBM. Across N GPUs the same kernels run per rank, and
the two exchanges move the data around them:

* gradients: the reduce-scatter is split into its data movement and its
  arithmetic. An all-to-all with the shards' uneven lengths sends rank r's
  16-bit gradient slice of shard k to rank k, where the N slices land as the N
  rows that ss_adam_step (or ss_grad_reduce) reads, and the fused kernel adds
  them in rank order in fp32. The result is the virtual-rank result bit for bit
  (a ring reduce-scatter would add in an order set by each rank's place in the
  ring). Per rank the link carries (N-1)/N x 2P bytes each way, what a ring
  reduce-scatter of 16-bit gradients carries; the receive buffer holds N rows
  of the shard, 2P/N x N bytes.
* parameters: each rank's 16-bit shard, padded to the longest shard
  (ceil(P/N) elements; floor(kP/N) shards differ by one element at most), is
  all-gathered into N rows, and ss_unshard places row k at floor(kP/N) of the
  flat unit buffer.

The exchanges move bytes only (uint8 views of the 16-bit buffers): no
arithmetic happens in a collective. They run on torch.distributed (NCCL
between GPUs; gloo moves CPU tensors the same way), on torch's current stream,
like the library's kernels. Remote data always lands in a local buffer before a
kernel reads it.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Sequence

import numpy as np

from . import ss_adam_step, ss_flatten_layout, ss_shard_segments, ss_unshard


@dataclass
class Partition:
    """The floor(kP/N) partition of one unit over `world` ranks, seen from `rank`."""

    numels: Sequence[int]
    world: int
    rank: int
    offsets: np.ndarray = field(init=False)
    bounds: np.ndarray = field(init=False)

    def __post_init__(self):
        if not 0 <= self.rank < self.world:
            raise ValueError(f"rank {self.rank} outside a world of {self.world}")
        self.offsets, self.bounds = ss_flatten_layout(list(self.numels), self.world)

    @property
    def P(self) -> int:
        return int(self.bounds[-1])

    @property
    def lo(self) -> int:
        return int(self.bounds[self.rank])

    @property
    def hi(self) -> int:
        return int(self.bounds[self.rank + 1])

    @property
    def n(self) -> int:
        """Length of this rank's shard."""
        return self.hi - self.lo

    @property
    def lengths(self) -> list[int]:
        return [int(self.bounds[k + 1] - self.bounds[k]) for k in range(self.world)]

    @property
    def max_len(self) -> int:
        """Row length of the parameter all-gather: the longest shard."""
        return max(self.lengths)

    def segments(self, shard: int | None = None):
        """(tensor, tensor_offset, shard_offset, length) pieces of a shard (default: this rank's)."""
        return ss_shard_segments(self.offsets, self.bounds, self.rank if shard is None else shard)


def _bytes(t):
    """The tensor's storage as uint8 (contiguous tensors only)."""
    import torch

    if not t.is_contiguous():
        raise ValueError("the exchanges need contiguous buffers")
    return t.view(torch.uint8)


def exchange_grads(full_grad16, part: Partition, out=None, group=None):
    """The data movement of the gradient reduce-scatter: returns (or fills) `out`, a
    (world, part.n) tensor of full_grad16's dtype whose row r is rank r's gradient slice
    [part.lo, part.hi). full_grad16: this rank's 16-bit gradient of the whole unit (P elements)."""
    import torch
    import torch.distributed as dist

    if full_grad16.numel() != part.P:
        raise ValueError(f"gradient has {full_grad16.numel()} elements, the unit {part.P}")
    if out is None:
        out = torch.empty((part.world, part.n), dtype=full_grad16.dtype, device=full_grad16.device)
    if tuple(out.shape) != (part.world, part.n) or out.dtype != full_grad16.dtype:
        raise ValueError("out must be (world, shard length) of the gradient's dtype")
    es = full_grad16.element_size()
    dist.all_to_all_single(_bytes(out).view(-1), _bytes(full_grad16).view(-1),
                           output_split_sizes=[part.n * es] * part.world,
                           input_split_sizes=[k * es for k in part.lengths], group=group)
    return out


def gather_params(shard16_padded, part: Partition, out=None, group=None):
    """The data movement of the parameter all-gather: returns (or fills) `out`, a
    (world, part.max_len) tensor whose row k holds rank k's 16-bit shard in its first
    lengths[k] elements. shard16_padded: this rank's shard, part.max_len elements."""
    import torch
    import torch.distributed as dist

    if shard16_padded.numel() != part.max_len:
        raise ValueError(f"the padded shard must have {part.max_len} elements")
    if out is None:
        out = torch.empty((part.world, part.max_len), dtype=shard16_padded.dtype, device=shard16_padded.device)
    dist.all_gather_into_tensor(_bytes(out).view(-1), _bytes(shard16_padded).view(-1), group=group)
    return out


def gathered_rows(gathered, part: Partition) -> list:
    """Views of the N shards inside the all-gathered rows."""
    return [gathered[k, :part.lengths[k]] for k in range(part.world)]


def shard_step(hp: dict, part: Partition, full_grad16, master, m, v, shard16_padded, flat, *, rows=None,
               gathered=None, post_scale: float = 1.0, group=None, **step_options) -> None:
    """One training-state update of this rank's shard across real ranks (CUDA tensors):
    exchange the gradients, run the fused rank-ordered reduce + AdamW + 16-bit cast on the
    shard (ss_adam_step; master, m, v are this rank's part.n-element fp32 state), all-gather
    the 16-bit shards and place them into the flat unit (ss_unshard). `rows` and `gathered`
    may be preallocated exchange buffers; extra keyword arguments go to ss_adam_step."""
    rows = exchange_grads(full_grad16, part, out=rows, group=group)
    ss_adam_step(hp, part.n, master, m, v, rank_grads=[rows[r] for r in range(part.world)],
                 post_scale=post_scale, param16=shard16_padded[:part.n], **step_options)
    gathered = gather_params(shard16_padded, part, out=gathered, group=group)
    ss_unshard(gathered_rows(gathered, part), part.bounds, flat)
