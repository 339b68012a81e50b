"""Data-parallel training step over token shards (POET-X summary page, "Practice notes":
distributed data parallelism).

Every rank holds the whole merged frozen weight and the whole parameter set (the packed
triangles q of every block), runs the layer forward and backward on its own tokens, and then
takes part in one exchange: a sum all-reduce of the parameter gradients dq.  The gradients of
all layers live in one flat fp32 buffer, so the exchange is a single collective; after it
every rank applies the same optimizer update to the same parameters.  Nothing else crosses
ranks (dx stays local; the CNP is recomputed per rank from the shared q).

The per-rank compute and the update are passed in as callables, so the same step runs the
CUDA library on GPU ranks (NCCL) and the fp64 oracle on CPU ranks (gloo) in the tests.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Optional, Sequence, Tuple

import torch
import torch.distributed as dist


class FlatBuffer:
    """One contiguous fp32 tensor cut into named views of given shapes (the dq, q or optimizer
    state of every layer side), each view starting on a 16-byte boundary."""

    def __init__(self, shapes: Sequence[Tuple[str, Tuple[int, ...]]], device, fill: float = 0.0):
        self.offsets: Dict[str, Tuple[int, Tuple[int, ...]]] = {}
        o = 0
        for name, shape in shapes:
            numel = 1
            for d in shape:
                numel *= d
            self.offsets[name] = (o, tuple(shape))
            o += -(-numel // 4) * 4  # 4 floats = 16 bytes
        self.flat = torch.full((max(o, 4),), fill, dtype=torch.float32, device=device)

    def view(self, name: str) -> torch.Tensor:
        o, shape = self.offsets[name]
        numel = 1
        for d in shape:
            numel *= d
        return self.flat[o:o + numel].view(shape)

    def names(self) -> List[str]:
        return list(self.offsets)


def world_size(group=None) -> int:
    if dist.is_available() and dist.is_initialized():
        return dist.get_world_size(group)
    return 1


def exchange(grads_flat: torch.Tensor, group=None) -> None:
    """The data-parallel exchange: grads_flat <- sum over ranks of grads_flat, in place (one
    collective).  A no-op on a single rank."""
    if world_size(group) > 1:
        dist.all_reduce(grads_flat, op=dist.ReduceOp.SUM, group=group)


def data_parallel_step(compute: Callable[[], None], grads_flat: torch.Tensor,
                       update: Optional[Callable[[], None]] = None, group=None) -> None:
    """One training step: this rank's forward + backward (``compute``, which writes its
    gradients into ``grads_flat``), the sum all-reduce of the gradients over ranks, then the
    optimizer update (``update``), identical on every rank."""
    compute()
    exchange(grads_flat, group)
    if update is not None:
        update()
