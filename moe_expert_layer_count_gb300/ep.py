"""Expert-parallel combine across ranks (one process per GPU).

Each rank runs the layer with its expert_map (its subset of the experts) and gets its
share of the output; the full output is the sum of the shares. `gather_partials` moves
the shares between ranks with torch.distributed (an all-gather, any backend); the sum
itself is the library's `moe_ep_combine` kernel. vLLM PR #20903 "[Kernel] DeepGemm MoE :
Integrate triton permute / unpermute kernels" (Purpose: DeepEP high-throughput
prepare/finalize with expert parallelism) runs the layer this way.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import moe_ep_combine


def gather_partials(partial: torch.Tensor, group=None):
    """The shares of all ranks of `group`, in rank order (bf16 [M, K] each). Moved as raw
    bytes, which every backend carries."""
    world = dist.get_world_size(group)
    raw = partial.contiguous().view(torch.uint8)
    parts = [torch.empty_like(raw) for _ in range(world)]
    dist.all_gather(parts, raw, group=group)
    return [p.view(torch.bfloat16) for p in parts]


def ep_combine(partial: torch.Tensor, group=None, out=None):
    """The layer output on every rank: all-gather of the shares, then their sum in rank
    order on this rank's GPU (moe_ep_combine)."""
    return moe_ep_combine(gather_partials(partial, group), out=out)
