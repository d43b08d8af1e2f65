"""Expert parallelism around the sharded forward of the C ABI.

The deployment on the pages is TP4/EP4: each rank holds a contiguous slice
of the experts (the local_expert_offset / local_num_experts arguments of
trtllm_bf16_routed_moe_lora, sglang PR #28953 summary page), routes every
token over all experts, computes only the slots routed to its own experts
(the others carry permuted index -1 and are skipped), and the layer output
is the sum of the ranks' partial outputs, completed by an all-reduce after
the MoE block (Flow 1(A) of "[WIP][LoRA] BF16 support for the
experimental_sgl_trtllm MoE-LoRA path & lora expert_outer_shared",
"downstream all_reduce (in qwen3_moe)").

Here a shard is a ``MoeLoraLayer`` built from its slice of the weights with
``local_expert_offset`` and ``num_router_experts``; ``all_reduce_partial``
sums the partial outputs over a ``torch.distributed`` process group (NCCL on
GPUs, gloo on CPUs).  The sum runs in float32 and is rounded to bf16 once.
"""
from __future__ import annotations

from typing import Tuple


def expert_shard(num_experts: int, world_size: int, rank: int) -> Tuple[int, int]:
    """(offset, count) of rank ``rank``'s experts: contiguous slices that cover
    [0, num_experts) once, sizes differing by at most one (the first
    num_experts % world_size ranks hold one more).  Every rank needs at least
    one expert."""
    if world_size < 1 or not 0 <= rank < world_size:
        raise ValueError("rank must be in [0, world_size)")
    if num_experts < world_size:
        raise ValueError("every rank needs at least one expert")
    base, extra = divmod(num_experts, world_size)
    count = base + (1 if rank < extra else 0)
    offset = rank * base + min(rank, extra)
    return offset, count


def all_reduce_partial(out, group=None):
    """Sum the ranks' partial outputs in place.

    bf16 / fp16 partials are summed in float32 and rounded once; wider types
    are summed in their own precision.  Returns ``out``.
    """
    import torch
    import torch.distributed as dist

    if out.dtype in (torch.bfloat16, torch.float16):
        acc = out.float()
        dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
        out.copy_(acc.to(out.dtype))
    else:
        dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    return out
