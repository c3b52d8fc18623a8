"""MXFP8 low-precision all-gather of dim-0 weight shards.

"MindSpeed LLM FSDP2量化特性：低比特大模型训练完全指南":

* "为什么需要 FSDP2 量化训练": FSDP2 keeps each weight split across the ranks
  and all-gathers the full weight before every layer's forward and backward
  computation.  Gathering MXFP8 (one-byte E4M3 codes plus one E8M0 scale per
  32 elements) instead of bf16 halves both the traffic and the memory of the
  gathered weight.
* "注意事项" 1: the shards split dim 0 (``shard_by_dim_0``).  Blocks of 32
  run along dim 1, so no block ever straddles two ranks and each rank can
  quantize its own rows.

Here a weight W [out, in] (PyTorch Linear layout) is split into equal
contiguous row ranges.  Each rank quantizes its rows row-wise (blocks along
the input features) with the CUDA quantizer, then codes and scales are
all-gathered.  The result is the forward GEMM's B operand (Y = X W^T) for
the whole weight, identical to quantizing the full W in one call.

Collectives go through ``torch.distributed`` (NCCL on GPUs).  The host logic
is also exercised with the gloo backend on CPU, where a test passes its own
shard quantizer.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import mxq


def shard_bounds(rows: int, world: int, rank: int) -> tuple[int, int]:
    """Row range [start, end) of `rank` when `rows` are split into `world` equal shards."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if rows % world != 0:
        raise ValueError(f"{rows} rows do not split evenly over {world} ranks")
    n = rows // world
    return rank * n, (rank + 1) * n


def gathered_bytes(out_features: int, in_features: int, fmt: str = "e4m3") -> int:
    """Bytes the all-gather moves into each rank: codes plus scales of the full weight."""
    code_bytes = out_features * in_features // (2 if mxq.FMTS[fmt] == mxq.E2M1 else 1)
    return code_bytes + out_features * in_features // 32


def gather_mx_weight(w_shard: torch.Tensor, group=None, fmt: str = "e4m3", quantize=None,
                     out=None):
    """All-gather the MX codes of this rank's dim-0 shard of a weight.

    w_shard: [out / world, in] bf16, this rank's rows (in % 32 == 0).
    quantize(x, axis, fmt) -> (codes, scales): the shard quantizer; the CUDA
    library's ``mxq.mx_quantize`` unless a test passes another.
    out: optional (codes [out][in or in/2], scales [out][in/32]) to fill.
    Returns (codes, scales) of the full weight, in rank order.
    """
    quantize = quantize or mxq.mx_quantize
    world = dist.get_world_size(group)
    codes_s, scales_s = quantize(w_shard, "row", fmt)
    rows = w_shard.shape[0] * world
    if out is None:
        out = (torch.empty((rows,) + tuple(codes_s.shape[1:]), dtype=torch.uint8,
                           device=codes_s.device),
               torch.empty((rows,) + tuple(scales_s.shape[1:]), dtype=torch.uint8,
                           device=scales_s.device))
    codes, scales = out
    dist.all_gather_into_tensor(codes, codes_s.contiguous(), group=group)
    dist.all_gather_into_tensor(scales, scales_s.contiguous(), group=group)
    return codes, scales
