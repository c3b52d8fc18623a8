"""World-size-2 and -4 gloo checks of the MXFP8 low-precision all-gather of
dim-0 weight shards ("MindSpeed LLM FSDP2量化特性", "为什么需要 FSDP2 量化训练"
and "注意事项" 1).

On CPU the shard quantizer is the oracle (passed in by the test); the
gathered codes and scales must equal the oracle's quantization of the whole
weight, because no block of 32 along dim 1 straddles two dim-0 shards.
"""

import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import mx_oracle as O
from precision_mx_quantize_gb300 import fsdp_gather


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_quantize(x, axis, fmt):
    c, s = O.mx_quantize(x.float().numpy(), axis, fmt)
    return torch.from_numpy(np.ascontiguousarray(c)), torch.from_numpy(np.ascontiguousarray(s))


def _weight(out_f, in_f):
    g = torch.Generator().manual_seed(11)
    return (torch.randn(out_f, in_f, generator=g) * 0.02).to(torch.bfloat16)


def _worker(rank, world, port, fmt, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        w = _weight(256, 96)
        lo, hi = fsdp_gather.shard_bounds(w.shape[0], world, rank)
        codes, scales = fsdp_gather.gather_mx_weight(w[lo:hi].contiguous(), fmt=fmt,
                                                     quantize=_oracle_quantize)
        out[rank] = (codes.numpy().tobytes(), scales.numpy().tobytes(), tuple(codes.shape))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_gathered_codes_equal_whole_weight_quantization(world, fmt):
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), fmt, out), nprocs=world, join=True)
    ec, es = O.mx_quantize(_weight(256, 96).float().numpy(), "row", fmt)
    for r in range(world):
        cb, sb, shape = out[r]
        assert shape == ec.shape
        assert cb == np.ascontiguousarray(ec).tobytes()
        assert sb == np.ascontiguousarray(es).tobytes()


def test_shard_bounds_and_traffic():
    assert fsdp_gather.shard_bounds(4096, 4, 0) == (0, 1024)
    assert fsdp_gather.shard_bounds(4096, 4, 3) == (3072, 4096)
    with pytest.raises(ValueError):
        fsdp_gather.shard_bounds(4097, 4, 0)
    with pytest.raises(ValueError):
        fsdp_gather.shard_bounds(4096, 4, 4)
    # MXFP8 moves 1 + 1/32 bytes per weight element against bf16's 2
    n = fsdp_gather.gathered_bytes(14336, 4096, "e4m3")
    assert n == 14336 * 4096 * 33 // 32
    assert n / (2 * 14336 * 4096) == pytest.approx(0.515625)
