"""The MXFP8 all-gather of dim-0 weight shards on one GPU (a world of one
rank over NCCL): the gathered operand equals the oracle's (and the CUDA
quantizer's) quantization of the whole weight and, fed to the forward GEMM,
matches the oracle."""

import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

from oracle import mx_oracle as O
from precision_mx_quantize_gb300 import fsdp_gather, mxq, synth
from tests.libutil import bf16_to_f32_np, ensure_built, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def group():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    yield None
    dist.destroy_process_group()


def test_gather_then_forward_gemm(group):
    w = synth.weight(6144, 4096, seed=1).cuda()
    x = synth.activation(1024, 4096, seed=2).cuda()
    lo, hi = fsdp_gather.shard_bounds(w.shape[0], 1, 0)
    codes, scales = fsdp_gather.gather_mx_weight(w[lo:hi].contiguous())
    torch.cuda.synchronize()
    wc, ws = mxq.mx_quantize(w, "row", "e4m3")
    mxq.check()
    assert torch.equal(codes, wc) and torch.equal(scales, ws)
    # the gathered operand is the oracle's quantization of the whole weight
    oc, os_ = O.mx_quantize(bf16_to_f32_np(w), "row", "e4m3")
    np.testing.assert_array_equal(to_np(codes), oc)
    np.testing.assert_array_equal(to_np(scales), os_)
    xc, xs = mxq.mx_quantize(x, "row", "e4m3")
    y = mxq.mx_gemm(xc, xs, codes, scales, "e4m3", 1024, 6144, 4096)
    mxq.check()
    rng = np.random.default_rng(3)
    rows = rng.choice(1024, 32, replace=False)
    cols = rng.choice(6144, 64, replace=False)
    oA, osA = O.mx_quantize(bf16_to_f32_np(x)[rows], "row", "e4m3")
    oB, osB = O.mx_quantize(bf16_to_f32_np(w)[cols], "row", "e4m3")
    ref, S = O.mx_gemm_f64(oA, osA, oB, osB, "e4m3")
    got = to_np(y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()]).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2e-4 * S)
