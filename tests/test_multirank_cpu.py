"""World-size-2 gloo checks of the multi-rank host logic of bench.py.

The MX path has no exchange step, so N GPUs run N replicas; the only
cross-rank work is the barrier and the max-over-ranks timing reduction that
turn per-rank times into the whole-job number.
"""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import argparse

    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        dist.barrier()
        ms = bench.reduce_max_ms(10.0 + 5.0 * rank)
        val = bench.aggregate_tflops(world, 1e12, 4, ms)
        args = argparse.Namespace(steps=1, warmup=0, tokens=8192)
        ref = bench.reference_arm(args, rank, world) if rank != 0 else "rank0"
        out[rank] = (ms, val, ref)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_and_aggregate():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, val, ref = out[r]
        assert ms == 15.0                      # the slowest rank's time, on every rank
        assert abs(val - 2 * 1e12 * 4 / 15e-3 / 1e12) < 1e-9
    assert out[1][2] is None                   # only rank 0 runs the reference arm


def test_step_work_counts():
    import bench
    plan = bench.layer_plan(8192)
    q, f8, f4 = bench.step_work(plan)
    macs = sum(L["T"] * L["fin"] * L["fout"] for L in plan)
    assert f8 == 4 * macs and f4 == 2 * macs
    assert bench.quant_bytes(32, 64, "e4m3", "e2m1") == 2 * 2048 + 2048 + 64 + 1024 + 64


@pytest.mark.timeout(300)
def test_reference_arm_line_matches_the_contract():
    # the oracle arm: rank 0 only, the main arm's metric, unit and config,
    # and the keys the reference line carries (impl, cpu_baseline, e2e with
    # no host-device bytes)
    import argparse

    import bench
    args = argparse.Namespace(steps=1, warmup=0, tokens=8192)
    assert bench.reference_arm(args, 1, 2) is None
    line = bench.reference_arm(args, 0, 1)
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
    assert line["higher_is_better"] is True
    assert line["config"] == bench.run_config(bench.layer_plan(8192), 8192, 1)
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_peak_basis_follows_the_clock_samples():
    # burst bf16 figure when the run held its maximum clock with no power
    # cap; the sustained figure otherwise
    import bench
    peaks = {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6700.0}
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.peak_basis(full, peaks) == ("burst", 1900.0)
    capped = dict(full, reasons=["sw_power_cap"])
    assert bench.peak_basis(capped, peaks) == ("sustained", 1700.0)
    slow = dict(full, sm_mhz=1700.0)
    assert bench.peak_basis(slow, peaks) == ("sustained", 1700.0)
    none = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
    assert bench.peak_basis(none, peaks) == ("sustained", 1700.0)
