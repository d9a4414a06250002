"""Host-side logic of bench.py on the CPU: the multi-rank timing reduction
(two gloo ranks, as torchrun starts them), the replica rank layout, and the
launch count of one step."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    # CPU ranks over gloo, as on a machine without GPUs, whatever this one has
    # (set before anything in the fresh process touches CUDA)
    os.environ["CUDA_VISIBLE_DEVICES"] = ""
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    w, r, local = bench.dist_setup()
    try:
        assert (w, r, local) == (world, rank, rank)
        bench.barrier(w)
        # every rank reports its own step time; all must see the slowest
        out[rank] = bench.max_over_ranks(1.5 + rank, w)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)


def test_launches_per_step():
    assert bench.launches_per_step(1, 1) == 4
    assert bench.launches_per_step(1, 4) == 6
    assert bench.launches_per_step(3, 2) == 8


def test_flop_counts_are_per_cell_and_peak_is_fp32():
    assert bench.FLOPS_PER_CELL["fwd"] < bench.FLOPS_PER_CELL["bwd"]
    assert bench.FP32_PEAK_TFLOPS == pytest.approx(152 * 128 * 2 * 2.07e9 / 1e12)
