"""Host-side logic of bench.py: the per-workload arithmetic and the multi-rank
timing reduction (world size 2 over gloo on the CPU)."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from gemma_dual_geometry_gb300 import workloads as W


def test_visible_pairs_closed_forms():
    # full causal attention over T tokens sees T(T+1)/2 pairs per head
    assert bench.visible_pairs(2048, 0, False) == 2048 * 2049 // 2 == 2_098_176
    assert bench.visible_pairs(4096, 0, False) == 8_390_656
    # sliding, window W: W(W+1)/2 for the first W queries, then W each
    assert bench.visible_pairs(2048, 512, True) == 512 * 513 // 2 + (2048 - 512) * 512 == 917_760
    assert bench.visible_pairs(4096, 512, True) == 1_966_336
    assert bench.visible_pairs(10, 1, True) == 10


def test_stack_workload_arithmetic():
    cfg = W.CONFIGS["stack42_bf16"]
    full = [l for l in range(42) if cfg["types"][l] == W.FULL]
    assert full == [5, 11, 17, 23, 29, 35, 41]
    # 4 * hd * H * B * pairs
    assert bench.prefill_flops(cfg, 5) == pytest.approx(1.0997e12, rel=1e-4)
    assert bench.prefill_flops(cfg, 0) == pytest.approx(0.12886e12, rel=1e-4)
    total = sum(bench.prefill_flops(cfg, l) for l in range(42))
    assert total == pytest.approx(12.21e12, rel=1e-3)
    # decode: about 1.248 GB of K/V per step across the 42 layers at the mean length
    step = sum(bench.decode_bytes(cfg, l, 4096 + 64) for l in range(42))
    assert step == pytest.approx(1.248e9, rel=5e-3)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w = bench.dist_init("gloo")
    bench.barrier()
    # each rank reports its own time; the job's time is the slowest rank's
    mx = bench.reduce_max(1.5 + rank)
    sm = bench.reduce_sum(100.0 * (rank + 1))
    out[rank] = (r, w, mx, sm)
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == (0, 2, 2.5, 300.0)
    assert out[1] == (1, 2, 2.5, 300.0)


def test_single_process_reduce_is_identity():
    assert bench.reduce_max(3.25) == 3.25
    assert bench.dist_env()[1] in (1, int(os.environ.get("WORLD_SIZE", "1")))
