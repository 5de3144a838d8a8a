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


def test_bidirectional_pairs_closed_forms():
    # every key on a global layer; on a sliding one 2W+1 keys per query less
    # W(W+1)/2 cut off at each end of the sequence (T >= W)
    assert bench.visible_pairs_bidirectional(2048, 0, False) == 2048 * 2048
    for T, Wn in ((2048, 512), (1000, 100), (300, 1), (7, 7)):
        assert bench.visible_pairs_bidirectional(T, Wn, True) == T * (2 * Wn + 1) - Wn * (Wn + 1)
    assert bench.visible_pairs_bidirectional(10, 0, True) == 10
    cfg = W.CONFIGS["encoder_bf16"]
    assert bench.prefill_flops(cfg, 0) == 4.0 * 256 * 8 * 4 * (2048 * 1025 - 512 * 513)
    assert bench.prefill_flops(cfg, 1) == 4.0 * 512 * 8 * 4 * 2048 * 2048


def test_ring_workload_builds_ring_caches_on_the_host():
    # the stack driver's tables, built on CPU tensors (no kernel runs): the
    # sliding layer's cache is a 512-row ring, the full layer's a linear cache
    from gemma_dual_geometry_gb300 import build as g4build
    from gemma_dual_geometry_gb300.stack import AttnStack
    g4build.build()
    cfg = dict(W.CONFIGS["ring_decode_bf16"], B=2)
    st = AttnStack(cfg, 8192, device="cpu")
    assert (st.table[0].ring, st.table[0].max_len) == (1, 512)
    assert (st.table[1].ring, st.table[1].max_len) == (0, 8192)
    assert st.caches[0][0].shape == (2, 2, 512, 256)
    assert st.caches[1][0].shape == (2, 2, 8192, 512)
    plain = AttnStack(dict(W.CONFIGS["decode_bf16"], B=2), 8192, device="cpu")
    assert (plain.table[0].ring, plain.table[0].max_len) == (0, 8192)
    # the decode bytes of a ring step are those of the linear cache
    assert all(bench.decode_bytes(cfg, l, L) == bench.decode_bytes(dict(W.CONFIGS["decode_bf16"], B=2), l, L)
               for l in (0, 1) for L in (1, 600, 8000))


def test_profiled_traffic_only_for_the_captured_kernel_source(monkeypatch):
    # a figure is reported while the kernel's sources hash to the digest taken
    # at the capture, and withheld (None) once they differ
    files = bench.WIN_SOURCES
    now = bench.kernel_sources_hash(files)
    monkeypatch.setitem(bench.PROFILED_TRAFFIC, "decode_sliding", (123, files, now, "capture"))
    assert bench.profiled_traffic("decode_sliding") == (123, "capture")
    monkeypatch.setitem(bench.PROFILED_TRAFFIC, "decode_sliding", (123, files, "0" * 16, "capture"))
    t, src = bench.profiled_traffic("decode_sliding")
    assert t is None and "changed" in src
    assert bench.profiled_traffic("no_such_kernel")[0] is None


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


def test_oracle_baseline_pool_runs_on_several_cores():
    # the CPU baseline's sample on a process pool (spawn), on the tiny stack:
    # every layer's append and (layer, query group) attention tasks run, and
    # the line reports the workers it used
    res = bench.oracle_worker(dict(workload="tiny_fp32_stack", steps=1, warmup=0, n_query=8, append_chunk=16,
                                   query_group=4, max_cores=2))
    assert res["cores"] == min(2, len(os.sched_getaffinity(0)))
    (step,) = res["steps"]
    assert step["t_append"] > 0 and step["t_attn"] > 0 and step["cpu_s"] > 0
    assert step["per_token_s"] == pytest.approx(step["t_append"] / 16 + step["t_attn"] / 8)


def test_projection_workload_arithmetic():
    # 2 M N K per launch: q/k/v rows (H + 2 Hkv) hd, o_proj K = H hd, D = 2048
    for name, per in (("qkv_proj_bf16", lambda hd: 2.0 * 32768 * 12 * hd * 2048),
                      ("out_proj_bf16", lambda hd: 2.0 * 32768 * 2048 * 8 * hd)):
        cfg = W.CONFIGS[name]
        job = bench.ProjJob.__new__(bench.ProjJob)
        job.cfg, job.M, job.D, job.kind = cfg, cfg["B"] * cfg["T"], cfg["D"], cfg["proj"]
        job.geo = [W.layer_geometry(cfg, l) for l in range(2)]
        assert [job.layer_work(l) for l in range(2)] == [per(256), per(512)]
