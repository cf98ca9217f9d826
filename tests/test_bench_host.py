"""Host-side logic of bench.py on the CPU: the replica aggregation over ranks
(two gloo processes) and the reference arm's JSON line."""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from tests.conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_replica_value():
    # 2 replicas x 1 GB per step x 10 steps in 4 s (the slowest rank)
    assert bench.replica_value(2, 10 ** 9, 10, 4.0) == pytest.approx(5.0)
    assert bench.replica_value(1, 2 * 10 ** 9, 1, 1.0) == pytest.approx(2.0)


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = [1.5, 2.5][rank]
    t_max = bench.max_over_ranks(t)
    q.put((rank, t_max, bench.replica_value(world, 100, 4, t_max)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_processes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]
    assert res[0][2] == pytest.approx(2 * 100 * 4 / 2.5 / 1e9)


def test_reference_arm_line_and_other_ranks():
    env = dict(os.environ)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny", "--steps", "3", "--warmup", "1"]
    out = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 3 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    # a non-zero rank of a torchrun launch prints nothing and exits 0
    env.update(RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_phase1_kernel_choice_and_profile_parsing():
    from gradient_aggregation_gb300 import workload
    # aligned, and long enough that the shifted variant is the faster one
    assert bench.phase1_kernel(workload.get("alexnet")) == "k_reduce_tma, shifted layout"
    assert bench.phase1_kernel(workload.get("tiny")) == "k_reduce_tma"
    assert bench.phase1_kernel(workload.get("stress")) == "k_reduce"      # 64 workers
    # layers at odd offsets, one address shift per layer for all workers
    assert bench.phase1_kernel(workload.get("googlenet")) == "k_reduce_tma, shifted layout"
    wl = workload.get("alexnet")
    # the committed summary is used only for the kernel source it was taken on
    assert bench.traffic_from_profile("not-the-current-source", wl) is None
    t = bench.traffic_from_profile(bench.kernel_source_hash(), wl)
    assert t is None or 2.0e9 < t < 3.0e9


def test_layer_groups_reverse_tile_the_layers_last_first(fc_lib):
    from gradient_aggregation_gb300 import fc, workload
    for name in ("tiny", "nin", "googlenet", "alexnet", "stress"):
        wl = workload.get(name)
        g = bench.layer_groups_reverse(wl.sizes, 4)
        assert g[0][1] == wl.L and g[-1][0] == 0
        assert all(a < b for a, b in g) and all(g[i][0] == g[i + 1][1] for i in range(len(g) - 1))
        assert 1 <= len(g) <= 4
        assert fc.layer_group_spans(wl.sizes, wl.chunk, g) == [
            (sum(wl.sizes[:a]), sum(wl.sizes[:b])) for a, b in g]
    # AlexNet: fc8+fc7, fc6, the convolutions (fc6 alone passes two marks)
    assert bench.layer_groups_reverse(workload.get("alexnet").sizes, 4) == [(12, 16), (10, 12), (0, 10)]


def test_group_major_layout_places_each_group_in_one_block():
    sizes, W = [5, 3, 7, 2], 3
    groups = [(2, 4), (0, 2)]
    span, pos = bench.group_major_layout(sizes, W, groups)
    assert span == [(0, 27), (27, 51)]
    buf = [None] * 51
    for w in range(W):
        for l, n in enumerate(sizes):
            for j in range(n):
                assert buf[pos[w][l] + j] is None
                buf[pos[w][l] + j] = (w, l, j)
    assert None not in buf
    for (a, b), (lo, hi) in zip(groups, span):      # a group's block holds its layers only
        assert {buf[i][1] for i in range(lo, hi)} == set(range(a, b))


def test_cpu_baseline_takes_the_median_of_several_oracle_steps():
    import numpy as np
    import oracle
    from gradient_aggregation_gb300 import workload
    wl = workload.get("tiny")
    line, (ws, g, first, out) = bench.cpu_baseline(wl, 0.3)
    assert line["kind"] == "oracle" and line["cores"] == 1 and line["value"] > 0
    assert "median of" in line["sample"] and line["host"]["cpus"] >= 1
    # the parity material is the state after exactly one step
    st = oracle.State(workload.initial_weights(ws))
    ref = oracle.step(g, st, ws.loss_scale, ws.chunk, ws.keep_percent, 100, ws.lr, ws.momentum)
    assert np.array_equal(ref["idx"], out["idx"])
    assert np.array_equal(st.weights.view(np.uint32), first.weights.view(np.uint32))


def test_phase1_is_timed_at_least_twenty_times_at_any_step_count():
    for steps in (20, 21, 50, 159, 160, 161, 2000, 50000):
        every = bench.phase1_every(steps)
        assert 1 <= every <= 8
        assert len(range(0, steps, every)) >= bench.MIN_PHASE1
    assert bench.phase1_every(2000) == 8 and bench.phase1_every(20) == 1


def test_algorithmic_bytes_per_kernel():
    """Phase 1 reads the gradients and the residual and writes `a` and one
    fp32 sum of squares per 256-element unit; the plain count is N(2W+32)."""
    from gradient_aggregation_gb300 import workload
    wl = workload.get("alexnet")
    W, N = wl.W, wl.N
    units = bench.units_of(N, wl.chunk)
    # 1904 chunks of 128 units, the last of 20840 elements: 82 units
    assert units == 1903 * 128 + 82
    b = bench.step_algorithmic_bytes(wl, 20)
    assert b["phase1"] == 2 * W * N + 8 * N + 4 * units == 2_496_108_424
    assert b["phase3"] == 16 * N + 8 * 20 * 32768 + 4 * 20 * 32768
    assert b["full_count"] == N * (2 * W + 32)
    assert b["step"] == b["phase1"] + b["phase2"] + b["phase3"]
    # keep-all: every element's a read, residual zeroed, send slots for all chunks
    nin = workload.get("nin")
    C = -(-nin.N // nin.chunk)
    assert bench.step_algorithmic_bytes(nin, C)["phase3"] == 16 * nin.N + 8 * nin.N + 4 * C * nin.chunk
