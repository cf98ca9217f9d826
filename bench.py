"""Benchmark of the gradient-aggregation engine on GB300.

One step = the whole hot path over one batch of synthetic gradients: the
workers' per-layer fp16 gradients are fused (through the layout, without a
copy), tree-reduced in fp32 with the loss-scale/W unscale and the residual,
scored by chunk L2 norm, the top chunks selected and compacted, and the
residual/momentum-SGD update applied (three kernels: fc_step).

Metric: worker-gradient GB/s = W * N * 2 bytes per step / time per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload alexnet]
                  [--impl reference]

With torchrun (N > 1) every rank runs an independent replica of the same
workload on its own GPU (the method has no cross-GPU exchange here): the
value is all ranks' bytes over the slowest rank's time.

`--impl reference` times the CPU oracle (single-threaded C, the plain
statement of the method) on a bounded sample of the same workload per step.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gradient_aggregation_gb300 import workload  # noqa: E402

METRIC = "worker-gradient GB/s aggregated (1xGB300) and % of HBM roofline vs CPU oracle"
UNIT = "GB/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default="alexnet", choices=sorted(workload.WORKLOADS))
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--elements", type=int, default=0,
                   help="use only the first ELEMENTS fused elements of the workload "
                        "(small cases for profiling)")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--phase1-every", type=int, default=0,
                   help="bracket phase 1 with events on every n-th timed step "
                        "(default: one in eight, more often on short runs)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def config_of(wl, extra=None):
    C = -(-wl.N // wl.chunk)
    cfg = {"workload": "%s-shaped: W=%d workers, N=%d fp16 elements in %d layer tensors, "
                       "chunk %d, keep %d%%" % (wl.name, wl.W, wl.N, wl.L, wl.chunk,
                                                wl.keep_percent),
           "W": wl.W, "N": wl.N, "layers": wl.L, "chunk": wl.chunk, "chunks": C,
           "keep_percent": wl.keep_percent, "loss_scale": wl.loss_scale,
           "lr": wl.lr, "momentum": wl.momentum}
    if extra:
        cfg.update(extra)
    return cfg


# ---- CPU oracle samples ---------------------------------------------------------

def sample_workload(wl, m):
    """The first m fused elements of wl: layers cut at m."""
    sizes, acc = [], 0
    for s in wl.sizes:
        if acc >= m:
            break
        take = min(s, m - acc)
        sizes.append(take)
        acc += take
    return workload.custom(W=wl.W, sizes=sizes, chunk=wl.chunk,
                           keep_percent=wl.keep_percent, loss_scale=wl.loss_scale,
                           grad_std=wl.grad_std, momentum=wl.momentum, lr=wl.lr,
                           config_id=wl.config_id, heavy_tail=wl.heavy_tail)


def oracle_step_time(wl_s, grads, state):
    import oracle
    t0 = time.perf_counter()
    oracle.step(grads, state, wl_s.loss_scale, wl_s.chunk, wl_s.keep_percent, 100,
                wl_s.lr, wl_s.momentum)
    return time.perf_counter() - t0


def oracle_elems_for(wl, seconds):
    """Calibrate how many fused elements the oracle handles in `seconds`."""
    import oracle
    m = min(wl.N, 1 << 18)
    ws = sample_workload(wl, m)
    g = workload.all_grads(ws, 0)
    st = oracle.State(workload.initial_weights(ws))
    oracle_step_time(ws, g, st)                    # warm (page faults, table)
    t = min(oracle_step_time(ws, g, st) for _ in range(2))
    return max(1024, min(wl.N, int(m * seconds / max(t, 1e-6))))


def host_description():
    """The machine the CPU baseline ran on: architecture, CPU count and,
    where the system reports one, the CPU model."""
    import platform
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"machine": platform.machine(), "cpus": os.cpu_count(), "model": model}


def cpu_baseline(wl, seconds):
    """Times the oracle on a sample of the workload sized so that one step
    takes about a third of `seconds`: steps (state carried) until `seconds`
    have passed, at least three; the median step counts.  Also returns what
    the parity check needs: the sample, its gradients, and the oracle's
    state and outputs after the first step."""
    import oracle
    m = oracle_elems_for(wl, seconds / 3.0)
    ws = sample_workload(wl, m)
    g = workload.all_grads(ws, 0)
    st = oracle.State(workload.initial_weights(ws))
    args = (ws.loss_scale, ws.chunk, ws.keep_percent, 100, ws.lr, ws.momentum)
    t0 = time.perf_counter()
    out = oracle.step(g, st, *args)
    times = [time.perf_counter() - t0]
    first = st.copy()
    while len(times) < 3 or sum(times) < seconds:
        t0 = time.perf_counter()
        oracle.step(g, st, *args)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    gbs = ws.W * ws.N * 2 / t / 1e9
    return ({"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
             "host": host_description(),
             "sample": "median of %d steps of the oracle (pack, tree reduce, norms, select, "
                       "update), %.1f s in all, on the first %d of %d fused elements of every "
                       "worker (%.1f%%)"
                       % (len(times), sum(times), ws.N, wl.N, 100.0 * ws.N / wl.N)},
            (ws, g, first, out))


def parity_check(ws, g, st, out, dev):
    """One fresh GPU step on the oracle's own inputs, compared with it: the
    kept indices exactly, residual, velocity and weights bit for bit, the
    threshold within the 1e-6 band."""
    import torch
    from gradient_aggregation_gb300 import fc
    eng = fc.Engine(ws.sizes, ws.W, ws.chunk, ws.keep_percent, 100, ws.loss_scale, ws.lr,
                    ws.momentum, torch.from_numpy(workload.initial_weights(ws)).to(dev))
    gd = [[torch.from_numpy(x).to(dev) for x in row] for row in g]
    eng.step(gd)
    torch.cuda.synchronize()

    def same(t, ref):
        return bool(np.array_equal(t.cpu().numpy().view(np.uint32), ref.view(np.uint32)))

    idx_same = bool(np.array_equal(eng.idx.cpu().numpy(), out["idx"]))
    thr, thr_ref = float(eng.threshold.cpu()[0]), float(out["threshold"])
    res = {"checked": "one step of the bench's sample (%d elements x %d workers) against "
                      "the oracle" % (ws.N, ws.W),
           "kept_indices_equal": idx_same,
           "residual_bits_equal": same(eng.residual, st.residual),
           "velocity_bits_equal": same(eng.velocity, st.velocity),
           "weights_bits_equal": same(eng.weights, st.weights),
           "threshold_rel_diff": abs(thr - thr_ref) / max(abs(thr_ref), 1e-30)}
    ok = idx_same and res["residual_bits_equal"] and res["velocity_bits_equal"] and \
        res["weights_bits_equal"] and res["threshold_rel_diff"] <= 1e-6
    res["verdict"] = "pass" if ok else "fail"
    del eng, gd
    torch.cuda.empty_cache()
    return res


def run_reference(args, wl, rank):
    if rank != 0:
        return 0
    import oracle
    budget = 90.0 / max(1, args.steps + args.warmup)
    m = oracle_elems_for(wl, budget)
    ws = sample_workload(wl, m)
    g = workload.all_grads(ws, 0)
    st = oracle.State(workload.initial_weights(ws))
    for _ in range(args.warmup):
        oracle_step_time(ws, g, st)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step_time(ws, g, st)
    dt = time.perf_counter() - t0
    value = ws.W * ws.N * 2 * args.steps / dt / 1e9
    sample = ("each step: the oracle (single-threaded C) on the first %d of %d fused "
              "elements of every worker" % (ws.N, wl.N))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded Gaussian fp16 gradients, workload-shaped)",
            "config": config_of(wl, {"sample_elements": ws.N}),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": sample,
                             "host": host_description()},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ---- clocks -------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid, out_path=None):
        self.uuid = uuid
        self.rows = []
        self.out_path = out_path
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        mine = [r for (t, r) in self.rows if len(r) >= 10 and (not self.uuid or r[1] == self.uuid)]
        during = [r for (t, r) in self.rows
                  if t0 <= t <= t1 + 0.15 and len(r) >= 10 and (not self.uuid or r[1] == self.uuid)]
        use = during if during else mine[-3:]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in use if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "in_timed_region": bool(during)}


# ---- GPU arm ---------------------------------------------------------------------------

def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("fc_reduce.cu", "fc_reduce_tma.cu", "fc_common.cuh"):
        with open(os.path.join(ROOT, "gradient_aggregation_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def phase1_kernel(wl, table=None) -> str:
    """The phase-1 kernel the library picks for this layout
    (fc_step_reduce_kernel).  Without a table of the gradients actually
    used, separately allocated 512-byte-aligned tensors are assumed."""
    from gradient_aggregation_gb300 import fc
    if table is None:
        table = fc.PtrTable.from_addresses(
            [[(1 + w * wl.L + l) << 20 for l in range(wl.L)] for w in range(wl.W)], wl.sizes)
    kind = fc.fc_step_reduce_kernel(table, wl.chunk)
    return {fc.FC_REDUCE_REGISTER: "k_reduce",
            fc.FC_REDUCE_STAGED: "k_reduce_tma",
            fc.FC_REDUCE_STAGED_SHIFTED: "k_reduce_tma, shifted layout"}[kind]


def layer_groups_reverse(sizes, n_groups):
    """Layer groups [first, end) in backprop order (last layer first), each
    closed once it holds about 1/n_groups of the elements."""
    total = sum(sizes)
    groups, end, acc, target = [], len(sizes), 0, 1
    for l in range(len(sizes) - 1, -1, -1):
        acc += sizes[l]
        if acc * n_groups >= total * target or l == 0:
            groups.append((l, end))
            end = l
            target = acc * n_groups // total + 1   # a large layer may pass several marks
    return groups


def group_major_layout(sizes, W, groups):
    """Buffer layout [group][worker][group's elements], groups in arrival
    order: the [begin, end) of each group in the buffer, and the position of
    every (worker, layer) tensor."""
    off = [0]
    for n in sizes:
        off.append(off[-1] + n)
    span, pos, acc = [], [[0] * len(sizes) for _ in range(W)], 0
    for a, b in groups:
        glen = off[b] - off[a]
        span.append((acc, acc + W * glen))
        for w in range(W):
            for l in range(a, b):
                pos[w][l] = acc + w * glen + off[l] - off[a]
        acc += W * glen
    return span, pos


def traffic_from_profile(src_hash, wl):
    """DRAM bytes per launch of the reduction kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "k_reduce_%s.md" % wl.name)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha") != src_hash:
        return None
    try:
        return float(vals["dram_bytes_per_full_launch"])
    except (KeyError, ValueError):
        return None


MIN_PHASE1 = 20   # phase-1 launches timed at least, at any --steps


def phase1_every(steps: int) -> int:
    """Time phase 1 on every n-th step: one in eight on long runs, more often
    on short ones so that at least MIN_PHASE1 launches are timed."""
    return max(1, min(8, steps // MIN_PHASE1))


def units_of(N: int, chunk: int) -> int:
    """256-element units of the fused vector (none straddles a chunk)."""
    C = -(-N // chunk)
    U = -(-chunk // 256)
    return (C - 1) * U + -(-(N - (C - 1) * chunk) // 256)


def step_algorithmic_bytes(wl, k: int) -> dict:
    """Algorithmic bytes of one pipeline step with `a` formed in place in the
    residual buffer, per kernel, and the plain count N*(2W+32):
      phase 1: the W workers' fp16 gradients, the residual read, `a`
               written, one fp32 sum of squares per 256-element unit;
      phase 2: the unit sums read; norms, mask, kept-slot map and idx
               written;
      phase 3: velocity and weights read and written for every element;
               for kept elements `a` read, the residual zeroed and the
               packed fp32 send buffer written.  In place, unkept elements'
               `a` is already their new residual: neither read nor written.
    The plain count also reads `a` and writes the residual for every
    element (8N more) and leaves out the unit sums and the selection."""
    W, N = wl.W, wl.N
    C = -(-N // wl.chunk)
    units = units_of(N, wl.chunk)
    kept_el = min(N, k * wl.chunk)       # at most; a kept short last chunk has fewer
    phase1 = 2 * W * N + 4 * N + 4 * N + 4 * units
    phase2 = 4 * units + 4 * C + C + 4 * C + 4 * k
    phase3 = 16 * N + 8 * kept_el + 4 * k * wl.chunk   # + the zero-padded send slots
    return {"phase1": phase1, "phase2": phase2, "phase3": phase3,
            "step": phase1 + phase2 + phase3, "full_count": N * (2 * W + 32)}


def max_over_ranks(x: float, device=None) -> float:
    """The largest of every rank's x (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(world: int, step_bytes: int, steps: int, t_max: float) -> float:
    """Whole-job worker-gradient GB/s: every replica processes step_bytes per
    step; the job takes as long as the slowest rank."""
    return world * step_bytes * steps / t_max / 1e9


def run_gpu(args, wl, rank, world, local):
    import torch
    from gradient_aggregation_gb300 import fc

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_t(x):
        return max_over_ranks(x, dev)

    fc.lib()
    W, N = wl.W, wl.N
    grads_np = workload.all_grads(wl, 0)
    # per-layer device tensors, as a training framework's autograd leaves them
    grads = [[torch.from_numpy(g).to(dev) for g in row] for row in grads_np]
    table = fc.PtrTable(grads)
    eng = fc.Engine(wl.sizes, W, wl.chunk, wl.keep_percent, 100, wl.loss_scale, wl.lr,
                    wl.momentum, torch.from_numpy(workload.initial_weights(wl)).to(dev))
    s = torch.cuda.Stream(device=dev)
    phases = list(eng.phases(table, s))
    # Small problems run fc_step as one launch: the timed step is then that
    # one kernel, and its events bracket the whole step.
    path = fc.fc_step_path(table, wl.chunk)
    one_launch = path in (fc.FC_STEP_ONE_LAUNCH, fc.FC_STEP_ONE_CLUSTER)
    one_kernel = ("k_step_grid: the whole fc_step in one cooperative launch, one CTA per SM"
                  if path == fc.FC_STEP_ONE_LAUNCH else
                  "k_step_small: the whole fc_step in one thread-block cluster launch")

    def step_phased(evs=None):
        if one_launch:
            if evs is not None:
                evs[0].record(s)
            eng.step(table, s)
            if evs is not None:
                evs[1].record(s)
            return
        if evs is not None:
            evs[0].record(s)
        phases[0]()
        if evs is not None:
            evs[1].record(s)
        phases[1]()
        phases[2]()

    K = args.steps
    # Phase-1 events bracket the reduction kernel on every EVERY-th step, so
    # that at least MIN_PHASE1 launches are timed at any step count: an event
    # between two kernels stops the next one from being scheduled early
    # (programmatic dependent launch), so long runs time one step in eight.
    EVERY = args.phase1_every if args.phase1_every > 0 else phase1_every(K)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           if i % EVERY == 0 else None for i in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.35)
    # warm-up directly before the timed steps: no idle gap in which the
    # clocks could drop
    torch.cuda.synchronize()
    barrier()
    warmup = max(3, args.warmup)   # at least three untimed steps
    for _ in range(warmup):
        step_phased()
    t_wall0 = time.time()
    start.record(s)
    for i in range(K):
        step_phased(evs[i])
    end.record(s)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    total_ms = start.elapsed_time(end)
    reduce_ms = [e[0].elapsed_time(e[1]) for e in evs if e is not None]
    t_max = max_t(total_ms / 1e3)
    step_bytes = W * N * 2
    value = replica_value(world, step_bytes, K, t_max)
    ms_per_step = t_max * 1e3 / K

    # roofline of the dominant kernel (phase 1: tree reduce + norm partials)
    C = -(-N // wl.chunk)
    alg = step_algorithmic_bytes(wl, eng.k)
    k_alg = alg["step"] if one_launch else alg["phase1"]
    k_ms = statistics.mean(reduce_ms)

    # the same phase-1 kernel launched back to back on its own (out of place,
    # so the engine's state is untouched), at least MIN_PHASE1 launches
    iso = None
    try:
        a_tmp = torch.empty(N, dtype=torch.float32, device=dev)
        def once():
            if one_launch:
                eng.step(table, s)
            else:
                fc.fc_step_reduce(table, wl.loss_scale, wl.chunk, eng.residual, a_tmp,
                                  eng.workspace, s)
        for _ in range(3):
            once()
        i0, i1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        KI = max(MIN_PHASE1, min(K, 200))
        i0.record(s)
        for _ in range(KI):
            once()
        i1.record(s)
        torch.cuda.synchronize()
        iso_ms = i0.elapsed_time(i1) / KI
        del a_tmp
        iso = {"avg_launch_ms": round(iso_ms, 5), "launches": KI}
    except Exception as exc:
        iso = {"unavailable": str(exc).splitlines()[0][:120] if str(exc) else type(exc).__name__}
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    achieved = k_alg / (k_ms / 1e3) / 1e9
    src_hash = kernel_source_hash()
    traffic = traffic_from_profile(src_hash, wl)

    # the rest of the step: select + update, measured as step minus phase 1
    rest_ms = ms_per_step - k_ms
    step_alg = alg["step"]
    if iso and "avg_launch_ms" in iso:
        iso["achieved"] = round(k_alg / (iso["avg_launch_ms"] / 1e3) / 1e9, 1)
        iso["frac"] = round(iso["achieved"] / peak, 4)

    # End to end through the public API: every step moves all workers'
    # gradients from pinned host memory to the GPU and reads the step's result
    # (kept indices + threshold) back on the host.  Two ways of moving the
    # gradients are timed: (a) one copy-engine copy into a device buffer
    # followed by fc_step, (b) fc_step reading the pinned host buffer in
    # place over the CPU-GPU link, so the reduction consumes the gradients
    # as they arrive (the transfer and the reduction overlap).
    # The materialised-pack mode, reported separately: the five calls one by
    # one, fc_fuse_pack writing the fused [W][N] buffer that the pipeline
    # never materialises, on buffers of their own.  Every rank reaches the
    # same collectives whether or not its run worked.
    mat, mat_err, mt_local = None, None, float("inf")
    KM = min(K, 200)
    torch.cuda.synchronize()
    barrier()
    try:
        fused = torch.empty(W * N, dtype=torch.float16, device=dev)
        m_a = torch.empty(N, dtype=torch.float32, device=dev)
        m_r = torch.zeros(N, dtype=torch.float32, device=dev)
        m_v = torch.zeros(N, dtype=torch.float32, device=dev)
        m_w = eng.weights.clone()
        m_norms = torch.empty(C, dtype=torch.float32, device=dev)
        m_idx = torch.empty(eng.k, dtype=torch.int32, device=dev)
        m_mask = torch.empty(C, dtype=torch.uint8, device=dev)
        m_packed = torch.empty(eng.k * wl.chunk, dtype=torch.float32, device=dev)
        m_thr = torch.empty(1, dtype=torch.float32, device=dev)

        def five_calls():
            fc.fc_fuse_pack(table, fused, s)
            fc.fc_tree_reduce(fused, W, N, wl.loss_scale, m_r, m_a, s)
            fc.fc_chunk_norms(m_a, N, wl.chunk, m_norms, s)
            fc.fc_chunk_select(m_norms, C, eng.k, m_a, N, wl.chunk, m_idx, m_mask, m_packed,
                               m_thr, None, 1.0, s)
            fc.fc_residual_sgd_update(m_a, m_mask, N, wl.chunk, wl.lr, wl.momentum, m_r, m_v,
                                      m_w, None, s)

        for _ in range(3):
            five_calls()
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        m0.record(s)
        for _ in range(KM):
            five_calls()
        m1.record(s)
        torch.cuda.synchronize()
        mt_local = m0.elapsed_time(m1) / 1e3
        del fused, m_a, m_r, m_v, m_w, m_norms, m_idx, m_mask, m_packed, m_thr
    except Exception as exc:
        mat_err = str(exc).splitlines()[0][:120] if str(exc) else type(exc).__name__
    mt = max_t(mt_local)
    if mat_err is None and mt != float("inf"):
        kept_el = min(N, eng.k * wl.chunk)
        # a1 read + write; a2 fused read, residual read, a write; a3 a read;
        # a4 norms and the kept chunks gathered; a5 a read, r write, v and w
        # read + write
        mat_alg = (4 * W * N) + (2 * W * N + 8 * N) + 4 * N + (4 * C + 8 * kept_el) + 24 * N
        mat = {"value": round(replica_value(world, W * N * 2, KM, mt), 3), "unit": UNIT,
               "ms_per_step": round(mt * 1e3 / KM, 5), "steps": KM,
               "algorithmic_bytes_per_step": int(mat_alg),
               "frac": round(mat_alg / (mt / KM) / 1e9 / peak, 4),
               "calls": "fc_fuse_pack, fc_tree_reduce, fc_chunk_norms, fc_chunk_select, "
                        "fc_residual_sgd_update"}
    else:
        mat = {"unavailable": mat_err or "the run failed on another rank"}
    torch.cuda.empty_cache()

    # the same step captured once in a CUDA graph and replayed: no host work
    # per step (the library's calls are capture-safe).  Every rank reaches
    # the same collectives whether or not its capture worked.
    graph, graph_err, gt_local, gm_local = None, None, float("inf"), float("inf")
    KG = min(K, 1000)
    SG = 50                      # steps captured in one graph for the second figure
    RG = max(2, KG // SG)
    torch.cuda.synchronize()
    barrier()
    try:
        gs = torch.cuda.Stream(device=dev)
        gs.wait_stream(s)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=gs):
            eng.step(table)
        with torch.cuda.stream(gs):
            for _ in range(max(3, warmup)):
                cg.replay()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            g0.record(gs)
            for _ in range(KG):
                cg.replay()
            g1.record(gs)
        torch.cuda.synchronize()
        gt_local = g0.elapsed_time(g1) / 1e3
        del cg
        # SG steps in one graph: the GPU time of a step with no per-step
        # graph launch either (what a step costs inside a longer captured
        # training iteration)
        cm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cm, stream=gs):
            for _ in range(SG):
                eng.step(table)
        with torch.cuda.stream(gs):
            cm.replay()
            g0.record(gs)
            for _ in range(RG):
                cm.replay()
            g1.record(gs)
        torch.cuda.synchronize()
        gm_local = g0.elapsed_time(g1) / 1e3
        del cm
    except Exception as exc:  # capture needs a driver that supports it
        graph_err = str(exc).splitlines()[0][:120] if str(exc) else type(exc).__name__
    gt = max_t(gt_local)
    gm = max_t(gm_local)
    if graph_err is None and gt != float("inf"):
        graph = {"value": round(replica_value(world, W * N * 2, KG, gt), 3), "unit": UNIT,
                 "ms_per_step": round(gt * 1e3 / KG, 5), "steps": KG,
                 "note": "one fc_step captured in a CUDA graph, replayed",
                 "many_steps_per_graph": {
                     "ms_per_step": round(gm * 1e3 / (RG * SG), 5), "steps": RG * SG,
                     "steps_per_graph": SG,
                     "note": "%d fc_steps captured in one CUDA graph, replayed %d times" % (SG, RG)}}
    else:
        graph = {"unavailable": graph_err or "capture failed on another rank"}

    e2e = None
    if args.e2e_steps > 0:
        host = torch.empty(W * N, dtype=torch.float16, pin_memory=True)
        hv = host.numpy()
        pos = 0
        for row in grads_np:
            for g in row:
                hv[pos:pos + g.size] = g
                pos += g.size
        stage = torch.empty(W * N, dtype=torch.float16, device=dev)

        def views(buf):
            out, p = [], 0
            for w in range(W):
                r = []
                for n in wl.sizes:
                    r.append(buf[p:p + n])
                    p += n
                out.append(r)
            return out

        res_idx = torch.empty(eng.k, dtype=torch.int32, pin_memory=True)
        res_thr = torch.empty(1, dtype=torch.float32, pin_memory=True)
        # (c): the copy split into four parts on four streams, so that
        # several copy engines share the transfer
        copy_streams = [torch.cuda.Stream(device=dev) for _ in range(4)]
        bounds = [len(hv) * i // 4 for i in range(5)]
        parts = [(host[bounds[i]:bounds[i + 1]], stage[bounds[i]:bounds[i + 1]])
                 for i in range(4)]
        # (d): backprop order, last layer first.  The buffers are laid out
        # group-major ([group][worker][group's elements]) so that each layer
        # group arrives with one copy on its own stream, and phase 1 reduces
        # the group's span as soon as its copy has landed (fc_step_reduce_span)
        groups = layer_groups_reverse(wl.sizes, 4)
        group_stream = torch.cuda.Stream(device=dev)
        gspan, gpos = group_major_layout(wl.sizes, W, groups)
        group_parts = [(host[a:b], stage[a:b]) for a, b in gspan]

        def group_views(buf):
            return [[buf[gpos[w][l]: gpos[w][l] + wl.sizes[l]] for l in range(wl.L)]
                    for w in range(W)]

        def fill_group_major():
            for w in range(W):
                for l in range(wl.L):
                    hv[gpos[w][l]: gpos[w][l] + wl.sizes[l]] = grads_np[w][l]

        variants = {}
        for name, copy_in in (("copy_engine", 1), ("copy_engine_x4", 4), ("zero_copy", 0),
                              ("layer_groups", 2)):
            if copy_in == 2:
                fill_group_major()
                e_table = fc.PtrTable(group_views(stage))
            else:
                e_table = fc.PtrTable(views(host if copy_in == 0 else stage))

            def one_step():
                if copy_in == 2:
                    group_stream.wait_stream(s)     # the previous step is done with `stage`
                    ready = []
                    with torch.cuda.stream(group_stream):
                        for hpart, dpart in group_parts:
                            dpart.copy_(hpart, non_blocking=True)
                            ev = torch.cuda.Event()
                            ev.record(group_stream)
                            ready.append(ev)
                    eng.step_layer_groups(e_table, groups, ready=ready, stream=s)
                    with torch.cuda.stream(s):
                        res_idx.copy_(eng.idx, non_blocking=True)
                        res_thr.copy_(eng.threshold, non_blocking=True)
                    s.synchronize()
                    return int(res_idx[0]), float(res_thr[0])
                if copy_in == 1:
                    with torch.cuda.stream(s):
                        stage.copy_(host, non_blocking=True)
                elif copy_in == 4:
                    for cs, (hpart, dpart) in zip(copy_streams, parts):
                        cs.wait_stream(s)       # the previous step is done with `stage`
                        with torch.cuda.stream(cs):
                            dpart.copy_(hpart, non_blocking=True)
                    for cs in copy_streams:
                        s.wait_stream(cs)
                eng.step(e_table, s)
                with torch.cuda.stream(s):
                    res_idx.copy_(eng.idx, non_blocking=True)
                    res_thr.copy_(eng.threshold, non_blocking=True)
                s.synchronize()         # the host reads the step's result
                return int(res_idx[0]), float(res_thr[0])

            for _ in range(2):
                one_step()
            barrier()
            E = args.e2e_steps
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(s)
            for _ in range(E):
                one_step()
            e1.record(s)
            torch.cuda.synchronize()
            et = max_t(e0.elapsed_time(e1) / 1e3)
            variants[name] = {"value": round(replica_value(world, step_bytes, E, et), 3),
                              "ms_per_step": round(et * 1e3 / E, 4), "steps": E}
        # the link itself: the same bytes copied host -> device, nothing else
        with torch.cuda.stream(s):
            stage.copy_(host, non_blocking=True)
        torch.cuda.synchronize()
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(s)
        with torch.cuda.stream(s):
            for _ in range(3):
                stage.copy_(host, non_blocking=True)
        l1.record(s)
        torch.cuda.synchronize()
        link_gbs = W * N * 2 * 3 / (l0.elapsed_time(l1) / 1e3) / 1e9
        best = max(variants, key=lambda k: variants[k]["value"])
        e2e = {"value": variants[best]["value"], "unit": UNIT,
               "link": {"h2d_copy_gbs": round(link_gbs, 1),
                        "frac": round(variants[best]["value"] / link_gbs, 4),
                        "note": "pinned host -> device copy of the step's gradients alone"},
               "h2d_bytes_per_step": W * N * 2, "d2h_bytes_per_step": 4 * eng.k + 4,
               "steps": variants[best]["steps"], "ms_per_step": variants[best]["ms_per_step"],
               "path": {"copy_engine": "one pinned-host -> device copy of all workers' "
                                       "gradients, then fc_step",
                        "copy_engine_x4": "the pinned-host -> device copy of all workers' "
                                          "gradients split over four streams, then fc_step",
                        "layer_groups": "layer groups copied in last layer first, one copy "
                                        "per group on a copy stream, phase 1 reducing each "
                                        "group's span as soon as its copy lands "
                                        "(fc_step_reduce_span), then select + update",
                        "zero_copy": "fc_step reading the pinned host gradients in place "
                                     "over the CPU-GPU link"}[best]
                       + "; kept indices + threshold copied back and read on the host",
               "variants": variants}
        del host, stage

    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, sample = cpu_baseline(wl, args.cpu_seconds)
        parity = parity_check(*sample, dev)
        del sample

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded Gaussian fp16 gradients, workload-shaped)",
            "config": config_of(wl, {
                "parallelism": "replicas" if world > 1 else "single GPU",
                "path": ("fc_step in one launch (%s): tree reduce + norms, ranked top-k "
                         "select, residual/momentum-SGD update with packed kept chunks"
                         % ("cooperative, every SM" if path == fc.FC_STEP_ONE_LAUNCH
                            else "one cluster")
                         if one_launch else
                         "fc_step: pack-elided tree reduce + norm partials, radix top-k select, "
                         "residual/momentum-SGD update with packed kept chunks (3 kernels)"),
                "l2": ("inputs larger than L2: %.2f GB fp16 gradients + %.2f GB fp32 state per "
                       "step" if step_bytes + 12 * N > 129e6 else
                       "inputs smaller than L2 (%.4f GB fp16 gradients + %.4f GB fp32 state): "
                       "the step runs from L2, a latency-bound size")
                      % (step_bytes / 1e9, 12 * N / 1e9)}),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic,
                         "traffic_source": ("dram__bytes_read.sum + dram__bytes_write.sum of "
                                            "one launch, from the committed ncu summary "
                                            "profiles/k_reduce_%s.md taken on this kernel "
                                            "source (not measured in this run)" % wl.name)
                                           if traffic is not None else None,
                         "kernel": (one_kernel if one_launch else
                                    "phase 1 of fc_step (%s)" % phase1_kernel(wl, table)),
                         "algorithmic_bytes_per_launch": k_alg,
                         "avg_launch_ms": round(k_ms, 5),
                         "median_launch_ms": round(statistics.median(reduce_ms), 5),
                         "peak_source": peak_src + " hbm_gbs",
                         "timed_launches": len(reduce_ms),
                         "isolated": iso},
            "step_roofline": {"algorithmic_bytes_per_step": int(step_alg),
                              "full_count_bytes_per_step": int(alg["full_count"]),
                              "achieved_gbs": round(step_alg / (ms_per_step / 1e3) / 1e9, 1),
                              "frac": round(step_alg / (ms_per_step / 1e3) / 1e9 / peak, 4),
                              "full_count_frac": round(alg["full_count"] / (ms_per_step / 1e3)
                                                         / 1e9 / peak, 4),
                              "select_update_ms": round(rest_ms, 5)},
            "cpu_baseline": cpu,
            "parity": parity,
            "e2e": e2e,
            "graph": graph,
            "materialised_pack": mat,
            "gpu_launches": (1 if one_launch else 3) * K,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    rank, world, local = dist_env()
    wl = workload.get(args.workload)
    if args.elements:
        wl = sample_workload(wl, args.elements)
    if args.impl == "reference":
        return run_reference(args, wl, rank)
    return run_gpu(args, wl, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
