"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Covers the five workloads at full size with state carried over their steps,
both the fused pipeline (fc_step) and the five separate calls, and small
random shapes that span several tiles with ragged tails, odd worker counts,
layers that break 16-byte alignment, short last chunks, ties, a single
element and the degenerate keep-all / keep-one cases.
"""

import numpy as np
import pytest
import torch

import oracle
from gradient_aggregation_gb300 import fc, workload
from tests.gpu_util import DeviceRun, bits_equal, dev_grads, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fc_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield


def _compare_paths(p, s):
    for key in ("a", "norms", "idx", "mask", "threshold", "residual", "velocity",
                "weights", "packed", "packed16", "w16"):
        if key in p and key in s:
            assert bits_equal(np.asarray(p[key]), np.asarray(s[key])), key


def _run_workload(wl, steps=None, both_paths=True, expect_kernel=None, to_dev=dev_grads):
    """Steps the pipeline (fc_step) and, with both_paths, the five separate
    calls; when fc_step runs the layout as one launch, also the three phase
    calls, so that the phase-1 kernel `expect_kernel` names really runs.
    Every path must give the same bits, and the oracle's."""
    steps = wl.steps if steps is None else steps
    runs = None
    st = oracle.State(workload.initial_weights(wl))
    reports = []
    for s in range(steps):
        g_np = workload.all_grads(wl, s)
        g_dev = to_dev(g_np)
        if runs is None:
            runs = [DeviceRun(wl, "pipeline")]
            if fc.fc_step_path(g_dev, wl.chunk) != fc.FC_STEP_THREE_KERNELS:
                runs.append(DeviceRun(wl, "phases"))
            if both_paths:
                runs.append(DeviceRun(wl, "separate"))
        if expect_kernel is not None:
            assert fc.fc_step_reduce_kernel(g_dev, wl.chunk) == expect_kernel
        snaps = []
        for r in runs:
            r.step(g_dev)
            snaps.append(r.snapshot())
        del g_dev
        for other in snaps[1:]:
            _compare_paths(snaps[0], other)
        if both_paths:
            assert runs[-1].offsets == list(oracle.layout(wl.sizes)[0])
        reports.append(oracle_step(g_np, st, wl, snaps[-1]))
        del g_np, snaps
    torch.cuda.empty_cache()
    return reports


WORKLOAD_KERNEL = {"tiny": fc.FC_REDUCE_STAGED, "nin": fc.FC_REDUCE_STAGED_SHIFTED,
                   "googlenet": fc.FC_REDUCE_STAGED_SHIFTED, "alexnet": fc.FC_REDUCE_STAGED_SHIFTED,
                   "stress": fc.FC_REDUCE_REGISTER}


@pytest.mark.parametrize("name", ["tiny", "nin", "googlenet", "alexnet", "stress"])
def test_workload_parity(name):
    wl = workload.get(name)
    reports = _run_workload(wl, both_paths=name != "stress",
                            expect_kernel=WORKLOAD_KERNEL[name])
    assert len(reports) == wl.steps


def _sizes_n8(sizes):
    """Pads the last layer so that N is a multiple of 8 (the staged kernels'
    condition)."""
    sizes = [int(x) for x in sizes]
    sizes[-1] += (-sum(sizes)) % 8
    return sizes


def _shifted_dev(shift_bytes):
    """Device copies of every worker's layers starting `shift_bytes` past a
    16-byte boundary (the same for all workers)."""
    def to_dev(g_np):
        out = []
        for row in g_np:
            r = []
            for g in row:
                buf = torch.empty(g.size + 8, dtype=torch.float16, device="cuda")
                view = buf[shift_bytes // 2: shift_bytes // 2 + g.size]
                view.copy_(torch.from_numpy(g))
                assert view.data_ptr() % 16 == shift_bytes
                r.append(view)
            out.append(r)
        return out
    return to_dev


def test_shifted_layout_odd_layer_sizes():
    """Layers of odd sizes: every layer has its own shift, pieces start and
    end inside tiles, the bulk copies run past the tile ends."""
    rng = np.random.default_rng(7)
    for W, chunk, cid in [(16, 512, 160), (8, 2048, 161), (4, 256, 162)]:
        sizes = _sizes_n8(np.exp(rng.uniform(0, np.log(5000), 40)).astype(int) + 1)
        wl = workload.custom(W=W, sizes=sizes, chunk=chunk, keep_percent=25,
                             config_id=cid, steps=2, loss_scale=512.0)
        _run_workload(wl, expect_kernel=fc.FC_REDUCE_STAGED_SHIFTED)


@pytest.mark.parametrize("W,L,cid", [(8, 300, 163), (16, 190, 167)])
def test_shifted_layout_many_tiny_layers(W, L, cid):
    """Hundreds of 1..20-element layers: tiles with more pieces than the
    stage's piece table, whose rest is read from global memory (with 16
    workers, at the second of the tile's two stages).  L stays within
    FC_MAX_TABLE_PTRS worker-layer pointers."""
    rng = np.random.default_rng(8)
    sizes = _sizes_n8(rng.integers(1, 21, L))
    wl = workload.custom(W=W, sizes=sizes, chunk=256, keep_percent=30, config_id=cid, steps=2)
    _run_workload(wl, expect_kernel=fc.FC_REDUCE_STAGED_SHIFTED)


def test_shifted_layout_gaps_past_the_slack():
    """Runs of 9-element layers lower the shift at every boundary, so the gaps
    between pieces outgrow the row's slack and later pieces are unstaged."""
    sizes = _sizes_n8([9] * 20 + [5000] + [9] * 40 + [3000, 17, 2500])
    for W, cid in [(4, 164), (16, 165)]:
        wl = workload.custom(W=W, sizes=sizes, chunk=256, keep_percent=20, config_id=cid,
                             steps=2)
        _run_workload(wl, expect_kernel=fc.FC_REDUCE_STAGED_SHIFTED)


@pytest.mark.parametrize("shift", [2, 6, 14])
def test_shifted_layout_uniform_pointer_shift(shift):
    """Layers at multiples of 8 elements, but every worker's tensors start
    `shift` bytes past a 16-byte boundary."""
    wl = workload.custom(W=16, sizes=[4096, 808, 8, 6000], chunk=256, keep_percent=25,
                         config_id=166 + shift, steps=2)
    _run_workload(wl, expect_kernel=fc.FC_REDUCE_STAGED_SHIFTED, to_dev=_shifted_dev(shift))


SMALL_CASES = [
    # W, sizes, chunk, keep percent
    (1, [1], 1, 100),
    (1, [7], 3, 50),
    (2, [9, 4], 4, 50),
    (3, [1000], 8, 10),
    (5, [17, 33, 1, 2048, 5], 100, 30),
    (7, [4096, 3, 4099], 2048, 40),
    (8, [2049, 2047], 2049, 50),
    (9, [12345], 5000, 67),
    (16, [96, 130, 1, 8, 7, 4000], 256, 25),
    (17, [3000, 3001], 64, 10),
    (33, [513, 1027], 512, 20),
    (64, [20000], 4096, 10),
    (65, [999], 128, 90),
    (4, [3, 0, 5, 0, 8], 2, 60),
    (2, [100000], 32768, 1),
]


@pytest.mark.parametrize("case", SMALL_CASES, ids=[str(i) for i in range(len(SMALL_CASES))])
def test_small_shapes(case):
    W, sizes, chunk, keep = case
    wl = workload.custom(W=W, sizes=sizes, chunk=chunk, keep_percent=keep,
                         config_id=100 + W, steps=3, loss_scale=1000.0)
    _run_workload(wl)


def test_heavy_tail_small():
    wl = workload.custom(W=8, sizes=[50000, 3], chunk=512, keep_percent=10,
                         heavy_tail=True, grad_std=1e-3, steps=3, config_id=140)
    _run_workload(wl)


def test_misaligned_gradient_pointers():
    """Layer tensors that start 2 bytes past a 16-byte boundary take the
    element-wise path and still match."""
    wl = workload.custom(W=6, sizes=[1001, 64, 3333], chunk=300, keep_percent=20,
                         config_id=150, steps=2)
    st = oracle.State(workload.initial_weights(wl))
    run = DeviceRun(wl, "pipeline")
    sep = DeviceRun(wl, "separate")
    for s in range(2):
        g_np = workload.all_grads(wl, s)
        g_dev = []
        for row in g_np:
            r = []
            for g in row:
                buf = torch.empty(g.size + 1, dtype=torch.float16, device="cuda")
                view = buf[1:]
                view.copy_(torch.from_numpy(g))
                assert view.data_ptr() % 16 == 2
                r.append(view)
            g_dev.append(r)
        run.step(g_dev)
        sep.step(g_dev)
        a, b = run.snapshot(), sep.snapshot()
        _compare_paths(a, b)
        oracle_step(g_np, st, wl, b)


def test_fused_buffer_with_ragged_rows():
    """N % 8 != 0: the fused rows are not 16-byte aligned."""
    wl = workload.custom(W=3, sizes=[1234, 7], chunk=100, keep_percent=50,
                         config_id=151, steps=1)
    g_np = workload.all_grads(wl, 0)
    run = DeviceRun(wl, "separate")
    run.step(dev_grads(g_np))
    oracle_step(g_np, oracle.State(workload.initial_weights(wl)), wl, run.snapshot())


def test_ties_keep_lowest_indices():
    """Every chunk has the same norm: the k lowest chunk indices are kept, by
    the one-launch step, the three pipeline kernels and the five calls."""
    W, N, cs = 4, 64 * 10, 64
    wl = workload.custom(W=W, sizes=[N], chunk=cs, keep_percent=30, config_id=152)
    g = [[np.full(N, 2.0, dtype=np.float16)] for _ in range(W)]
    for path in ("pipeline", "phases", "separate"):
        run = DeviceRun(wl, path)
        run.step(dev_grads(g))
        snap = run.snapshot()
        assert list(snap["idx"]) == [0, 1, 2]
        oracle_step(g, oracle.State(workload.initial_weights(wl)), wl, snap)


@pytest.mark.parametrize("C", [40, 1000, 5000])
def test_threshold_inside_a_group_of_ties(C):
    """Every fifth chunk is large, all others share one smaller norm, and
    the k-th chunk falls among the equal ones: the large chunks and the
    lowest-indexed equal ones are kept, on every path."""
    W, cs = 4, 64
    wl = workload.custom(W=W, sizes=[C * cs], chunk=cs, keep_percent=30, config_id=153)
    vals = np.where(np.arange(C) % 5 == 0, 4.0, 1.0).astype(np.float16)
    g = [[np.repeat(vals, cs)] for _ in range(W)]
    k = fc.fc_keep_count(C, 30, 100)
    big = [c for c in range(C) if c % 5 == 0]
    rest = [c for c in range(C) if c % 5][: k - len(big)]
    want = sorted(big + rest)
    for path in ("pipeline", "phases", "separate"):
        run = DeviceRun(wl, path)
        run.step(dev_grads(g))
        snap = run.snapshot()
        assert list(snap["idx"]) == want, path
        oracle_step(g, oracle.State(workload.initial_weights(wl)), wl, snap)


def test_keep_one_and_partial_last_chunk_padding():
    wl = workload.custom(W=2, sizes=[1000], chunk=300, keep_percent=1, config_id=153)
    g = [[np.zeros(1000, np.float16)] for _ in range(2)]
    g[0][0][950:] = 4.0       # the short last chunk (100 elements) wins
    run = DeviceRun(wl, "pipeline")
    run.packed.fill_(7.0)
    run.step(dev_grads(g))
    snap = run.snapshot()
    assert list(snap["idx"]) == [3]
    assert np.all(snap["packed"][100:] == 0.0)
    oracle_step(g, oracle.State(workload.initial_weights(wl)), wl, snap)


@pytest.mark.parametrize("path", ["pipeline", "phases"])
def test_inplace_matches_out_of_place_and_is_deterministic(path):
    wl = workload.custom(W=16, sizes=[40000, 123, 70001], chunk=4096, keep_percent=25,
                         config_id=154, steps=3)
    runs = [DeviceRun(wl, path, inplace=True), DeviceRun(wl, path, inplace=False),
            DeviceRun(wl, path, inplace=True)]
    for s in range(3):
        g = dev_grads(workload.all_grads(wl, s))
        snaps = []
        for r in runs:
            r.step(g)
            snaps.append(r.snapshot())
        for other in snaps[1:]:
            for key in ("residual", "velocity", "weights", "idx", "mask", "norms",
                        "packed", "w16", "threshold"):
                assert bits_equal(np.asarray(snaps[0][key]), np.asarray(other[key])), key


@pytest.mark.parametrize("path", ["pipeline", "phases"])
def test_checkpoint_resume_is_bit_exact(path):
    wl = workload.custom(W=8, sizes=[30000, 5000], chunk=1024, keep_percent=20,
                         config_id=155, steps=5)
    grads = [dev_grads(workload.all_grads(wl, s)) for s in range(5)]
    straight = DeviceRun(wl, path, inplace=True)
    for s in range(5):
        straight.step(grads[s])
    end = straight.snapshot()
    first = DeviceRun(wl, path, inplace=True)
    for s in range(3):
        first.step(grads[s])
    torch.cuda.synchronize()
    saved = {k: getattr(first, k).cpu().clone() for k in ("residual", "velocity", "weights")}
    resumed = DeviceRun(wl, path, inplace=True)
    for k, v in saved.items():
        getattr(resumed, k).copy_(v.cuda())
    for s in range(3, 5):
        resumed.step(grads[s])
    got = resumed.snapshot()
    for key in ("residual", "velocity", "weights", "idx", "w16"):
        assert bits_equal(end[key], got[key]), key


@pytest.mark.parametrize("path", ["pipeline", "phases"])
def test_cuda_graph_replay_matches_eager(path):
    wl = workload.custom(W=4, sizes=[5000, 77], chunk=256, keep_percent=10,
                         config_id=156, steps=3)
    grads = dev_grads(workload.all_grads(wl, 0))
    eager = DeviceRun(wl, path, inplace=True)
    graphed = DeviceRun(wl, path, inplace=True)
    table = fc.PtrTable(grads)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graphed.step(table, s)          # warm-up outside capture (step 1)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.step(table)
    eager.step(grads)
    for _ in range(3):                  # steps 2..4
        eager.step(grads)
        g.replay()
    a, b = eager.snapshot(), graphed.snapshot()
    for key in ("residual", "velocity", "weights", "idx", "norms"):
        assert bits_equal(a[key], b[key]), key


def test_device_argument_errors():
    dev = "cuda"
    a = torch.zeros(1000, dtype=torch.float32, device=dev)
    with pytest.raises(fc.FcError) as e:
        fc.fc_chunk_norms(a[1:], 999, 10, torch.empty(100, device=dev))
    assert e.value.status == fc.FC_ERR_ALIGNMENT
    wl = workload.custom(W=2, sizes=[1000], chunk=100, keep_percent=10, config_id=157)
    run = DeviceRun(wl, "pipeline")
    run.ws = run.ws[:16]
    with pytest.raises(fc.FcError) as e:
        run.step(dev_grads(workload.all_grads(wl, 0)))
    assert e.value.status == fc.FC_ERR_WORKSPACE


ORDER_CASES = [
    (3, [1000, 7], 64),
    (5, [17, 33, 1, 2048, 5], 100),
    (16, [40000, 123, 70001], 4096),
    (64, [20000], 4096),
    (7, [3], 2),
]


@pytest.mark.parametrize("order", [oracle.ORDER_SEQUENTIAL, oracle.ORDER_RING])
@pytest.mark.parametrize("case", ORDER_CASES, ids=[str(i) for i in range(len(ORDER_CASES))])
def test_summation_orders(order, case):
    """Parameter-server and ring orders: the materialised path and the
    pipeline's phase 1 both match the oracle bit for bit, and the pipeline's
    norms follow."""
    W, sizes, chunk = case
    wl = workload.custom(W=W, sizes=sizes, chunk=chunk, keep_percent=20,
                         config_id=180 + W, loss_scale=1000.0)
    g_np = workload.all_grads(wl, 0)
    rng = np.random.default_rng(W)
    r_np = (rng.standard_normal(wl.N) * 1e-3).astype(np.float32)
    want = oracle.reduce_ordered(oracle.fuse_pack(g_np), wl.loss_scale, r_np, order)
    g = dev_grads(g_np)
    r = torch.from_numpy(r_np).cuda()
    fused = torch.empty(W * wl.N, dtype=torch.float16, device="cuda")
    fc.fc_fuse_pack(g, fused)
    out = torch.empty(wl.N, dtype=torch.float32, device="cuda")
    fc.fc_reduce_ordered(fused, W, wl.N, wl.loss_scale, r, out, order)
    ws = torch.zeros(fc.fc_step_workspace_size(wl.N, chunk), dtype=torch.uint8, device="cuda")
    a = torch.empty(wl.N, dtype=torch.float32, device="cuda")
    fc.fc_step_reduce_ordered(g, wl.loss_scale, chunk, r, a, order, ws)
    C = fc.fc_num_chunks(wl.N, chunk)
    norms = torch.empty(C, dtype=torch.float32, device="cuda")
    idx = torch.empty(1, dtype=torch.int32, device="cuda")
    mask = torch.empty(C, dtype=torch.uint8, device="cuda")
    thr = torch.empty(1, dtype=torch.float32, device="cuda")
    fc.fc_step_select(wl.N, chunk, 1, norms, idx, mask, thr, ws)
    torch.cuda.synchronize()
    assert bits_equal(out.cpu().numpy(), want)
    assert bits_equal(a.cpu().numpy(), want)
    from tests.gpu_util import assert_close, RTOL_NORM
    assert_close("norms", norms.cpu().numpy(), oracle.chunk_norms(want, chunk), RTOL_NORM)


@pytest.mark.parametrize("order", [oracle.ORDER_SEQUENTIAL, oracle.ORDER_RING])
def test_summation_orders_googlenet(order):
    wl = workload.get("googlenet")
    g_np = workload.all_grads(wl, 0)
    want = oracle.reduce_ordered(oracle.fuse_pack(g_np), wl.loss_scale, None, order)
    ws = torch.zeros(fc.fc_step_workspace_size(wl.N, wl.chunk), dtype=torch.uint8,
                     device="cuda")
    a = torch.empty(wl.N, dtype=torch.float32, device="cuda")
    fc.fc_step_reduce_ordered(dev_grads(g_np), wl.loss_scale, wl.chunk, None, a, order, ws)
    torch.cuda.synchronize()
    assert bits_equal(a.cpu().numpy(), want)
    # the orders differ from the tree by rounding only
    tree = oracle.tree_reduce(oracle.fuse_pack(g_np), wl.loss_scale)
    from tests.gpu_util import assert_close
    assert_close("order vs tree", want, tree, 1e-5)


def test_engine_phase_calls_equal_fused_step():
    """The three phase entry points in sequence are fc_step; Engine state
    round-trips through state_dict."""
    wl = workload.custom(W=16, sizes=[8192, 4096, 24576], chunk=2048, keep_percent=25,
                         config_id=190, steps=2)
    w0 = torch.from_numpy(workload.initial_weights(wl)).cuda()
    engines = [fc.Engine(wl.sizes, wl.W, wl.chunk, wl.keep_percent, 100, wl.loss_scale,
                         wl.lr, wl.momentum, w0, want_fp16=True, want_packed_fp16=True,
                         send_scale=wl.loss_scale) for _ in range(2)]
    for s in range(2):
        table = fc.PtrTable(dev_grads(workload.all_grads(wl, s)))
        engines[0].step(table)
        for phase in engines[1].phases(table):
            phase()
    torch.cuda.synchronize()
    a, b = engines
    for name in ("residual", "velocity", "weights", "weights_fp16", "norms", "idx", "mask",
                 "packed", "packed_fp16", "threshold"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    sd = a.state_dict()
    c = fc.Engine(wl.sizes, wl.W, wl.chunk, wl.keep_percent, 100, wl.loss_scale, wl.lr,
                  wl.momentum, w0)
    c.load_state_dict(sd)
    assert torch.equal(c.weights, a.weights) and torch.equal(c.residual, a.residual)


def test_tree_order_entry_points_agree():
    wl = workload.custom(W=8, sizes=[3000, 5000], chunk=512, keep_percent=10, config_id=191)
    g = dev_grads(workload.all_grads(wl, 0))
    fused = torch.empty(wl.W * wl.N, dtype=torch.float16, device="cuda")
    fc.fc_fuse_pack(g, fused)
    outs = [torch.empty(wl.N, dtype=torch.float32, device="cuda") for _ in range(4)]
    fc.fc_tree_reduce(fused, wl.W, wl.N, wl.loss_scale, None, outs[0])
    fc.fc_reduce_ordered(fused, wl.W, wl.N, wl.loss_scale, None, outs[1], fc.FC_ORDER_TREE)
    ws = torch.zeros(fc.fc_step_workspace_size(wl.N, wl.chunk), dtype=torch.uint8, device="cuda")
    fc.fc_step_reduce(g, wl.loss_scale, wl.chunk, None, outs[2], ws)
    fc.fc_step_reduce_ordered(g, wl.loss_scale, wl.chunk, None, outs[3], fc.FC_ORDER_TREE, ws)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_capacity_limits_many_workers_and_layers():
    """The largest pointer tables one call accepts: W*L = FC_MAX_TABLE_PTRS
    (3072 workers of one layer; 6 workers of 512 layers)."""
    for W, sizes, chunk in ((fc.FC_MAX_TABLE_PTRS, [24], 8),
                            (6, [1 + (i * 7) % 13 for i in range(fc.FC_MAX_TABLE_LAYERS)], 64)):
        wl = workload.custom(W=W, sizes=sizes, chunk=chunk, keep_percent=30,
                             config_id=200 + (W % 100), loss_scale=4096.0)
        _run_workload(wl, steps=1, both_paths=True)


def test_more_chunks_than_the_select_kernel_keeps_in_shared_memory():
    """C = 12,000 chunks of one element (above the 11,264 keys the selection
    holds in shared memory): the keys are read from global memory."""
    wl = workload.custom(W=3, sizes=[12000], chunk=1, keep_percent=10, config_id=210)
    _run_workload(wl, steps=2)


def test_select_with_only_the_fp16_send_buffer():
    wl = workload.custom(W=4, sizes=[5000], chunk=100, keep_percent=20, config_id=211)
    g_np = workload.all_grads(wl, 0)
    a_np = oracle.tree_reduce(oracle.fuse_pack(g_np), wl.loss_scale)
    norms_np = oracle.chunk_norms(a_np, wl.chunk)
    k = oracle.keep_count(norms_np.size, wl.keep_percent, 100)
    idx_o, mask_o, packed_o, thr_o = oracle.chunk_select(norms_np, k, a_np, wl.chunk)
    a = torch.from_numpy(a_np).cuda()
    norms = torch.from_numpy(norms_np).cuda()
    idx = torch.empty(k, dtype=torch.int32, device="cuda")
    mask = torch.empty(norms_np.size, dtype=torch.uint8, device="cuda")
    thr = torch.empty(1, dtype=torch.float32, device="cuda")
    p16 = torch.empty(k * wl.chunk, dtype=torch.float16, device="cuda")
    fc.fc_chunk_select(norms, norms_np.size, k, a, wl.N, wl.chunk, idx, mask, None, thr,
                       packed_fp16=p16, send_scale=wl.loss_scale)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    assert np.array_equal(mask.cpu().numpy(), mask_o)
    assert bits_equal(p16.cpu().numpy().view(np.uint16), oracle.pack_fp16(packed_o, wl.loss_scale))


def _norm_patterns(kind, C, rng):
    """Non-negative finite binary32 norms whose bit patterns agree above a
    chosen bit: the radix select's digits are then constant in its first
    passes and spread only in the last ones (or, for "wide", from the
    first)."""
    if kind == "low5":        # differ in bits 4..0 only
        bits = 0x3F800000 + rng.integers(0, 32, C)
    elif kind == "low20":     # differ in bits 19..0
        bits = 0x3C500000 + rng.integers(0, 1 << 20, C)
    elif kind == "wide":      # every exponent from 2^-126 up
        bits = rng.integers(0x00800000, 0x7F000000, C)
    elif kind == "equal":     # all keys the same
        bits = np.full(C, 0x3E4CCCCD)
    elif kind == "two":       # two values in bit 0 only, many ties at tau
        bits = 0x3F000000 + (rng.random(C) < 0.5)
    else:
        raise ValueError(kind)
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


@pytest.mark.parametrize("kind", ["low5", "low20", "wide", "equal", "two"])
@pytest.mark.parametrize("C", [1, 37, 1904, 11264, 11265])
def test_select_on_norms_sharing_leading_bits(kind, C):
    """fc_chunk_select against the oracle's selection on norms that share
    their leading bits, for k = 1, 30 %, C - 1 and C: kept set, index list
    and threshold exact.  C = 11,265 keys are more than the selection holds
    in shared memory, so they are read from global memory."""
    rng = np.random.default_rng(300 + C + len(kind))
    norms_np = _norm_patterns(kind, C, rng)
    norms = torch.from_numpy(norms_np).cuda()
    for k in sorted({1, max(1, (3 * C) // 10), max(1, C - 1), C}):
        idx_o, mask_o, _, thr_o = oracle.chunk_select(norms_np, k)
        idx = torch.empty(k, dtype=torch.int32, device="cuda")
        mask = torch.empty(C, dtype=torch.uint8, device="cuda")
        thr = torch.empty(1, dtype=torch.float32, device="cuda")
        fc.fc_chunk_select(norms, C, k, None, C, 1, idx, mask, None, thr)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), idx_o), (kind, C, k)
        assert np.array_equal(mask.cpu().numpy(), mask_o), (kind, C, k)
        assert bits_equal(thr.cpu().numpy(), np.asarray(thr_o, np.float32).reshape(1)), (kind, C, k)


@pytest.mark.parametrize("inplace", [False, True], ids=["separate_a", "inplace"])
@pytest.mark.parametrize("W,sizes,kind", [
    (16, [8192, 16384, 40960], fc.FC_REDUCE_STAGED),
    (16, [8191, 16385, 40960], fc.FC_REDUCE_STAGED_SHIFTED),
    (8, [8191, 16385, 40960], fc.FC_REDUCE_STAGED_SHIFTED)],
    ids=["aligned", "shifted", "shifted_w8"])
def test_staged_reduction_reports_a_wait_that_runs_out(W, sizes, kind, inplace):
    """Failure path of the TMA-staged reduction, without any fault: the test
    hook makes the next launch issue no copies for tile 0, so the waits on it
    run out (20 ms limit).  The step reports it (NaN threshold, nothing kept,
    idx -1, FC_ERR_TIMEOUT from fc_step_status) and is not applied: velocity,
    weights and the fp16 weights keep their bits, and with a separate `a`
    buffer so does the residual, so the same step can be run again and then
    matches the oracle.  The context stays usable throughout.  With 16
    workers in the shifted layout each tile is two stages (worker halves);
    with 8, two CTAs share an SM."""
    wl = workload.custom(W=W, sizes=sizes, chunk=4096, keep_percent=25,
                         config_id=220, steps=3)
    run = DeviceRun(wl, "pipeline", inplace=inplace)
    st = oracle.State(workload.initial_weights(wl))
    g_np = [workload.all_grads(wl, s) for s in range(2)]
    g0, g1 = dev_grads(g_np[0]), dev_grads(g_np[1])
    assert fc.fc_step_reduce_kernel(g0, wl.chunk) == kind
    run.step(g0)                                   # a good step first: state is non-trivial
    before = run.snapshot()
    oracle_step(g_np[0], st, wl, before, check_a=False)
    assert fc.fc_step_status(run.ws, run.N, wl.chunk) == fc.FC_OK
    fc.fc_test_stage_loss(0, 20_000_000)
    run.step(g1)                                   # this one fails
    snap = run.snapshot()
    assert np.isnan(snap["threshold"])
    assert not snap["mask"].any() and np.all(snap["idx"] == -1)
    assert fc.fc_step_status(run.ws, run.N, wl.chunk) == fc.FC_ERR_TIMEOUT
    unchanged = ["velocity", "weights", "w16", "packed", "packed16"]
    if not inplace:
        unchanged.append("residual")
    for key in unchanged:
        assert bits_equal(snap[key], before[key]), key + " changed by a step that failed"
    if not inplace:
        # the step is retried as it is and gives the oracle's bits
        run.step(g1)
        oracle_step(g_np[1], st, wl, run.snapshot(), check_a=False)
        assert fc.fc_step_status(run.ws, run.N, wl.chunk) == fc.FC_OK
    else:
        # in place, phase 1 consumed the residual: the caller restores it
        run.residual.copy_(torch.from_numpy(before["residual"]).cuda())
        run.step(g1)
        oracle_step(g_np[1], st, wl, run.snapshot(), check_a=False)
        assert fc.fc_step_status(run.ws, run.N, wl.chunk) == fc.FC_OK


def test_bucketed_gradients_merge_into_one_segment():
    """Each worker's layers back to back in one bucket (odd layer sizes):
    the table merges them, the staged reduction applies, and the results are
    those of separately allocated layer tensors, bit for bit."""
    wl = workload.custom(W=16, sizes=[1001, 33, 4099, 7, 60000, 3, 8185],
                         chunk=4096, keep_percent=25, config_id=230, steps=2)
    assert wl.N % 8 == 0
    sep = DeviceRun(wl, "phases")      # phase 1 as its own call: the staged kernel runs
    buck = DeviceRun(wl, "phases")
    buck1 = DeviceRun(wl, "pipeline")  # and the whole step in one launch
    st = oracle.State(workload.initial_weights(wl))
    for s in range(2):
        g_np = workload.all_grads(wl, s)
        bucket = torch.empty(wl.W * wl.N, dtype=torch.float16, device="cuda")
        views, pos = [], 0
        for w in range(wl.W):
            row = []
            for g in g_np[w]:
                v = bucket[pos:pos + g.size]
                v.copy_(torch.from_numpy(g))
                row.append(v)
                pos += g.size
            views.append(row)
        if s == 0:
            assert fc.fc_step_reduce_kernel(views, wl.chunk) == fc.FC_REDUCE_STAGED
        sep.step(dev_grads(g_np))
        buck.step(views)
        buck1.step(views)
        a, b = sep.snapshot(), buck.snapshot()
        _compare_paths(a, b)
        _compare_paths(a, buck1.snapshot())
        oracle_step(g_np, st, wl, b)


def _engine(wl):
    w0 = torch.from_numpy(workload.initial_weights(wl)).cuda()
    return fc.Engine(wl.sizes, wl.W, wl.chunk, wl.keep_percent, 100, wl.loss_scale, wl.lr,
                     wl.momentum, w0, want_fp16=True, want_packed=True,
                     want_packed_fp16=True, send_scale=wl.loss_scale)


def _engine_bits(e):
    return {k: getattr(e, k).cpu().numpy() for k in
            ("residual", "velocity", "weights", "weights_fp16", "norms", "idx", "mask",
             "packed", "packed_fp16", "threshold")}


def _engine_snapshot(e):
    """An Engine's state and outputs in the form oracle_step compares (the
    reduced gradient is formed in place, so there is no separate `a`)."""
    torch.cuda.synchronize()
    b = _engine_bits(e)
    return dict(norms=b["norms"], idx=b["idx"], mask=b["mask"],
                threshold=np.float32(b["threshold"][0]), residual=b["residual"],
                velocity=b["velocity"], weights=b["weights"], packed=b["packed"],
                packed16=b["packed_fp16"].view(np.uint16), send_scale=e.send_scale,
                w16=b["weights_fp16"].view(np.uint16))


def _groupings(L, rng):
    cuts = sorted(rng.choice(np.arange(1, L), size=min(2, L - 1), replace=False)) if L > 1 else []
    b = [0] + [int(c) for c in cuts] + [L]
    three = [(b[i], b[i + 1]) for i in range(len(b) - 1)]
    per_layer = [(l, l + 1) for l in range(L)]
    return [three[::-1], three, per_layer[::-1], [(0, L)]]


SPAN_CASES = {
    "googlenet": None, "nin": None, "tiny": None,
    "aligned16": dict(W=16, sizes=[12288, 808, 8, 60000, 8000], chunk=1024, keep_percent=20),
    "register5": dict(W=5, sizes=[1001, 64, 3333, 2, 700], chunk=300, keep_percent=30),
}


SPAN_KERNEL = {"googlenet": fc.FC_REDUCE_STAGED_SHIFTED, "nin": fc.FC_REDUCE_STAGED_SHIFTED,
               "tiny": fc.FC_REDUCE_STAGED, "aligned16": fc.FC_REDUCE_STAGED,
               "register5": fc.FC_REDUCE_REGISTER}


@pytest.mark.parametrize("name", list(SPAN_CASES))
def test_layer_group_streaming_matches_the_oracle(name):
    """Phase 1 streamed per layer group (fc_step_reduce_span), in backprop
    order (last layer first), in layer order, one group per layer and one
    group for everything: every streamed engine matches the oracle element
    by element on every step (residual, velocity, weights, fp16 weights and
    send buffers bit-exact, the kept set exact outside the 1e-6 band, norms
    within 1e-6), on each of the three phase-1 kernels, and gives the bits
    of fc_step."""
    kw = SPAN_CASES[name]
    wl = workload.get(name) if kw is None else workload.custom(config_id=170, steps=2, **kw)
    rng = np.random.default_rng(11)
    groupings = _groupings(wl.L, rng)
    ref = _engine(wl)
    runs = [_engine(wl) for _ in groupings]
    states = [oracle.State(workload.initial_weights(wl)) for _ in groupings]
    for s in range(2):
        g_np = workload.all_grads(wl, s)
        g_dev = dev_grads(g_np)
        assert fc.fc_step_reduce_kernel(g_dev, wl.chunk) == SPAN_KERNEL[name]
        ref.step(g_dev)
        for eng, groups in zip(runs, groupings):
            eng.step_layer_groups(g_dev, groups)
        want = _engine_bits(ref)
        for eng, groups, st in zip(runs, groupings, states):
            got = _engine_bits(eng)
            for k in want:
                assert bits_equal(got[k], want[k]), (name, groups, k)
            oracle_step(g_np, st, wl, _engine_snapshot(eng))


def test_layer_group_streaming_waits_for_each_group():
    """Gradients copied in group by group (last layer first) on another
    stream, each span waiting only for its own group's event."""
    wl = workload.get("googlenet")
    groups = [(40, 57), (20, 40), (0, 20)]
    ref, eng = _engine(wl), _engine(wl)
    src = dev_grads(workload.all_grads(wl, 0))
    dst = [[torch.full_like(t, float("nan")) for t in row] for row in src]
    ref.step(src)
    copy, comp = torch.cuda.Stream(), torch.cuda.Stream()
    copy.wait_stream(torch.cuda.current_stream())
    comp.wait_stream(torch.cuda.current_stream())
    ready = []
    with torch.cuda.stream(copy):
        for a, b in groups:
            for w in range(wl.W):
                for l in range(a, b):
                    dst[w][l].copy_(src[w][l], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(copy)
            ready.append(ev)
    eng.step_layer_groups(dst, groups, ready=ready, stream=comp)
    torch.cuda.synchronize()
    want, got = _engine_bits(ref), _engine_bits(eng)
    for k in want:
        assert bits_equal(got[k], want[k]), k
    st = oracle.State(workload.initial_weights(wl))
    oracle_step(workload.all_grads(wl, 0), st, wl, _engine_snapshot(eng))


def _counter_words(ws, N, chunk):
    """The first eight 32-bit words of the pipeline workspace's counter block
    (after the fp32 unit sums, at a 256-byte boundary): the selection's
    count of finished blocks, the staged reduction's error word, the step's
    outcome, and the staged reduction's tile counter and finished-producer
    count."""
    C = -(-N // chunk)
    U = -(-chunk // 256)
    units = (C - 1) * U + -(-(N - (C - 1) * chunk) // 256)
    off = -(-units * 4 // 256) * 256
    return ws[off: off + 32].cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("name", ["googlenet", "tiny", "aligned16"])
def test_pipeline_leaves_its_counters_at_zero(name):
    """The workspace's counter block (the selection's count of finished
    blocks, the staged reduction's error word and tile counters, and the
    outcome of a step that was applied) is zero again after whole steps and
    after steps streamed per layer group: a workspace zeroed once serves
    every later step."""
    kw = SPAN_CASES.get(name)
    wl = workload.get(name) if kw is None else workload.custom(config_id=171, steps=1, **kw)
    g = dev_grads(workload.all_grads(wl, 0))
    assert fc.fc_step_reduce_kernel(g, wl.chunk) != fc.FC_REDUCE_REGISTER
    eng = _engine(wl)
    for _ in range(3):
        eng.step(g)
    torch.cuda.synchronize()
    assert not _counter_words(eng.workspace, eng.N, eng.chunk).any()
    groups = [(wl.L // 2, wl.L), (0, wl.L // 2)] if wl.L > 1 else [(0, 1)]
    eng.step_layer_groups(g, groups)
    torch.cuda.synchronize()
    assert not _counter_words(eng.workspace, eng.N, eng.chunk).any()


def _fuzz_case(i):
    """Seeded random layout: worker count, layer sizes (with tiny layers),
    chunk, keep fraction, and per-layer pointer offsets that are either the
    same for every worker (staged, shifted) or differ (register kernel)."""
    rng = np.random.default_rng(1000 + i)
    W = int(rng.choice([4, 8, 16, 4, 8, 16, 4, 8, 16, 3, 5, 32]))
    L = int(rng.integers(1, 9))
    sizes = [int(x) for x in np.exp(rng.uniform(0, np.log(60000), L)).astype(int) + 1]
    if rng.random() < 0.3:                     # a run of tiny layers
        pos = int(rng.integers(0, L + 1))
        sizes[pos:pos] = [int(x) for x in rng.integers(1, 9, int(rng.integers(2, 12)))]
    if rng.random() < 0.85:                    # N % 8 == 0, as the staged kernel needs
        sizes[-1] += (-sum(sizes)) % 8
    chunk = int(rng.choice([256, 512, 1024, 2048, 4096, 300, 777]))
    keep = int(rng.integers(1, 101))
    mode = rng.choice(["fresh", "uniform", "uniform", "skewed"])
    shifts = rng.integers(0, 8, len(sizes)) * 2
    return W, sizes, chunk, keep, str(mode), [int(x) for x in shifts]


@pytest.mark.parametrize("i", range(32))
def test_fuzzed_layouts_match_the_oracle(i):
    W, sizes, chunk, keep, mode, shifts = _fuzz_case(i)
    wl = workload.custom(W=W, sizes=sizes, chunk=chunk, keep_percent=keep,
                         config_id=300 + i, steps=2, loss_scale=256.0)

    def to_dev(g_np):
        if mode == "fresh":
            return dev_grads(g_np)
        out = []
        for w, row in enumerate(g_np):
            r = []
            for l, g in enumerate(row):
                sh = shifts[l] if mode == "uniform" else (shifts[l] + 2 * w) % 16
                buf = torch.empty(g.size + 8, dtype=torch.float16, device="cuda")
                view = buf[sh // 2: sh // 2 + g.size]
                view.copy_(torch.from_numpy(g))
                r.append(view)
            out.append(r)
        return out

    kinds = set()
    run = DeviceRun(wl, "pipeline")
    phases = DeviceRun(wl, "phases")   # the phase-1 kernel runs even where fc_step takes one launch
    st = oracle.State(workload.initial_weights(wl))
    for s in range(2):
        g_np = workload.all_grads(wl, s)
        g_dev = to_dev(g_np)
        kinds.add(fc.fc_step_reduce_kernel(g_dev, wl.chunk))
        run.step(g_dev)
        phases.step(g_dev)
        snap = run.snapshot()
        _compare_paths(snap, phases.snapshot())
        oracle_step(g_np, st, wl, snap)
    assert len(kinds) == 1


_GUARD_BYTES = 512
_GUARD_FILL = {torch.float32: (torch.int32, 0x7FA5A5A5), torch.int32: (torch.int32, 0x7FA5A5A5),
               torch.float16: (torch.int16, 0x7DA5), torch.uint8: (torch.uint8, 0xA5)}


def _guard(run):
    """Moves every device buffer of a DeviceRun into the middle of a larger
    tensor whose margins (512 bytes each side) hold a sentinel pattern;
    returns the bases and their original contents."""
    saved = []
    names = ["weights", "residual", "velocity", "a", "w16", "norms", "idx", "mask", "packed",
             "packed16", "threshold", "ws", "fused"]
    inplace_a = run.a is run.residual
    for name in names:
        t = getattr(run, name, None)
        if t is None or (name == "a" and inplace_a):
            continue
        g = _GUARD_BYTES // t.element_size()
        base = torch.empty(t.numel() + 2 * g, dtype=t.dtype, device=t.device)
        itype, pat = _GUARD_FILL[t.dtype]
        base.view(itype).fill_(pat if itype != torch.int16 else pat - 65536 * (pat > 32767))
        view = base[g: g + t.numel()]
        view.copy_(t)
        setattr(run, name, view)
        saved.append((name, base, g, t.numel(), base.clone()))
    if inplace_a:
        run.a = run.residual
    return saved


@pytest.mark.parametrize("case", [
    dict(W=16, sizes=[4096, 808, 8, 6000], chunk=256, keep_percent=25),      # aligned staged
    dict(W=16, sizes=[1001, 64, 3333, 2, 700, 5000 + 4], chunk=512, keep_percent=30),  # shifted
    dict(W=5, sizes=[1001, 64, 3333], chunk=300, keep_percent=20),            # register
    dict(W=3, sizes=[1234, 7], chunk=100, keep_percent=50),                   # N % 8 != 0
], ids=["aligned", "shifted", "register", "ragged"])
@pytest.mark.parametrize("path", ["pipeline", "phases", "separate"])
def test_no_call_writes_outside_its_buffers(case, path):
    """Guard margins around every output, state and workspace buffer stay
    bit-for-bit untouched over two steps: a memory checker's out-of-bounds
    write detection, done by the test itself."""
    wl = workload.custom(config_id=400, steps=2, **case)
    run = DeviceRun(wl, path)
    saved = _guard(run)
    st = oracle.State(workload.initial_weights(wl))
    for s in range(2):
        g_np = workload.all_grads(wl, s)
        run.step(dev_grads(g_np))
        oracle_step(g_np, st, wl, run.snapshot())
    torch.cuda.synchronize()
    for name, base, g, n, orig in saved:
        assert torch.equal(base[:g].view(torch.uint8), orig[:g].view(torch.uint8)), name + " head"
        assert torch.equal(base[g + n:].view(torch.uint8), orig[g + n:].view(torch.uint8)), name + " tail"


def test_engines_on_several_host_threads_match_sequential_runs():
    """Six host threads, each stepping its own engine on its own stream, give
    the bits of the same steps run one after another: the host-side caches
    and the thread-local tables are safe to use concurrently.  Four layouts
    are past the one-launch size (staged shifted, staged aligned, register
    and large-table), and two run as one cooperative launch each, so those
    launches from several streams also queue behind one another correctly,
    each with its own barrier words."""
    import threading
    big = 1 << 19
    cases = [dict(W=16, sizes=[big + 75001, 64, 3333, 2, 700, 5004], chunk=512, keep_percent=30),
             dict(W=8, sizes=[big, 808, 8, 6000], chunk=256, keep_percent=25),
             dict(W=5, sizes=[big + 75000, 64, 3333], chunk=300, keep_percent=20),
             dict(W=16, sizes=[13000 + 8 * i for i in range(40)], chunk=256, keep_percent=10),
             dict(W=4, sizes=[20000, 3000], chunk=256, keep_percent=10),
             dict(W=16, sizes=[1001, 64, 3333, 2, 700, 5004], chunk=512, keep_percent=30)]
    paths = [fc.FC_STEP_THREE_KERNELS] * 4 + [fc.FC_STEP_ONE_LAUNCH] * 2
    wls = [workload.custom(config_id=420 + i, steps=3, **c) for i, c in enumerate(cases)]
    grads = [[dev_grads(workload.all_grads(wl, s)) for s in range(3)] for wl in wls]
    for wl, g, path in zip(wls, grads, paths):
        assert fc.fc_step_path(g[0], wl.chunk) == path

    def run(i, engine, stream):
        with torch.cuda.stream(stream):
            for s in range(3):
                engine.step(grads[i][s], stream)
        stream.synchronize()

    seq = [_engine(wl) for wl in wls]
    for i, e in enumerate(seq):
        run(i, e, torch.cuda.Stream())
    par = [_engine(wl) for wl in wls]
    streams = [torch.cuda.Stream() for _ in wls]
    errors = []

    def worker(i):
        try:
            run(i, par[i], streams[i])
        except Exception as exc:  # reported below
            errors.append(exc)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(wls))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    for a, b in zip(seq, par):
        wa, wb = _engine_bits(a), _engine_bits(b)
        for k in wa:
            assert bits_equal(wa[k], wb[k]), k


# ---- fc_step in one launch (small problems) ------------------------------------------

ONE_LAUNCH_KINDS = {"grid": fc.FC_STEP_ONE_LAUNCH, "cluster": fc.FC_STEP_ONE_CLUSTER}


@pytest.fixture(params=list(ONE_LAUNCH_KINDS))
def one_launch_kind(request):
    """Runs the test with the cooperative (every SM) and with the cluster
    form of the one-launch step."""
    kind = ONE_LAUNCH_KINDS[request.param]
    fc.fc_test_one_launch_kind(kind)
    try:
        yield kind
    finally:
        fc.fc_test_one_launch_kind(fc.FC_STEP_ONE_LAUNCH)


ONE_LAUNCH_CASES = {
    "tiny": None,
    "w1": dict(W=1, sizes=[3000, 17], chunk=256, keep_percent=10),
    "w3_ragged": dict(W=3, sizes=[1234, 7], chunk=104, keep_percent=50),
    "w5": dict(W=5, sizes=[1001, 64, 3333, 2, 700], chunk=304, keep_percent=30),
    "w7_keep_all": dict(W=7, sizes=[5000, 33, 12000], chunk=1000, keep_percent=100),
    "w16_shifted": dict(W=16, sizes=[1001, 64, 3333, 2, 700, 5004], chunk=512, keep_percent=25),
    "w16_one_chunk": dict(W=16, sizes=[4096, 808, 8, 6000], chunk=16384, keep_percent=10),
    "w64": dict(W=64, sizes=[40000], chunk=256, keep_percent=10),
    "w8_chunk8": dict(W=8, sizes=[7000, 1], chunk=8, keep_percent=1),
    "w16_many_chunks": dict(W=16, sizes=[262144], chunk=256, keep_percent=37),
}


@pytest.mark.parametrize("inplace", [False, True], ids=["separate_a", "inplace"])
@pytest.mark.parametrize("name", list(ONE_LAUNCH_CASES))
def test_one_launch_step_matches_three_kernels_and_the_oracle(name, inplace, one_launch_kind):
    """Small problems run fc_step as one launch: cooperative over every SM,
    or one thread-block cluster.  Its results, over two steps with state
    carried, are the bits of the three pipeline kernels called one by one
    and match the oracle element by element (send buffers and fp16 weights
    included)."""
    kw = ONE_LAUNCH_CASES[name]
    wl = workload.get(name) if kw is None else workload.custom(config_id=500, steps=2, **kw)
    one = DeviceRun(wl, "pipeline", inplace=inplace)
    three = DeviceRun(wl, "phases", inplace=inplace)
    st = oracle.State(workload.initial_weights(wl))
    for s in range(2):
        g_np = workload.all_grads(wl, s)
        g = dev_grads(g_np)
        assert fc.fc_step_path(g, wl.chunk) == one_launch_kind
        one.step(g)
        three.step(g)
        a, b = one.snapshot(), three.snapshot()
        _compare_paths(a, b)
        oracle_step(g_np, st, wl, a)
        assert fc.fc_step_status(one.ws, one.N, wl.chunk) == fc.FC_OK


def test_one_launch_step_with_ties_and_misaligned_pointers(one_launch_kind):
    """All-equal norms (ties keep the lowest indices) and gradient pointers
    shifted differently per worker (the element path), in one launch."""
    wl = workload.custom(W=4, sizes=[2048, 2048], chunk=256, keep_percent=25,
                         config_id=510, steps=1)
    g_np = [[np.full(n, 0.5, np.float16) for n in wl.sizes] for _ in range(wl.W)]
    one = DeviceRun(wl, "pipeline")
    st = oracle.State(workload.initial_weights(wl))
    out = []
    for w, row in enumerate(g_np):
        r = []
        for g in row:
            buf = torch.empty(g.size + 8, dtype=torch.float16, device="cuda")
            view = buf[1 + w % 3: 1 + w % 3 + g.size]
            view.copy_(torch.from_numpy(g))
            r.append(view)
        out.append(r)
    assert fc.fc_step_path(out, wl.chunk) == one_launch_kind
    one.step(out)
    snap = one.snapshot()
    assert list(snap["idx"]) == list(range(one.k))
    oracle_step(g_np, st, wl, snap)


def test_step_path_choice():
    """The one-launch path needs chunk sizes that are multiples of 8 and a
    small problem; the rest take the three kernels."""
    small = dev_grads(workload.all_grads(workload.custom(W=4, sizes=[4096], chunk=256,
                                                          keep_percent=10, config_id=520,
                                                          steps=1), 0))
    assert fc.fc_step_path(small, 256) == fc.FC_STEP_ONE_LAUNCH
    assert fc.fc_step_path(small, 100) == fc.FC_STEP_THREE_KERNELS      # chunk % 8 != 0
    assert fc.fc_step_path(small, 12) == fc.FC_STEP_THREE_KERNELS       # chunk % 8 != 0
    assert fc.fc_step_path(small, 8) == fc.FC_STEP_ONE_LAUNCH           # 512 chunks
    big = fc.PtrTable.from_addresses([[1 << 20], [2 << 20]], [1 << 20])
    assert fc.fc_step_path(big, 4096) == fc.FC_STEP_THREE_KERNELS       # 2^20 elements
    # the cluster form, where a device runs no cooperative launch
    fc.fc_test_one_launch_kind(fc.FC_STEP_ONE_CLUSTER)
    try:
        assert fc.fc_step_path(small, 256) == fc.FC_STEP_ONE_CLUSTER
        assert fc.fc_step_path(small, 100) == fc.FC_STEP_THREE_KERNELS
    finally:
        fc.fc_test_one_launch_kind(fc.FC_STEP_ONE_LAUNCH)
    with pytest.raises(fc.FcError):
        fc.fc_test_one_launch_kind(fc.FC_STEP_THREE_KERNELS)


@pytest.mark.parametrize("inplace", [False, True], ids=["separate_a", "inplace"])
def test_one_launch_barrier_wait_runs_out(inplace):
    """Failure path of the cooperative one-launch step, without any fault:
    the test hook makes one CTA give up before the grid barrier, so every
    other CTA's wait runs out (20 ms limit).  The step reports FC_ERR_TIMEOUT
    and is not applied: velocity, weights, the fp16 weights, the send
    buffers, idx, mask and threshold keep their bits (and, with a separate
    `a` buffer, the residual).  After the workspace is zeroed again (and, in
    place, the residual restored) the same step matches the oracle."""
    wl = workload.custom(W=4, sizes=[20000, 3000], chunk=256, keep_percent=10,
                         config_id=530, steps=3)
    run = DeviceRun(wl, "pipeline", inplace=inplace)
    st = oracle.State(workload.initial_weights(wl))
    g_np = [workload.all_grads(wl, s) for s in range(2)]
    g0, g1 = dev_grads(g_np[0]), dev_grads(g_np[1])
    assert fc.fc_step_path(g0, wl.chunk) == fc.FC_STEP_ONE_LAUNCH
    run.step(g0)
    before = run.snapshot()
    oracle_step(g_np[0], st, wl, before, check_a=False)
    assert fc.fc_step_status(run.ws, run.N, wl.chunk) == fc.FC_OK
    fc.fc_test_barrier_loss(5, 20_000_000)
    run.step(g1)                                   # this one gives up
    snap = run.snapshot()
    assert fc.fc_step_status(run.ws, run.N, wl.chunk) == fc.FC_ERR_TIMEOUT
    unchanged = ["velocity", "weights", "w16", "packed", "packed16", "idx", "mask", "threshold"]
    if not inplace:
        unchanged.append("residual")
    for key in unchanged:
        assert bits_equal(snap[key], before[key]), key + " changed by a step that gave up"
    run.ws.zero_()
    if inplace:
        run.residual.copy_(torch.from_numpy(before["residual"]).cuda())
    run.step(g1)
    oracle_step(g_np[1], st, wl, run.snapshot(), check_a=False)
    assert fc.fc_step_status(run.ws, run.N, wl.chunk) == fc.FC_OK
    with pytest.raises(fc.FcError):
        fc.fc_test_barrier_loss(0, 0)
