"""The C ABI without a GPU: the library builds and loads, exports every entry
point that include/fc.h declares, computes the host-side layout and counts,
and rejects bad arguments with a status before touching any device."""

import ctypes
import os
import re

import pytest

from tests.conftest import ROOT, read_golden

HEADER = os.path.join(ROOT, "include", "fc.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"FC_API\s+[\w\s\*]+?\b(fc_\w+)\s*\(", text)))


def test_header_declares_the_five_calls_and_the_pipeline():
    names = declared_functions()
    for n in ["fc_fuse_pack", "fc_tree_reduce", "fc_chunk_norms", "fc_chunk_select",
              "fc_residual_sgd_update", "fc_step", "fc_step_reduce", "fc_step_select",
              "fc_step_update", "fc_step_workspace_size", "fc_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(fc_lib):
    for name in declared_functions():
        assert hasattr(fc_lib, name), name


def test_num_chunks_and_keep_counts(fc_lib):
    from gradient_aggregation_gb300 import fc
    for name, N, cs, C, p, k, last in read_golden("workload_counts.txt"):
        assert fc.fc_num_chunks(int(N), int(cs)) == int(C)
        assert fc.fc_keep_count(int(C), int(p), 100) == int(k)
    assert fc.fc_num_chunks(0, 4) == 0
    assert fc.fc_num_chunks(5, 0) == -1
    assert fc.fc_keep_count(10, 0, 100) == 1
    assert fc.fc_keep_count(10, 250, 100) == 10
    assert fc.fc_keep_count(0, 1, 1) == -1
    # no overflow of C * keep_num for a large denominator: ceil(4096 * 10^17 / 10^18) = 410
    assert fc.fc_keep_count(4096, 10 ** 17, 10 ** 18) == 410


def test_layout_matches_hand_worked_offsets(fc_lib):
    from gradient_aggregation_gb300 import fc
    rows = read_golden("alexnet_offsets.txt")
    sizes = [int(r[1]) for r in rows[:-1]]
    off, n = fc.fc_layout(sizes)
    assert off == [int(r[2]) for r in rows[:-1]]
    assert n == int(rows[-1][1])
    assert fc.fc_layout([0, 3, 0, 2]) == ([0, 0, 3, 3], 5)


def _status(fn, *args):
    return int(fn(*args))


def test_argument_errors_return_before_any_device_work(fc_lib):
    from gradient_aggregation_gb300 import fc
    L = fc_lib
    P = ctypes.c_void_p
    fake = 0x10000          # never dereferenced: every case fails validation
    odd = 0x10002           # 2-byte aligned only

    def grads(n, p=fake):
        arr = (ctypes.c_void_p * n)(*([p] * n))
        return ctypes.cast(arr, P), arr

    sizes = (ctypes.c_int64 * 2)(8, 8)
    g, keep = grads(4)
    # fuse pack
    assert L.fc_fuse_pack(None, 2, 2, ctypes.cast(sizes, P), None, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_fuse_pack(g, 0, 2, ctypes.cast(sizes, P), None, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_fuse_pack(g, 2, 2, ctypes.cast(sizes, P), None, None, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_fuse_pack(g, 2, 2, ctypes.cast(sizes, P), None, odd, None) == fc.FC_ERR_ALIGNMENT
    gm, keep2 = grads(4, 0x10001)
    assert L.fc_fuse_pack(gm, 2, 2, ctypes.cast(sizes, P), None, fake, None) == fc.FC_ERR_ALIGNMENT
    big = 1600
    gb, keep3 = grads(big * 2)
    sizes2 = (ctypes.c_int64 * 2)(8, 8)
    assert L.fc_fuse_pack(gb, big, 2, ctypes.cast(sizes2, P), None, fake, None) == fc.FC_ERR_LIMIT
    assert b"FC_MAX_TABLE_PTRS" in L.fc_last_error()
    neg = (ctypes.c_int64 * 2)(8, -1)
    assert L.fc_fuse_pack(g, 2, 2, ctypes.cast(neg, P), None, fake, None) == fc.FC_ERR_INVALID_ARG
    # tree reduce
    assert L.fc_tree_reduce(fake, 0, 10, 1.0, None, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_tree_reduce(fake, 2, 0, 1.0, None, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_tree_reduce(fake, 2, 10, 0.0, None, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_tree_reduce(fake, 2, 10, float("inf"), None, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_tree_reduce(fake, 2, 10, 1.0, None, fake + 4, None) == fc.FC_ERR_ALIGNMENT
    assert L.fc_tree_reduce(fake + 1, 2, 10, 1.0, None, fake, None) == fc.FC_ERR_ALIGNMENT
    # norms
    assert L.fc_chunk_norms(fake, 10, 0, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_chunk_norms(fake + 8, 10, 4, fake, None) == fc.FC_ERR_ALIGNMENT
    # select
    assert L.fc_chunk_select(fake, 4, 5, None, 0, 0, fake, fake, None, None, 1.0, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_chunk_select(fake, 4, 0, None, 0, 0, fake, fake, None, None, 1.0, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_chunk_select(fake, 4, 2, None, 0, 0, None, fake, None, None, 1.0, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_chunk_select(fake, 4, 2, fake, 100, 10, fake, fake, fake, None, 1.0, fake, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_chunk_select(fake, 4, 2, fake, 40, 10, fake, fake, None, fake + 8, 1.0, fake, None) == fc.FC_ERR_ALIGNMENT
    assert L.fc_chunk_select(fake, 4, 2, fake, 40, 10, fake, fake, None, fake, float("inf"), fake, None) == fc.FC_ERR_INVALID_ARG
    # update
    assert L.fc_residual_sgd_update(fake, fake, 10, 0, 0.1, 0.9, fake, fake, fake, None, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_residual_sgd_update(fake, None, 10, 2, 0.1, 0.9, fake, fake, fake, None, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_residual_sgd_update(fake, fake, 10, 2, float("nan"), 0.9, fake, fake, fake, None, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_residual_sgd_update(fake, fake, 10, 2, 0.1, 0.9, fake, fake + 4, fake, None, None) == fc.FC_ERR_ALIGNMENT
    # pipeline workspace
    ws = fc.fc_step_workspace_size(1000, 64)
    assert ws > 0 and ws % 256 == 0
    assert fc.fc_step_workspace_size(0, 64) == 0
    assert L.fc_step_reduce(g, 2, 2, ctypes.cast(sizes, P), 1.0, 4, None, fake, None, 0, None) == fc.FC_ERR_WORKSPACE
    assert L.fc_step_reduce(g, 2, 2, ctypes.cast(sizes, P), 1.0, 4, None, fake, fake, 1, None) == fc.FC_ERR_WORKSPACE
    assert L.fc_step_reduce(g, 2, 2, ctypes.cast(sizes, P), 1.0, 4, None, fake, fake + 16, 10 ** 6, None) == fc.FC_ERR_ALIGNMENT
    assert L.fc_step_reduce(g, 2, 2, ctypes.cast(sizes, P), 1.0, 4, None, None, fake, 10 ** 6, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_step_select(16, 4, 9, fake, fake, fake, fake, fake, 10 ** 6, None) == fc.FC_ERR_INVALID_ARG
    assert L.fc_step_update(fake, 16, 4, 0.1, 0.9, fake, fake, fake, None, fake, fake + 4, None, 1.0, fake, 10 ** 6, None) == fc.FC_ERR_ALIGNMENT
    assert L.fc_step(g, 2, 2, ctypes.cast(sizes, P), 1.0, 4, 5, 0.1, 0.9, fake, fake, fake, fake,
                     None, fake, fake, fake, None, None, 1.0, fake, fake, 10 ** 6, None) == fc.FC_ERR_INVALID_ARG
    assert b"k = 5" in L.fc_last_error()


def test_status_codes_match_the_header(fc_lib):
    """The binding's status constants are the header's enum values, with the
    timeout status at -5 and the capacity limit at -6."""
    from gradient_aggregation_gb300 import fc
    text = open(HEADER).read()
    enum = dict((m.group(1), int(m.group(2)))
                for m in re.finditer(r"\b(FC_(?:OK|ERR_\w+))\s*=\s*(-?\d+)", text))
    assert enum == {"FC_OK": 0, "FC_ERR_INVALID_ARG": -1, "FC_ERR_ALIGNMENT": -2,
                    "FC_ERR_WORKSPACE": -3, "FC_ERR_CUDA": -4, "FC_ERR_TIMEOUT": -5,
                    "FC_ERR_LIMIT": -6}
    for name, value in enum.items():
        assert getattr(fc, name) == value, name
    assert fc.fc_version() == 200


def test_select_needs_no_workspace(fc_lib):
    from gradient_aggregation_gb300 import fc
    for C in (1, 520, 4096, 11264, 11265, 1 << 30):
        assert fc.fc_chunk_select_workspace(C) == 0


def test_noalloc_and_status_check_every_argument_before_device_work(fc_lib):
    """fc_step_noalloc validates every argument (the same checks as fc_step)
    before it looks up its scratch array or queues the clearing of it, so an
    invalid call returns a status here, with no GPU in the process."""
    from gradient_aggregation_gb300 import fc
    L = fc_lib
    P = ctypes.c_void_p
    fake = 0x10000
    arr = (ctypes.c_void_p * 4)(*([fake] * 4))
    g = ctypes.cast(arr, P)
    sizes = (ctypes.c_int64 * 2)(8, 8)

    def noalloc(k=1, loss_scale=1.0, residual=fake, idx=fake, packed=None, send_scale=1.0,
                chunk=4, W=2):
        return L.fc_step_noalloc(g, W, 2, ctypes.cast(sizes, P), loss_scale, chunk, k, 0.1,
                                 0.9, residual, fake, fake, fake, None, fake, idx, fake, packed,
                                 None, send_scale, fake, None)
    assert noalloc(k=5) == fc.FC_ERR_INVALID_ARG and b"k = 5" in L.fc_last_error()
    assert noalloc(loss_scale=0.0) == fc.FC_ERR_INVALID_ARG
    assert noalloc(residual=fake + 4) == fc.FC_ERR_ALIGNMENT
    assert noalloc(idx=None) == fc.FC_ERR_INVALID_ARG
    assert noalloc(packed=fake + 8) == fc.FC_ERR_ALIGNMENT
    assert noalloc(send_scale=float("nan")) == fc.FC_ERR_INVALID_ARG
    assert noalloc(chunk=0) == fc.FC_ERR_INVALID_ARG
    assert noalloc(W=0) == fc.FC_ERR_INVALID_ARG
    # the same checks in fc_step, before its workspace is looked at
    assert L.fc_step(g, 2, 2, ctypes.cast(sizes, P), 0.0, 4, 1, 0.1, 0.9, fake, fake, fake,
                     fake, None, fake, fake, fake, None, None, 1.0, fake, None, 0,
                     None) == fc.FC_ERR_INVALID_ARG
    # fc_step_status checks its workspace before reading it
    assert L.fc_step_status(None, 10 ** 6, 16, 4, None) == fc.FC_ERR_WORKSPACE
    assert L.fc_step_status(fake, 1, 16, 4, None) == fc.FC_ERR_WORKSPACE
    assert L.fc_step_status(fake + 16, 10 ** 6, 16, 4, None) == fc.FC_ERR_ALIGNMENT
    assert L.fc_step_status(fake, 10 ** 6, 0, 4, None) == fc.FC_ERR_INVALID_ARG


def test_python_binding_raises_with_message(fc_lib):
    from gradient_aggregation_gb300 import fc
    with pytest.raises(fc.FcError) as e:
        fc._check(fc_lib.fc_tree_reduce(0x10000, 0, 10, 1.0, None, 0x10000, None))
    assert e.value.status == fc.FC_ERR_INVALID_ARG and "W = 0" in str(e.value)


def test_reduce_kernel_choice_from_layout(fc_lib):
    """fc_step_reduce_kernel inspects addresses only: fake ones will do."""
    from gradient_aggregation_gb300 import fc
    T = fc.PtrTable.from_addresses

    def separate(W, sizes, skew=lambda w, l: 0):
        return T([[((1 + w * len(sizes) + l) << 20) + skew(w, l) for l in range(len(sizes))]
                  for w in range(W)], sizes)

    def bucket(W, sizes):
        off, n = fc.fc_layout(sizes)
        return T([[((1 + w) << 32) + 2 * o for o in off] for w in range(W)], sizes)

    even, odd = [4096, 800, 8], [1001, 64, 3333, 2]       # N = 4904, 4400
    k = fc.fc_step_reduce_kernel
    assert k(separate(16, even), 256) == fc.FC_REDUCE_STAGED
    # aligned but long (at least 8192 tiles of 2048): the shifted variant
    assert k(separate(16, [8192 * 2048]), 256) == fc.FC_REDUCE_STAGED_SHIFTED
    assert k(separate(16, [8191 * 2048]), 256) == fc.FC_REDUCE_REGISTER
    # mid-size aligned runs stream faster in the register kernel
    assert k(separate(16, [1536 * 2048]), 256) == fc.FC_REDUCE_REGISTER
    assert k(separate(16, [1535 * 2048]), 256) == fc.FC_REDUCE_STAGED
    assert k(separate(8, [1000, 3000 * 2048 - 1000]), 256) == fc.FC_REDUCE_REGISTER
    # shifted layouts stay staged at any length
    assert k(separate(16, [3001, 3000 * 2048 - 3001]), 256) == fc.FC_REDUCE_STAGED_SHIFTED
    assert k(separate(8, odd), 512) == fc.FC_REDUCE_STAGED_SHIFTED
    assert k(separate(4, odd), 256) == fc.FC_REDUCE_STAGED_SHIFTED
    # a bucket per worker is one aligned segment, whatever the layer sizes
    assert k(bucket(16, odd), 256) == fc.FC_REDUCE_STAGED
    # every worker 2 bytes past a 16-byte boundary: one shift for all
    assert k(separate(16, even, lambda w, l: 2), 256) == fc.FC_REDUCE_STAGED_SHIFTED
    # one worker shifted differently from the others: register kernel
    assert k(separate(16, even, lambda w, l: 2 if (w, l) == (3, 1) else 0), 256) == \
        fc.FC_REDUCE_REGISTER
    # worker counts, orders, chunk sizes and N the staged kernel does not serve
    assert k(separate(32, even), 256) == fc.FC_REDUCE_REGISTER
    assert k(separate(32, odd), 256) == fc.FC_REDUCE_REGISTER
    assert k(separate(64, [8192 * 2048]), 256) == fc.FC_REDUCE_REGISTER
    assert k(separate(24, odd), 256) == fc.FC_REDUCE_REGISTER
    assert k(separate(2, even), 256) == fc.FC_REDUCE_REGISTER
    assert k(separate(8, even), 256, fc.FC_ORDER_SEQUENTIAL) == fc.FC_REDUCE_REGISTER
    assert k(separate(8, even), 256, fc.FC_ORDER_RING) == fc.FC_REDUCE_REGISTER
    assert k(separate(8, even), 300) == fc.FC_REDUCE_REGISTER
    assert k(separate(8, [1001, 64, 3333]), 256) == fc.FC_REDUCE_REGISTER   # N % 8 != 0
    with pytest.raises(fc.FcError):
        k(separate(8, even), 256, 7)
    with pytest.raises(fc.FcError):
        k(separate(8, even), 0)
    with pytest.raises(fc.FcError):
        k(separate(8, even, lambda w, l: 1), 256)                          # odd address


def _unit_starts(N, chunk):
    """Unit starts by their definition: each chunk cut into 256-element units."""
    starts = []
    for c0 in range(0, N, chunk):
        starts.extend(range(c0, min(c0 + chunk, N), 256))
    return starts


def test_unit_start_matches_the_unit_definition(fc_lib):
    from gradient_aggregation_gb300 import fc
    for N, chunk in [(1, 1), (1000, 64), (5000, 300), (70000, 32768), (4096, 4096), (9999, 256)]:
        starts = _unit_starts(N, chunk)
        for f in range(0, N, max(1, N // 997)):
            assert fc.fc_unit_start(N, chunk, f) == max(x for x in starts if x <= f)
        assert fc.fc_unit_start(N, chunk, N) == N
    assert fc.fc_unit_start(10, 4, 11) == -1
    assert fc.fc_unit_start(10, 0, 1) == -1
    assert fc.fc_unit_start(10, 4, -1) == -1


def test_layer_group_spans_own_every_unit_once_when_ready(fc_lib):
    """The spans of a layer grouping give every unit to exactly one call, and
    only once every layer the unit touches has arrived."""
    from gradient_aggregation_gb300 import fc
    sizes = [1001, 64, 3333, 2, 700, 5000]
    off, N = fc.fc_layout(sizes)
    off = off + [N]
    groupings = [[(4, 6), (2, 4), (0, 2)], [(0, 1), (1, 5), (5, 6)], [(0, 6)],
                 [(5, 6), (4, 5), (3, 4), (2, 3), (1, 2), (0, 1)],
                 [(0, 1), (1, 2), (2, 3), (3, 4), (4, 5), (5, 6)]]
    for chunk in (256, 300, 1024, 20000):
        starts = _unit_starts(N, chunk)
        for groups in groupings:
            spans = fc.layer_group_spans(sizes, chunk, groups)
            owned = [[x for x in starts if a <= x < b] for a, b in spans]
            assert sorted(sum(owned, [])) == starts
            ready = []
            for (ga, gb), own in zip(groups, owned):
                ready.append((off[ga], off[gb]))
                for x in own:
                    last = min(x + 256, (x // chunk + 1) * chunk, N) - 1
                    for f in (x, last):
                        assert any(a <= f < b for a, b in ready), (chunk, groups, x)
    with pytest.raises(ValueError):
        fc.layer_group_spans(sizes, 256, [(0, 3), (2, 6)])            # overlap
    with pytest.raises(ValueError):
        fc.layer_group_spans(sizes, 256, [(0, 3)])                    # missing layers
    with pytest.raises(ValueError):
        fc.layer_group_spans(sizes, 256, [(2, 4), (0, 2), (4, 6)])    # neither order


def test_span_arguments_are_checked_before_device_work(fc_lib):
    from gradient_aggregation_gb300 import fc
    P = ctypes.c_void_p
    fake = 0x10000
    arr = (ctypes.c_void_p * 4)(*([fake] * 4))
    g = ctypes.cast(arr, P)
    sizes = (ctypes.c_int64 * 2)(8, 8)
    sp = lambda b, e: int(fc_lib.fc_step_reduce_span(g, 2, 2, ctypes.cast(sizes, P), 1.0, 4, None,
                                                     fake, b, e, fake, 10 ** 6, None))
    assert sp(-1, 4) == fc.FC_ERR_INVALID_ARG
    assert sp(5, 4) == fc.FC_ERR_INVALID_ARG
    assert sp(0, 17) == fc.FC_ERR_INVALID_ARG and b"span" in fc_lib.fc_last_error()
