"""fc_step_noalloc: the fused pipeline for callers that cannot allocate
device memory when they step (inside CUDA-graph capture, under a framework
whose pool allocator owns all device memory, or in loops that forbid
allocation after start-up).  It keeps its scratch in a fixed array built
into libfc instead of a caller workspace.

Its results must match fc_step with a caller workspace on the same inputs,
and the oracle, over two calls in a row (the second call finds the array as
the first one left it).  This file is collected last so that a failure here
does not stop the other GPU tests.
"""

import numpy as np
import pytest
import torch

import oracle
from gradient_aggregation_gb300 import fc, workload
from tests.gpu_util import DeviceRun, bits_equal, dev_grads, assert_close, oracle_step, RTOL_F32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fc_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield


def _noalloc_step(run, grads):
    wl = run.wl
    fc.fc_step_noalloc(grads, wl.loss_scale, wl.chunk, run.k, wl.lr, wl.momentum,
                       run.residual, run.a, run.velocity, run.weights, run.w16, run.norms,
                       run.idx, run.mask, run.packed, run.threshold, None,
                       run.packed16, run.send_scale)


@pytest.mark.parametrize("name", ["tiny", "custom", "shifted", "shifted_big"])
def test_noalloc_matches_workspace_pipeline_on_two_calls(name):
    if name == "tiny":                # one launch
        wl = workload.get("tiny")
    elif name == "custom":            # one launch (7 workers)
        wl = workload.custom(W=7, sizes=[5000, 33, 12000], chunk=1000, keep_percent=30,
                             config_id=170, steps=2)
    elif name == "shifted":           # one launch
        wl = workload.custom(W=16, sizes=[1001, 64, 3333, 2, 700, 5004], chunk=512,
                             keep_percent=30, config_id=171, steps=2)
    else:                             # past the one-launch size: the staged kernel's
        # shifted layout, the selection and the update kernels
        wl = workload.custom(W=16, sizes=[(1 << 19) + 75001, 64, 3333, 2, 700, 5004],
                             chunk=512, keep_percent=30, config_id=172, steps=2)
    ref = DeviceRun(wl, "pipeline")      # fc_step with a caller workspace
    new = DeviceRun(wl, "pipeline")      # same buffers, stepped by fc_step_noalloc
    st = oracle.State(workload.initial_weights(wl))
    for step in range(2):
        g_np = workload.all_grads(wl, step)
        g = dev_grads(g_np)
        ref.step(g)
        _noalloc_step(new, g)
        a, b = ref.snapshot(), new.snapshot()
        for key in ("a", "residual", "velocity", "weights", "norms", "threshold"):
            assert_close(key, b[key], a[key], RTOL_F32)
        for key in ("a", "residual", "velocity", "weights", "norms", "idx", "mask",
                    "packed", "packed16", "w16", "threshold"):
            assert bits_equal(np.asarray(a[key]), np.asarray(b[key])), (step, key)
        # and against the oracle, element by element
        oracle_step(g_np, st, wl, b)


def test_noalloc_keeps_the_callers_current_device():
    """The call runs on the device that owns its output and leaves the
    caller's current device as it found it.  With two or more GPUs visible
    the output lives on another device than the current one."""
    wl = workload.get("tiny")
    dev = 1 if torch.cuda.device_count() > 1 else 0
    torch.cuda.set_device(0)
    run = DeviceRun(wl, "pipeline", device="cuda:%d" % dev)
    g = dev_grads(workload.all_grads(wl, 0), device="cuda:%d" % dev)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream().cuda_stream
    fc.fc_step_noalloc(g, wl.loss_scale, wl.chunk, run.k, wl.lr, wl.momentum, run.residual,
                       run.a, run.velocity, run.weights, run.w16, run.norms, run.idx,
                       run.mask, run.packed, run.threshold, stream, run.packed16,
                       run.send_scale)
    assert torch.cuda.current_device() == 0
    st = oracle.State(workload.initial_weights(wl))
    with torch.cuda.device(dev):
        oracle_step(workload.all_grads(wl, 0), st, wl, run.snapshot())


def test_noalloc_rejects_problems_larger_than_its_array():
    W, N = 2, 300_000_000            # needs more than 4 MiB of scratch
    assert fc.fc_step_workspace_size(N, 256) > fc.FC_NOALLOC_WORKSPACE_BYTES
    small = torch.zeros(16, dtype=torch.float16, device="cuda")
    table = fc.PtrTable([[small], [small]])
    table._sizes[0] = N              # the size check comes before any device work
    out = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(fc.FcError) as e:
        fc.fc_step_noalloc(table, 1.0, 256, 1, 0.1, 0.9, out, out, out, out, None, out,
                           out.view(torch.int32), out.view(torch.uint8), None, out)
    assert e.value.status == fc.FC_ERR_LIMIT
    assert "built-in" in str(e.value)
