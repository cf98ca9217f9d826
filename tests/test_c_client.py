"""The C ABI from plain C: tests/c/fc_client.c includes include/fc.h, links
libfc.so and the CUDA runtime, and runs fc_step with no Python or torch in
the process.  On the CPU the client must compile and link (-std=c99, warnings
as errors); on a GPU its results must equal the oracle's, bit for bit."""

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from gradient_aggregation_gb300 import build, workload
from tests.conftest import ROOT

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
SRC = os.path.join(ROOT, "tests", "c", "fc_client.c")


def build_client(out_dir):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(build.build_library())
    exe = os.path.join(out_dir, "fc_client")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA_HOME, "include"), SRC, "-o", exe,
           "-L", lib_dir, "-lfc", "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart",
           "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + os.path.join(CUDA_HOME, "lib64")]
    p = subprocess.run(cmd, capture_output=True, text=True)
    assert p.returncode == 0, p.stderr
    return exe


def test_c_client_compiles_and_links(fc_lib, tmp_path):
    assert os.access(build_client(str(tmp_path)), os.X_OK)


def _write_input(path, wl, steps):
    num, den = workload.keep_fraction(wl)
    with open(path, "wb") as f:
        f.write(np.array([wl.W, wl.L], np.int32).tobytes())
        f.write(np.array(wl.sizes, np.int64).tobytes())
        f.write(np.array([wl.chunk, num, den], np.int64).tobytes())
        f.write(np.array([wl.loss_scale, wl.lr, wl.momentum], np.float32).tobytes())
        f.write(np.array([steps], np.int32).tobytes())
        f.write(workload.initial_weights(wl).astype(np.float32).tobytes())
        for s in range(steps):
            for row in workload.all_grads(wl, s):
                for g in row:
                    f.write(np.ascontiguousarray(g, np.float16).tobytes())


@pytest.mark.gpu
@pytest.mark.parametrize("case", [
    None,                                                            # tiny: one launch
    dict(W=5, sizes=[1001, 64, 3333], chunk=300, keep_percent=20),   # register kernel
    dict(W=16, sizes=[1001, 64, 3333, 2, 700, 5004], chunk=512, keep_percent=30),  # one launch
    dict(W=16, sizes=[(1 << 19) + 75001, 64, 3333, 2, 700, 5004], chunk=512,
         keep_percent=30),                                          # shifted staged
    dict(W=8, sizes=[1 << 19, 808, 8, 6000], chunk=256, keep_percent=25),  # aligned staged
], ids=["tiny", "w5", "w16", "w16_shifted_staged", "w8_aligned_staged"])
def test_c_client_matches_the_oracle(fc_lib, tmp_path, case):
    wl = workload.get("tiny") if case is None else workload.custom(config_id=410, steps=2, **case)
    steps = 2
    exe = build_client(str(tmp_path))
    inp, outp = str(tmp_path / "in.bin"), str(tmp_path / "out.bin")
    _write_input(inp, wl, steps)
    p = subprocess.run([exe, inp, outp], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    raw = open(outp, "rb").read()
    k = int(np.frombuffer(raw[:8], np.int64)[0])
    pos = 8
    idx = np.frombuffer(raw[pos: pos + 4 * k], np.int32)
    pos += 4 * k
    thr = np.frombuffer(raw[pos: pos + 4], np.float32)[0]
    pos += 4
    N = wl.N
    res, vel, wts = (np.frombuffer(raw[pos + 4 * N * i: pos + 4 * N * (i + 1)], np.float32)
                     for i in range(3))
    st = oracle.State(workload.initial_weights(wl))
    num, den = workload.keep_fraction(wl)
    for s in range(steps):
        out = oracle.step(workload.all_grads(wl, s), st, wl.loss_scale, wl.chunk, num, den,
                          wl.lr, wl.momentum)
    assert np.array_equal(idx, out["idx"])
    # norms (hence the threshold) agree with the oracle's binary64 ones to rounding
    assert abs(float(thr) - float(out["threshold"])) <= 1e-6 * float(out["threshold"])
    for got, want in ((res, st.residual), (vel, st.velocity), (wts, st.weights)):
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
