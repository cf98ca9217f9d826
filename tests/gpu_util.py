"""Helpers of the GPU parity tests: run a step through the CUDA library (the
fused pipeline or the five separate calls) and check it against the oracle.

Tolerances (the engine's stated bars): reduced gradients, residuals and
weights within 1e-5 relative (fp32), the fp16 weight copy within 1e-3
relative, the kept-chunk set exact except for chunks whose norm lies within
1e-6 relative of the threshold.  The CUDA path is designed to meet all of them
bit-exactly (same binary32 operations in the same order, no FMA), and the
tests check that stronger claim too; chunk norms differ from the oracle's
binary64 sums by rounding only and are checked to 1e-6 relative.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from gradient_aggregation_gb300 import fc, workload

RTOL_F32 = 1e-5
RTOL_F16 = 1e-3
BAND = 1e-6
RTOL_NORM = 1e-6


def dev_grads(grads_np, device="cuda"):
    return [[torch.from_numpy(g).to(device) for g in row] for row in grads_np]


class DeviceRun:
    """Device state and buffers of one engine instance for a workload."""

    def __init__(self, wl: workload.Workload, path: str = "pipeline",
                 inplace: bool = False, want_w16: bool = True,
                 want_packed: bool = True, device: str = "cuda",
                 weights: np.ndarray = None, want_packed16: bool = True,
                 send_scale: float = None):
        self.wl, self.path, self.inplace = wl, path, inplace
        N, W = wl.N, wl.W
        self.N = N
        self.C = fc.fc_num_chunks(N, wl.chunk)
        self.k = fc.fc_keep_count(self.C, *workload.keep_fraction(wl))
        w0 = workload.initial_weights(wl) if weights is None else weights
        self.weights = torch.from_numpy(np.ascontiguousarray(w0, np.float32)).to(device)
        self.residual = torch.zeros(N, dtype=torch.float32, device=device)
        self.velocity = torch.zeros(N, dtype=torch.float32, device=device)
        self.a = self.residual if inplace else torch.empty(N, dtype=torch.float32, device=device)
        self.w16 = torch.empty(N, dtype=torch.float16, device=device) if want_w16 else None
        self.norms = torch.empty(self.C, dtype=torch.float32, device=device)
        self.idx = torch.empty(self.k, dtype=torch.int32, device=device)
        self.mask = torch.empty(self.C, dtype=torch.uint8, device=device)
        self.packed = (torch.empty(self.k * wl.chunk, dtype=torch.float32, device=device)
                       if want_packed else None)
        self.packed16 = (torch.empty(self.k * wl.chunk, dtype=torch.float16, device=device)
                         if want_packed16 else None)
        self.send_scale = float(wl.loss_scale if send_scale is None else send_scale)
        self.threshold = torch.empty(1, dtype=torch.float32, device=device)
        self.ws = torch.zeros(fc.fc_step_workspace_size(N, wl.chunk), dtype=torch.uint8,
                              device=device)
        self.fused = (torch.empty(W * N, dtype=torch.float16, device=device)
                      if path == "separate" else None)
        self.offsets = None

    def step(self, grads_dev, stream=None):
        wl = self.wl
        if self.path == "pipeline":
            fc.fc_step(grads_dev, wl.loss_scale, wl.chunk, self.k, wl.lr, wl.momentum,
                       self.residual, self.a, self.velocity, self.weights, self.w16,
                       self.norms, self.idx, self.mask, self.packed, self.threshold,
                       self.ws, stream, self.packed16, self.send_scale)
        elif self.path == "phases":
            # the pipeline's three kernels called one by one (never the
            # one-launch path)
            fc.fc_step_reduce(grads_dev, wl.loss_scale, wl.chunk, self.residual, self.a,
                              self.ws, stream)
            fc.fc_step_select(self.N, wl.chunk, self.k, self.norms, self.idx, self.mask,
                              self.threshold, self.ws, stream)
            fc.fc_step_update(self.a, self.N, wl.chunk, wl.lr, wl.momentum, self.residual,
                              self.velocity, self.weights, self.w16, self.mask, self.packed,
                              self.ws, self.packed16, self.send_scale, stream)
        else:
            self.offsets = fc.fc_fuse_pack(grads_dev, self.fused, stream)
            fc.fc_tree_reduce(self.fused, wl.W, self.N, wl.loss_scale, self.residual,
                              self.a, stream)
            fc.fc_chunk_norms(self.a, self.N, wl.chunk, self.norms, stream)
            fc.fc_chunk_select(self.norms, self.C, self.k, self.a, self.N, wl.chunk,
                               self.idx, self.mask, self.packed, self.threshold,
                               self.packed16, self.send_scale, stream)
            fc.fc_residual_sgd_update(self.a, self.mask, self.N, wl.chunk, wl.lr,
                                      wl.momentum, self.residual, self.velocity,
                                      self.weights, self.w16, stream)

    def snapshot(self) -> dict:
        torch.cuda.synchronize()
        out = dict(norms=self.norms.cpu().numpy(), idx=self.idx.cpu().numpy(),
                   mask=self.mask.cpu().numpy(),
                   threshold=np.float32(self.threshold.cpu().numpy()[0]),
                   residual=self.residual.cpu().numpy(),
                   velocity=self.velocity.cpu().numpy(),
                   weights=self.weights.cpu().numpy())
        if not self.inplace:
            out["a"] = self.a.cpu().numpy()
        if self.packed is not None:
            out["packed"] = self.packed.cpu().numpy()
        if self.packed16 is not None:
            out["packed16"] = self.packed16.cpu().numpy().view(np.uint16)
            out["send_scale"] = self.send_scale
        if self.w16 is not None:
            out["w16"] = self.w16.cpu().numpy().view(np.uint16)
        if self.fused is not None:
            out["fused"] = self.fused.cpu().numpy().reshape(self.wl.W, self.N)
        return out


def bits_equal(x: np.ndarray, y: np.ndarray) -> bool:
    x = np.ascontiguousarray(x)
    y = np.ascontiguousarray(y)
    return x.shape == y.shape and np.array_equal(x.view(np.uint8), y.view(np.uint8))


def assert_close(name, got, want, rtol):
    got = got.astype(np.float64)
    want = want.astype(np.float64)
    scale = np.abs(want).max() if want.size else 0.0
    err = np.abs(got - want)
    bad = err > rtol * np.abs(want) + rtol * scale
    assert not bad.any(), "%s: %d elements off, worst %g at %d" % (
        name, int(bad.sum()), float(err.max()), int(np.argmax(err)))


def oracle_step(grads_np, st: oracle.State, wl: workload.Workload, gpu: dict,
                check_a: bool = True, pack_check: bool = True) -> dict:
    """Advance the oracle state by one step and compare the GPU snapshot of
    that step with it.  Returns a small report."""
    fused = oracle.fuse_pack(grads_np)
    if "fused" in gpu:
        assert bits_equal(gpu["fused"], fused), "fused layout differs"
    a = oracle.tree_reduce(fused, wl.loss_scale, st.residual)
    del fused
    if check_a and "a" in gpu:
        assert_close("a", gpu["a"], a, RTOL_F32)
        assert bits_equal(gpu["a"], a), "a is not bit-exact"
    norms = oracle.chunk_norms(a, wl.chunk)
    C = norms.size
    k = oracle.keep_count(C, *workload.keep_fraction(wl))
    assert gpu["idx"].size == k
    assert_close("norms", gpu["norms"], norms, RTOL_NORM)
    idx, mask, packed, thr = oracle.chunk_select(norms, k, a, wl.chunk)
    # kept set: exact outside the band around the threshold
    outside = np.abs(norms.astype(np.float64) - float(thr)) > BAND * float(thr)
    assert np.array_equal(gpu["mask"][outside], mask[outside]), "kept set differs"
    gmask = gpu["mask"]
    assert int(gmask.sum()) == k
    assert np.array_equal(gpu["idx"], np.nonzero(gmask)[0].astype(np.int32))
    assert abs(float(gpu["threshold"]) - float(thr)) <= RTOL_NORM * float(thr) + 1e-30
    same_mask = np.array_equal(gmask, mask)
    if same_mask:
        assert np.array_equal(gpu["idx"], idx)
    if pack_check and "packed" in gpu:
        exp = np.zeros(k * wl.chunk, np.float32)
        for q, c in enumerate(gpu["idx"]):
            seg = a[c * wl.chunk:(c + 1) * wl.chunk]
            exp[q * wl.chunk:q * wl.chunk + seg.size] = seg
        if same_mask:
            assert bits_equal(exp, packed)
        assert bits_equal(gpu["packed"], exp), "packed differs"
        if "packed16" in gpu:
            exp16 = oracle.pack_fp16(exp, gpu["send_scale"])
            assert_close("packed16", gpu["packed16"].view(np.float16).astype(np.float32),
                         exp16.view(np.float16).astype(np.float32), RTOL_F16)
            assert bits_equal(gpu["packed16"], exp16), "fp16 send buffer differs"
    # the update, following the GPU's kept set (identical outside the band)
    w16 = oracle.residual_sgd_update(a, gmask, wl.chunk, wl.lr, wl.momentum, st.residual,
                                     st.velocity, st.weights, want_w16="w16" in gpu)
    for name, want in (("residual", st.residual), ("velocity", st.velocity),
                       ("weights", st.weights)):
        assert_close(name, gpu[name], want, RTOL_F32)
        assert bits_equal(gpu[name], want), name + " is not bit-exact"
    if "w16" in gpu:
        assert_close("w16", gpu["w16"].view(np.float16), w16.view(np.float16), RTOL_F16)
        assert bits_equal(gpu["w16"], w16), "w16 is not bit-exact"
    return dict(same_mask=same_mask, in_band=int((~outside).sum()))
