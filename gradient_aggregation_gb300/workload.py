"""Seeded synthetic workloads for the gradient-aggregation engine.

This module only draws inputs: layer sizes, per-worker fp16 gradients and the
initial fp32 master weights.  It holds none of the method's arithmetic (no
offsets, sums, norms, selection or update), so that both the CUDA path and
the CPU oracle can consume the very same arrays without sharing any code of
the method.  numpy's PCG64 generator and its float32 normal sampler are
stable across platforms, so x86 and Arm hosts draw identical bits.

The five workloads follow the shapes the pages' systems were evaluated on:
FireCaffe (arXiv 1511.00175) trains Network-in-Network and GoogLeNet (§7) and
discusses AlexNet's large fully-connected layers (§5); GradientFlow
(arXiv 1902.06855, abstract) trains AlexNet with mixed precision and
chunk-sparse communication.  ImageNet-trained gradients are not needed (and
not present): Gaussian fp16 gradients with the stated loss scales stand in.

Seeds: worker ``w``'s gradients at step ``s`` of workload ``i`` come from
``numpy.random.default_rng(1000*i + 17*s + w)``; layer sizes from
``default_rng(1000*i + 999)``; initial weights ``N(0, 0.05)`` from
``default_rng(1000*i + 998)``; the heavy-tailed per-chunk scales of the stress
workload from ``default_rng(1000*i + 17*s + 997)``.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    config_id: int
    W: int                      # simulated workers
    sizes: tuple                # per-layer element counts, in layer order
    grad_std: float             # std of the unscaled gradient
    loss_scale: float           # S: gradients are stored as fp16(g * S)
    chunk: int                  # chunk size in elements
    keep_percent: int           # top fraction of chunks kept, in percent
    momentum: float
    lr: float
    steps: int                  # steps the parity tests carry state over
    heavy_tail: bool = False    # per-chunk log-normal magnitude (sigma = 2)

    @property
    def N(self) -> int:
        return int(sum(self.sizes))

    @property
    def L(self) -> int:
        return len(self.sizes)


def _rescaled_log_uniform(rng: np.random.Generator, lo: Sequence[float],
                          hi: Sequence[float], total: int) -> List[int]:
    """Sizes drawn log-uniform in [lo_j, hi_j], then scaled so they sum to
    ``total``: each scaled size is floored (at least 1) and the remainder is
    added to the largest tensor."""
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    raw = np.exp(rng.uniform(np.log(lo), np.log(hi)))
    scaled = np.maximum(1, np.floor(raw * (total / raw.sum()))).astype(np.int64)
    big = int(np.argmax(scaled))
    scaled[big] += total - int(scaled.sum())
    assert scaled.sum() == total and scaled.min() >= 1
    return [int(x) for x in scaled]


# AlexNet: conv1..conv5, fc6..fc8, each weight followed by its bias (ungrouped
# convolutions, as the shapes are listed).
_ALEXNET_SHAPES = [
    (96, 3, 11, 11), (96,), (256, 96, 5, 5), (256,), (384, 256, 3, 3), (384,),
    (384, 384, 3, 3), (384,), (256, 384, 3, 3), (256,), (4096, 9216), (4096,),
    (4096, 4096), (4096,), (1000, 4096), (1000,),
]


def _nin_sizes() -> List[int]:
    rng = np.random.default_rng(1000 * 1 + 999)
    # 12 conv weights in [96, 2^20], each followed by its bias in [96, 1024].
    lo, hi = [], []
    for _ in range(12):
        lo += [96.0, 96.0]
        hi += [1048576.0, 1024.0]
    return _rescaled_log_uniform(rng, lo, hi, 7_600_000)


def _googlenet_sizes() -> List[int]:
    rng = np.random.default_rng(1000 * 2 + 999)
    return _rescaled_log_uniform(rng, [64.0] * 57, [1048576.0] * 57, 6_998_552)


def _build_workloads() -> dict:
    w = {}
    w["tiny"] = Workload("tiny", 0, 4, (1728, 131072, 256), 0.01, 1024.0,
                         256, 10, 0.9, 0.01, 2)
    w["nin"] = Workload("nin", 1, 8, tuple(_nin_sizes()), 1e-3, 128.0,
                        4096, 100, 0.9, 0.01, 1)
    w["googlenet"] = Workload("googlenet", 2, 16, tuple(_googlenet_sizes()),
                              1e-3, 1024.0, 4096, 25, 0.9, 0.01, 3)
    w["alexnet"] = Workload("alexnet", 3, 16,
                            tuple(int(np.prod(s)) for s in _ALEXNET_SHAPES),
                            1e-3, 512.0, 32768, 1, 0.9, 0.01, 1)
    w["stress"] = Workload("stress", 4, 64, (16_777_216,), 1e-3, 1024.0,
                           4096, 10, 0.9, 0.01, 5, heavy_tail=True)
    return w


WORKLOADS = _build_workloads()


def get(name: str) -> Workload:
    return WORKLOADS[name]


def custom(W: int, sizes: Sequence[int], chunk: int, keep_percent: int = 10,
           loss_scale: float = 1024.0, grad_std: float = 0.01,
           momentum: float = 0.9, lr: float = 0.01, config_id: int = 90,
           heavy_tail: bool = False, steps: int = 1) -> Workload:
    """A small workload of arbitrary shape for edge-case tests."""
    return Workload("custom", config_id, int(W), tuple(int(s) for s in sizes),
                    grad_std, float(loss_scale), int(chunk), int(keep_percent),
                    momentum, lr, steps, heavy_tail)


def _chunk_scales(wl: Workload, step: int) -> np.ndarray:
    """Per-chunk magnitude multipliers exp(2 z), z ~ N(0, 1), one per chunk of
    the concatenated gradient, shared by all workers at a given step."""
    nchunks = -(-wl.N // wl.chunk)
    rng = np.random.default_rng(1000 * wl.config_id + 17 * step + 997)
    return np.exp(2.0 * rng.standard_normal(nchunks)).astype(np.float32)


def worker_grads(wl: Workload, step: int, worker: int) -> List[np.ndarray]:
    """Worker ``worker``'s fp16 gradient tensors at ``step``, one flat array
    per layer, already multiplied by the loss scale (values saturate at the
    fp16 maximum 65504)."""
    rng = np.random.default_rng(1000 * wl.config_id + 17 * step + worker)
    mul = np.float32(wl.grad_std * wl.loss_scale)
    scales = None
    if wl.heavy_tail:
        # element e of the concatenation lies in chunk e // chunk
        scales = np.repeat(_chunk_scales(wl, step), wl.chunk)[:wl.N]
    out = []
    pos = 0
    for n in wl.sizes:
        z = rng.standard_normal(n, dtype=np.float32)
        z *= mul
        if scales is not None:
            z *= scales[pos:pos + n]
        np.clip(z, -65504.0, 65504.0, out=z)
        out.append(z.astype(np.float16))
        pos += n
    return out


def all_grads(wl: Workload, step: int, threads: Optional[int] = None
              ) -> List[List[np.ndarray]]:
    """``[worker][layer]`` fp16 arrays for one step.  Workers are drawn on a
    thread pool; each has its own generator, so the bits do not depend on the
    number of threads."""
    import concurrent.futures as cf
    import os
    n = threads or min(wl.W, os.cpu_count() or 1, 16)
    if n <= 1 or wl.N * wl.W < (1 << 22):
        return [worker_grads(wl, step, w) for w in range(wl.W)]
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        return list(ex.map(lambda w: worker_grads(wl, step, w), range(wl.W)))


def initial_weights(wl: Workload) -> np.ndarray:
    """fp32 master weights over the concatenated parameter vector."""
    rng = np.random.default_rng(1000 * wl.config_id + 998)
    return (rng.standard_normal(wl.N, dtype=np.float32) * np.float32(0.05))


def keep_fraction(wl: Workload) -> tuple:
    """The kept fraction as a rational (numerator, denominator)."""
    return (wl.keep_percent, 100)
