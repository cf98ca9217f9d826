"""CPU oracle of the gradient-aggregation engine (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``.  The product (the CUDA library
and its Python binding) never imports this package.

The arithmetic lives in ``fc_oracle.c`` (plain C, single-threaded, compiled
with ``-ffp-contract=off``); this module only marshals numpy arrays.  Each
function cites the passage it follows in its C counterpart.

Pins: every function here is checked in ``tests/test_oracle_pins.py``
against facts fixed by the pages or by mathematics (hand-worked examples in
``tests/golden/``, an order-discriminating tree example, exact integer sums,
brute force on tiny inputs, closed forms and library routines).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fc_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liborc.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
          "-fno-strict-aliasing", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liborc.so``."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        sig = {
            "orc_half_to_float": (f32, [ctypes.c_uint16]),
            "orc_float_to_half": (ctypes.c_uint16, [f32]),
            "orc_layout": (i64, [i32, P, P]),
            "orc_fuse_pack": (None, [i32, i32, P, P, P]),
            "orc_tree_sum": (f32, [P, i32]),
            "orc_unscale_factor": (f32, [f32, i32]),
            "orc_tree_reduce": (None, [i32, i64, P, f32, P, P]),
            "orc_num_chunks": (i64, [i64, i64]),
            "orc_chunk_norms": (None, [P, i64, i64, P]),
            "orc_keep_count": (i64, [i64, i64, i64]),
            "orc_chunk_select": (None, [P, i64, i64, P, i64, i64, P, P, P, P]),
            "orc_residual_sgd_update": (None, [P, P, i64, i64, f32, f32, P, P, P, P]),
            "orc_pack_fp16": (None, [P, i64, f32, P]),
            "orc_sequential_sum": (f32, [P, i32]),
            "orc_ring_segment": (i32, [i64, i64, i32]),
            "orc_reduce_ordered": (None, [i32, i64, P, f32, P, P, i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- element conversions ------------------------------------------------

def half_to_float(bits: int) -> float:
    return float(_load().orc_half_to_float(int(bits) & 0xFFFF))


def float_to_half(x: float) -> int:
    return int(_load().orc_float_to_half(float(x)))


# ---- a1: fusion -----------------------------------------------------------

def layout(sizes: Sequence[int]):
    """(offsets, N): layers concatenated in order, no padding (GradientFlow
    abstract, lazy allreduce: many operations fused into one)."""
    s = _c(sizes, np.int64)
    off = np.zeros(max(len(s), 1), dtype=np.int64)
    n = _load().orc_layout(len(s), _ptr(s), _ptr(off))
    return off[:len(s)], int(n)


def fuse_pack(grads: List[List[np.ndarray]]) -> np.ndarray:
    """``grads[w][l]`` fp16 arrays -> fused ``[W, N]`` fp16 (bitwise copy)."""
    W, L = len(grads), len(grads[0])
    sizes = _c([g.size for g in grads[0]], np.int64)
    flat = [_c(grads[w][l], np.float16) for w in range(W) for l in range(L)]
    ptrs = (ctypes.c_void_p * (W * L))(*[f.ctypes.data for f in flat])
    N = int(sizes.sum())
    fused = np.empty((W, N), dtype=np.float16)
    _load().orc_fuse_pack(W, L, _ptr(sizes), ctypes.cast(ptrs, ctypes.c_void_p),
                          _ptr(fused))
    return fused


# ---- a2: tree reduce --------------------------------------------------------

def tree_sum(x: Sequence[float]) -> np.float32:
    """Level-order binary-tree sum of float32 values (FireCaffe §6: a
    binary reduction tree, depth the base-2 log of the worker count)."""
    a = _c(x, np.float32).copy()
    return np.float32(_load().orc_tree_sum(_ptr(a), len(a)))


def unscale_factor(loss_scale: float, W: int) -> np.float32:
    return np.float32(_load().orc_unscale_factor(float(loss_scale), int(W)))


def tree_reduce(fused: np.ndarray, loss_scale: float,
                residual: Optional[np.ndarray] = None) -> np.ndarray:
    """fused ``[W, N]`` fp16 -> a ``[N]`` fp32."""
    f = _c(fused, np.float16)
    W, N = f.shape
    r = None if residual is None else _c(residual, np.float32)
    out = np.empty(N, dtype=np.float32)
    _load().orc_tree_reduce(W, N, _ptr(f), float(loss_scale), _ptr(r), _ptr(out))
    return out


ORDER_TREE, ORDER_SEQUENTIAL, ORDER_RING = 0, 1, 2


def sequential_sum(x: Sequence[float]) -> np.float32:
    """Left-to-right fp32 sum (parameter-server order, FireCaffe §6)."""
    a = _c(x, np.float32).copy()
    return np.float32(_load().orc_sequential_sum(_ptr(a), len(a)))


def ring_segment(i: int, N: int, W: int) -> int:
    return int(_load().orc_ring_segment(int(i), int(N), int(W)))


def reduce_ordered(fused: np.ndarray, loss_scale: float,
                   residual: Optional[np.ndarray] = None, order: int = 0) -> np.ndarray:
    """a2 with a selectable summation order: 0 tree, 1 parameter server
    (sequential), 2 ring reduce-scatter (GradientFlow abstract)."""
    f = _c(fused, np.float16)
    W, N = f.shape
    r = None if residual is None else _c(residual, np.float32)
    out = np.empty(N, dtype=np.float32)
    _load().orc_reduce_ordered(W, N, _ptr(f), float(loss_scale), _ptr(r), _ptr(out),
                               int(order))
    return out


# ---- a3: norms --------------------------------------------------------------

def num_chunks(N: int, chunk: int) -> int:
    return int(_load().orc_num_chunks(int(N), int(chunk)))


def chunk_norms(a: np.ndarray, chunk: int) -> np.ndarray:
    a = _c(a, np.float32)
    C = num_chunks(a.size, chunk)
    out = np.empty(C, dtype=np.float32)
    _load().orc_chunk_norms(_ptr(a), a.size, int(chunk), _ptr(out))
    return out


# ---- a4: select -------------------------------------------------------------

def keep_count(C: int, num: int, den: int) -> int:
    return int(_load().orc_keep_count(int(C), int(num), int(den)))


def chunk_select(norms: np.ndarray, k: int, a: Optional[np.ndarray] = None,
                 chunk: int = 1, N: int = 0, want_packed: bool = True):
    """Returns (idx int32[k] ascending, mask uint8[C], packed float32[k*chunk]
    or None, threshold float32)."""
    n = _c(norms, np.float32)
    C = n.size
    idx = np.empty(k, dtype=np.int32)
    mask = np.empty(C, dtype=np.uint8)
    thr = np.zeros(1, dtype=np.float32)
    packed = None
    av = None
    if want_packed and a is not None:
        av = _c(a, np.float32)
        N = av.size
        packed = np.empty(k * chunk, dtype=np.float32)
    _load().orc_chunk_select(_ptr(n), C, int(k), _ptr(av), int(N), int(chunk),
                             _ptr(idx), _ptr(mask), _ptr(packed), _ptr(thr))
    return idx, mask, packed, np.float32(thr[0])


def pack_fp16(packed: np.ndarray, send_scale: float = 1.0) -> np.ndarray:
    """fp16 send buffer of the packed kept chunks (GradientFlow abstract:
    mixed precision): binary16(packed * send_scale), as uint16 bits."""
    p = _c(packed, np.float32)
    out = np.empty(p.size, dtype=np.uint16)
    _load().orc_pack_fp16(_ptr(p), p.size, float(send_scale), _ptr(out))
    return out


# ---- a5: update -------------------------------------------------------------

def residual_sgd_update(a: np.ndarray, mask: np.ndarray, chunk: int,
                        lr: float, momentum: float, residual: np.ndarray,
                        velocity: np.ndarray, weights: np.ndarray,
                        want_w16: bool = False):
    """Updates residual, velocity, weights in place (they must be C-contiguous
    float32 arrays); returns the fp16 weight copy (as uint16 bits) or None."""
    a = _c(a, np.float32)
    m = _c(mask, np.uint8)
    for x in (residual, velocity, weights):
        assert x.dtype == np.float32 and x.flags.c_contiguous
    w16 = np.empty(a.size, dtype=np.uint16) if want_w16 else None
    _load().orc_residual_sgd_update(_ptr(a), _ptr(m), a.size, int(chunk),
                                    float(lr), float(momentum), _ptr(residual),
                                    _ptr(velocity), _ptr(weights), _ptr(w16))
    return w16


# ---- one full step ------------------------------------------------------------

class State:
    """Engine state carried across steps: residual, velocity, weights."""

    def __init__(self, weights: np.ndarray):
        self.weights = _c(weights, np.float32).copy()
        self.residual = np.zeros_like(self.weights)
        self.velocity = np.zeros_like(self.weights)

    def copy(self) -> "State":
        s = State(self.weights)
        s.residual = self.residual.copy()
        s.velocity = self.velocity.copy()
        return s


def step(grads: List[List[np.ndarray]], state: State, loss_scale: float,
         chunk: int, keep_num: int, keep_den: int, lr: float, momentum: float,
         want_w16: bool = False, mask_override: Optional[np.ndarray] = None):
    """pack -> tree reduce (+residual) -> norms -> select -> update, in place
    on ``state``.  ``mask_override`` replaces the selection's mask in the
    update (used to follow a selection that differs only inside the
    tolerance band around the threshold).  Returns a dict of every
    intermediate."""
    fused = fuse_pack(grads)
    a = tree_reduce(fused, loss_scale, state.residual)
    norms = chunk_norms(a, chunk)
    C = norms.size
    k = keep_count(C, keep_num, keep_den)
    idx, mask, packed, thr = chunk_select(norms, k, a, chunk)
    use_mask = mask if mask_override is None else mask_override
    w16 = residual_sgd_update(a, use_mask, chunk, lr, momentum, state.residual,
                              state.velocity, state.weights, want_w16)
    return dict(fused=fused, a=a, norms=norms, k=k, idx=idx, mask=mask,
                packed=packed, threshold=thr, w16=w16)
