"""Python binding of libfc (the engine's C ABI, ``include/fc.h``).

Argument marshalling only: every function here passes raw device pointers,
sizes and the current CUDA stream to the C entry point of the same name and
raises ``FcError`` on a non-zero status.  No step of the method runs in
Python, and there is no fallback: if ``libfc.so`` has not been built, the
first call raises.  PyTorch provides device memory and streams.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import List, Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfc.so")

FC_OK = 0
FC_ERR_INVALID_ARG = -1
FC_ERR_ALIGNMENT = -2
FC_ERR_WORKSPACE = -3
FC_ERR_CUDA = -4
FC_ERR_TIMEOUT = -5
FC_ERR_LIMIT = -6
FC_MAX_TABLE_PTRS = 3072
FC_MAX_TABLE_LAYERS = 512
FC_NOALLOC_WORKSPACE_BYTES = 4 << 20
FC_ORDER_TREE, FC_ORDER_SEQUENTIAL, FC_ORDER_RING = 0, 1, 2
FC_REDUCE_REGISTER, FC_REDUCE_STAGED, FC_REDUCE_STAGED_SHIFTED = 0, 1, 2
FC_STEP_THREE_KERNELS, FC_STEP_ONE_LAUNCH, FC_STEP_ONE_CLUSTER = 0, 1, 2

_lock = threading.Lock()
_lib = None

_P, _I32, _I64, _F32, _SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                             ctypes.c_float, ctypes.c_size_t)
_SIGS = {
    "fc_last_error": (ctypes.c_char_p, []),
    "fc_version": (_I32, []),
    "fc_num_chunks": (_I64, [_I64, _I64]),
    "fc_keep_count": (_I64, [_I64, _I64, _I64]),
    "fc_layout": (ctypes.c_int, [_I32, _P, _P, _P]),
    "fc_fuse_pack": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P, _P]),
    "fc_tree_reduce": (ctypes.c_int, [_P, _I32, _I64, _F32, _P, _P, _P]),
    "fc_reduce_ordered": (ctypes.c_int, [_P, _I32, _I64, _F32, _P, _P, _I32, _P]),
    "fc_step_reduce_ordered": (ctypes.c_int, [_P, _I32, _I32, _P, _F32, _I64, _P, _P, _I32,
                                              _P, _SZ, _P]),
    "fc_step_reduce_kernel": (_I32, [_P, _I32, _I32, _P, _I64, _I32]),
    "fc_step_path": (_I32, [_P, _I32, _I32, _P, _I64]),
    "fc_step_reduce_span": (ctypes.c_int, [_P, _I32, _I32, _P, _F32, _I64, _P, _P, _I64, _I64,
                                           _P, _SZ, _P]),
    "fc_unit_start": (_I64, [_I64, _I64, _I64]),
    "fc_chunk_norms": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "fc_chunk_select": (ctypes.c_int, [_P, _I64, _I64, _P, _I64, _I64, _P, _P, _P, _P, _F32,
                                       _P, _P]),
    "fc_residual_sgd_update": (ctypes.c_int, [_P, _P, _I64, _I64, _F32, _F32, _P, _P, _P, _P, _P]),
    "fc_step_workspace_size": (_SZ, [_I64, _I64]),
    "fc_chunk_select_workspace": (_SZ, [_I64]),
    "fc_step_status": (ctypes.c_int, [_P, _SZ, _I64, _I64, _P]),
    "fc_test_stage_loss": (ctypes.c_int, [_I64, ctypes.c_uint64]),
    "fc_test_one_launch_kind": (ctypes.c_int, [_I32]),
    "fc_test_barrier_loss": (ctypes.c_int, [_I32, ctypes.c_uint64]),
    "fc_step_reduce": (ctypes.c_int, [_P, _I32, _I32, _P, _F32, _I64, _P, _P, _P, _SZ, _P]),
    "fc_step_select": (ctypes.c_int, [_I64, _I64, _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "fc_step_update": (ctypes.c_int, [_P, _I64, _I64, _F32, _F32, _P, _P, _P, _P, _P, _P, _P,
                                      _F32, _P, _SZ, _P]),
    "fc_step": (ctypes.c_int, [_P, _I32, _I32, _P, _F32, _I64, _I64, _F32, _F32, _P, _P, _P,
                               _P, _P, _P, _P, _P, _P, _P, _F32, _P, _P, _SZ, _P]),
    "fc_step_noalloc": (ctypes.c_int, [_P, _I32, _I32, _P, _F32, _I64, _I64, _F32, _F32, _P,
                                       _P, _P, _P, _P, _P, _P, _P, _P, _P, _F32, _P, _P]),
}


class FcError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("libfc status %d: %s" % (status, message))
        self.status = status


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libfc.so is not built (%s); run `python -m "
                    "gradient_aggregation_gb300.build`" % LIB_PATH)
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def _check(status: int) -> None:
    if status != FC_OK:
        raise FcError(status, lib().fc_last_error().decode())


def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _s(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return stream or None


def _i64(values: Sequence[int]):
    return (ctypes.c_int64 * len(values))(*[int(v) for v in values])


class PtrTable:
    """Host table of W*L device pointers, worker-major, plus the sizes."""

    def __init__(self, grads: List[List[torch.Tensor]]):
        self.W = len(grads)
        self.L = len(grads[0])
        sizes = [int(t.numel()) for t in grads[0]]
        for w in range(self.W):
            if len(grads[w]) != self.L:
                raise ValueError("every worker needs the same layers")
            for l in range(self.L):
                t = grads[w][l]
                if t.dtype != torch.float16 or not t.is_contiguous() or t.numel() != sizes[l]:
                    raise ValueError("gradient [%d][%d] must be contiguous fp16 of %d elements"
                                     % (w, l, sizes[l]))
        self.sizes = sizes
        self.N = sum(sizes)
        self._ptrs = (ctypes.c_void_p * (self.W * self.L))(
            *[grads[w][l].data_ptr() for w in range(self.W) for l in range(self.L)])
        self._sizes = _i64(sizes)
        self._keep = grads  # keep the tensors alive while the table is used

    @classmethod
    def from_addresses(cls, addresses: List[List[int]], sizes: Sequence[int]) -> "PtrTable":
        """A table of plain device addresses ([worker][layer]), for calls
        that only inspect the layout (fc_step_reduce_kernel)."""
        t = cls.__new__(cls)
        t.W, t.L = len(addresses), len(sizes)
        t.sizes = [int(x) for x in sizes]
        t.N = sum(t.sizes)
        t._ptrs = (ctypes.c_void_p * (t.W * t.L))(
            *[int(addresses[w][l]) for w in range(t.W) for l in range(t.L)])
        t._sizes = _i64(t.sizes)
        t._keep = None
        return t

    @property
    def ptrs(self):
        return ctypes.cast(self._ptrs, ctypes.c_void_p)

    @property
    def sizes_c(self):
        return ctypes.cast(self._sizes, ctypes.c_void_p)


def _table(grads) -> PtrTable:
    return grads if isinstance(grads, PtrTable) else PtrTable(grads)


# ---- host helpers -------------------------------------------------------------

def fc_version() -> int:
    return int(lib().fc_version())


def fc_num_chunks(N: int, chunk: int) -> int:
    return int(lib().fc_num_chunks(int(N), int(chunk)))


def fc_keep_count(C: int, keep_num: int, keep_den: int) -> int:
    return int(lib().fc_keep_count(int(C), int(keep_num), int(keep_den)))


def fc_layout(sizes: Sequence[int]) -> Tuple[List[int], int]:
    s = _i64(sizes)
    off = (ctypes.c_int64 * max(1, len(sizes)))()
    n = ctypes.c_int64(0)
    _check(lib().fc_layout(len(sizes), ctypes.cast(s, _P), ctypes.cast(off, _P),
                           ctypes.cast(ctypes.pointer(n), _P)))
    return [int(off[i]) for i in range(len(sizes))], int(n.value)


def fc_step_workspace_size(N: int, chunk: int) -> int:
    return int(lib().fc_step_workspace_size(int(N), int(chunk)))


def fc_chunk_select_workspace(C: int) -> int:
    return int(lib().fc_chunk_select_workspace(int(C)))


def fc_test_stage_loss(tile: int, wait_limit_ns: int = 20_000_000) -> None:
    """Test hook: the next TMA-staged reduction drops the copies of `tile`
    and bounds its waits by wait_limit_ns (see include/fc.h)."""
    _check(lib().fc_test_stage_loss(int(tile), int(wait_limit_ns)))


def fc_test_one_launch_kind(kind: int) -> None:
    """Test hook: FC_STEP_ONE_CLUSTER forces the cluster form of the
    one-launch step, FC_STEP_ONE_LAUNCH restores the default."""
    _check(lib().fc_test_one_launch_kind(int(kind)))


def fc_test_barrier_loss(cta: int, wait_limit_ns: int = 20_000_000) -> None:
    """Test hook: in the next cooperative one-launch step CTA `cta` skips the
    grid barrier and the others wait at most wait_limit_ns (see
    include/fc.h)."""
    _check(lib().fc_test_barrier_loss(int(cta), int(wait_limit_ns)))


# ---- the five calls ---------------------------------------------------------------

def fc_fuse_pack(grads, fused: torch.Tensor, stream=None) -> List[int]:
    t = _table(grads)
    off = (ctypes.c_int64 * t.L)()
    _check(lib().fc_fuse_pack(t.ptrs, t.W, t.L, t.sizes_c, ctypes.cast(off, _P),
                              _p(fused), _s(stream)))
    return [int(x) for x in off]


def fc_tree_reduce(fused: torch.Tensor, W: int, N: int, loss_scale: float,
                   residual_in: Optional[torch.Tensor], out: torch.Tensor,
                   stream=None) -> None:
    _check(lib().fc_tree_reduce(_p(fused), int(W), int(N), float(loss_scale),
                                _p(residual_in), _p(out), _s(stream)))


def fc_reduce_ordered(fused: torch.Tensor, W: int, N: int, loss_scale: float,
                      residual_in: Optional[torch.Tensor], out: torch.Tensor, order: int,
                      stream=None) -> None:
    _check(lib().fc_reduce_ordered(_p(fused), int(W), int(N), float(loss_scale),
                                   _p(residual_in), _p(out), int(order), _s(stream)))


def fc_chunk_norms(a: torch.Tensor, N: int, chunk: int, norms: torch.Tensor,
                   stream=None) -> None:
    _check(lib().fc_chunk_norms(_p(a), int(N), int(chunk), _p(norms), _s(stream)))


def fc_chunk_select(norms: torch.Tensor, C: int, k: int, a: Optional[torch.Tensor],
                    N: int, chunk: int, idx: torch.Tensor, mask: torch.Tensor,
                    packed: Optional[torch.Tensor], threshold: torch.Tensor,
                    packed_fp16: Optional[torch.Tensor] = None, send_scale: float = 1.0,
                    stream=None) -> None:
    _check(lib().fc_chunk_select(_p(norms), int(C), int(k), _p(a), int(N), int(chunk),
                                 _p(idx), _p(mask), _p(packed), _p(packed_fp16),
                                 float(send_scale), _p(threshold), _s(stream)))


def fc_residual_sgd_update(a: torch.Tensor, mask: torch.Tensor, N: int, chunk: int,
                           lr: float, momentum: float, residual: torch.Tensor,
                           velocity: torch.Tensor, weights: torch.Tensor,
                           weights_fp16: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    _check(lib().fc_residual_sgd_update(_p(a), _p(mask), int(N), int(chunk), float(lr),
                                        float(momentum), _p(residual), _p(velocity),
                                        _p(weights), _p(weights_fp16), _s(stream)))


# ---- the fused pipeline ---------------------------------------------------------------

def fc_step_reduce(grads, loss_scale: float, chunk: int,
                   residual: Optional[torch.Tensor], a: torch.Tensor,
                   workspace: torch.Tensor, stream=None) -> None:
    t = _table(grads)
    _check(lib().fc_step_reduce(t.ptrs, t.W, t.L, t.sizes_c, float(loss_scale), int(chunk),
                                _p(residual), _p(a), _p(workspace), workspace.numel(),
                                _s(stream)))


def fc_step_reduce_ordered(grads, loss_scale: float, chunk: int,
                           residual: Optional[torch.Tensor], a: torch.Tensor, order: int,
                           workspace: torch.Tensor, stream=None) -> None:
    t = _table(grads)
    _check(lib().fc_step_reduce_ordered(t.ptrs, t.W, t.L, t.sizes_c, float(loss_scale),
                                        int(chunk), _p(residual), _p(a), int(order),
                                        _p(workspace), workspace.numel(), _s(stream)))


def fc_step_reduce_span(grads, loss_scale: float, chunk: int,
                        residual: Optional[torch.Tensor], a: torch.Tensor, f_begin: int,
                        f_end: int, workspace: torch.Tensor, stream=None) -> None:
    t = _table(grads)
    _check(lib().fc_step_reduce_span(t.ptrs, t.W, t.L, t.sizes_c, float(loss_scale),
                                     int(chunk), _p(residual), _p(a), int(f_begin), int(f_end),
                                     _p(workspace), workspace.numel(), _s(stream)))


def fc_unit_start(N: int, chunk: int, f: int) -> int:
    return int(lib().fc_unit_start(int(N), int(chunk), int(f)))


def layer_group_spans(sizes: Sequence[int], chunk: int,
                      groups: Sequence[Tuple[int, int]]) -> List[Tuple[int, int]]:
    """Spans for fc_step_reduce_span, one per layer group [first, end) in
    the order the groups' gradients become ready.  The groups must tile the
    layers and arrive last layer first or first layer first."""
    off, N = fc_layout(sizes)
    off = off + [N]
    rng = [(off[a], off[b]) for a, b in groups]
    if not rng:
        raise ValueError("no layer groups")
    if sorted(rng) != sorted(set(rng)) or any(a > b for a, b in rng):
        raise ValueError("layer groups must be disjoint ranges")
    srt = sorted(rng)
    if srt[0][0] != 0 or srt[-1][1] != N or any(srt[i][1] != srt[i + 1][0]
                                                  for i in range(len(srt) - 1)):
        raise ValueError("layer groups must cover every layer once")
    if rng == srt:                       # first layer first
        return [(fc_unit_start(N, chunk, a), fc_unit_start(N, chunk, b)) for a, b in rng]
    if rng == srt[::-1]:                 # last layer first (backprop order)
        return list(rng)
    raise ValueError("layer groups must arrive in layer order or in reverse layer order")


def fc_step_reduce_kernel(grads, chunk: int, order: int = FC_ORDER_TREE) -> int:
    """FC_REDUCE_* of the phase-1 kernel the library picks for this layout
    (host only; `grads` is [worker][layer] tensors or a PtrTable, which
    PtrTable.from_addresses can build from plain addresses)."""
    t = _table(grads)
    r = int(lib().fc_step_reduce_kernel(t.ptrs, t.W, t.L, t.sizes_c, int(chunk), int(order)))
    if r < 0:
        _check(FC_ERR_INVALID_ARG)
    return r


def fc_step_path(grads, chunk: int) -> int:
    """FC_STEP_* of how fc_step runs this layout on the current device
    (one launch for small problems: cooperative over every SM, or one
    thread-block cluster; else three kernels)."""
    t = _table(grads)
    r = int(lib().fc_step_path(t.ptrs, t.W, t.L, t.sizes_c, int(chunk)))
    if r < 0:
        _check(FC_ERR_INVALID_ARG)
    return r


def fc_step_select(N: int, chunk: int, k: int, norms: torch.Tensor, idx: torch.Tensor,
                   mask: torch.Tensor, threshold: torch.Tensor, workspace: torch.Tensor,
                   stream=None) -> None:
    _check(lib().fc_step_select(int(N), int(chunk), int(k), _p(norms), _p(idx), _p(mask),
                                _p(threshold), _p(workspace), workspace.numel(), _s(stream)))


def fc_step_update(a: torch.Tensor, N: int, chunk: int, lr: float, momentum: float,
                   residual: torch.Tensor, velocity: torch.Tensor, weights: torch.Tensor,
                   weights_fp16: Optional[torch.Tensor], mask: torch.Tensor,
                   packed: Optional[torch.Tensor], workspace: torch.Tensor,
                   packed_fp16: Optional[torch.Tensor] = None, send_scale: float = 1.0,
                   stream=None) -> None:
    _check(lib().fc_step_update(_p(a), int(N), int(chunk), float(lr), float(momentum),
                                _p(residual), _p(velocity), _p(weights), _p(weights_fp16),
                                _p(mask), _p(packed), _p(packed_fp16), float(send_scale),
                                _p(workspace), workspace.numel(), _s(stream)))


def fc_step(grads, loss_scale: float, chunk: int, k: int, lr: float, momentum: float,
            residual: torch.Tensor, a: torch.Tensor, velocity: torch.Tensor,
            weights: torch.Tensor, weights_fp16: Optional[torch.Tensor],
            norms: torch.Tensor, idx: torch.Tensor, mask: torch.Tensor,
            packed: Optional[torch.Tensor], threshold: torch.Tensor,
            workspace: torch.Tensor, stream=None,
            packed_fp16: Optional[torch.Tensor] = None, send_scale: float = 1.0) -> None:
    t = _table(grads)
    _check(lib().fc_step(t.ptrs, t.W, t.L, t.sizes_c, float(loss_scale), int(chunk), int(k),
                         float(lr), float(momentum), _p(residual), _p(a), _p(velocity),
                         _p(weights), _p(weights_fp16), _p(norms), _p(idx), _p(mask),
                         _p(packed), _p(packed_fp16), float(send_scale), _p(threshold),
                         _p(workspace), workspace.numel(), _s(stream)))


def fc_step_status(workspace: torch.Tensor, N: int, chunk: int, stream=None) -> int:
    """Outcome of the last pipeline step on this workspace: FC_OK if it was
    applied, FC_ERR_TIMEOUT if it was not (a bounded wait ran out).
    Synchronises the stream; raises FcError only for bad arguments or a
    failed CUDA call."""
    st = int(lib().fc_step_status(_p(workspace), workspace.numel(), int(N), int(chunk),
                                  _s(stream)))
    if st not in (FC_OK, FC_ERR_TIMEOUT):
        _check(st)
    return st


def fc_step_noalloc(grads, loss_scale: float, chunk: int, k: int, lr: float,
                    momentum: float, residual: torch.Tensor, a: torch.Tensor,
                    velocity: torch.Tensor, weights: torch.Tensor,
                    weights_fp16: Optional[torch.Tensor], norms: torch.Tensor,
                    idx: torch.Tensor, mask: torch.Tensor, packed: Optional[torch.Tensor],
                    threshold: torch.Tensor, stream=None,
                    packed_fp16: Optional[torch.Tensor] = None,
                    send_scale: float = 1.0) -> None:
    """fc_step with the library's built-in scratch array instead of a
    caller workspace, for callers that cannot allocate device memory when
    they step (see include/fc.h)."""
    t = _table(grads)
    _check(lib().fc_step_noalloc(t.ptrs, t.W, t.L, t.sizes_c, float(loss_scale), int(chunk),
                                 int(k), float(lr), float(momentum), _p(residual), _p(a),
                                 _p(velocity), _p(weights), _p(weights_fp16), _p(norms),
                                 _p(idx), _p(mask), _p(packed), _p(packed_fp16),
                                 float(send_scale), _p(threshold), _s(stream)))


# ---- engine: device buffers for repeated steps ---------------------------------------

class Engine:
    """Owns the device state and scratch of repeated aggregation steps.

    State (caller-visible tensors): ``residual``, ``velocity``, ``weights``
    (fp32 [N]) and optionally ``weights_fp16``.  Per-step outputs: ``norms``
    [C], ``idx`` [k], ``mask`` [C], ``packed`` [k*chunk] and ``threshold``.
    The reduced gradient is formed in the residual buffer (in place), so
    ``a`` is not kept unless ``keep_a`` is set.
    """

    def __init__(self, sizes: Sequence[int], W: int, chunk: int, keep_num: int,
                 keep_den: int, loss_scale: float, lr: float, momentum: float,
                 weights: torch.Tensor, want_fp16: bool = False,
                 want_packed: bool = True, keep_a: bool = False,
                 want_packed_fp16: bool = False, send_scale: float = 1.0):
        dev = weights.device
        self.sizes = [int(s) for s in sizes]
        self.W = int(W)
        self.N = sum(self.sizes)
        self.chunk = int(chunk)
        self.C = fc_num_chunks(self.N, self.chunk)
        self.k = fc_keep_count(self.C, keep_num, keep_den)
        self.loss_scale, self.lr, self.momentum = float(loss_scale), float(lr), float(momentum)
        self.weights = weights.to(torch.float32).contiguous().clone()
        self.residual = torch.zeros(self.N, dtype=torch.float32, device=dev)
        self.velocity = torch.zeros(self.N, dtype=torch.float32, device=dev)
        self.a = torch.empty(self.N, dtype=torch.float32, device=dev) if keep_a else self.residual
        self.weights_fp16 = (torch.empty(self.N, dtype=torch.float16, device=dev)
                             if want_fp16 else None)
        self.norms = torch.empty(self.C, dtype=torch.float32, device=dev)
        self.idx = torch.empty(self.k, dtype=torch.int32, device=dev)
        self.mask = torch.empty(self.C, dtype=torch.uint8, device=dev)
        self.packed = (torch.empty(self.k * self.chunk, dtype=torch.float32, device=dev)
                       if want_packed else None)
        self.packed_fp16 = (torch.empty(self.k * self.chunk, dtype=torch.float16, device=dev)
                            if want_packed_fp16 else None)
        self.send_scale = float(send_scale)
        self.threshold = torch.empty(1, dtype=torch.float32, device=dev)
        # zero-filled once; the pipeline keeps its counters at zero
        self.workspace = torch.zeros(fc_step_workspace_size(self.N, self.chunk),
                                     dtype=torch.uint8, device=dev)

    def step(self, grads, stream=None) -> None:
        fc_step(grads, self.loss_scale, self.chunk, self.k, self.lr, self.momentum,
                self.residual, self.a, self.velocity, self.weights, self.weights_fp16,
                self.norms, self.idx, self.mask, self.packed, self.threshold,
                self.workspace, stream, self.packed_fp16, self.send_scale)

    def phases(self, grads, stream=None):
        """The three phases as separate calls (for per-phase timing)."""
        yield lambda: fc_step_reduce(grads, self.loss_scale, self.chunk, self.residual,
                                     self.a, self.workspace, stream)
        yield lambda: fc_step_select(self.N, self.chunk, self.k, self.norms, self.idx,
                                     self.mask, self.threshold, self.workspace, stream)
        yield lambda: fc_step_update(self.a, self.N, self.chunk, self.lr, self.momentum,
                                     self.residual, self.velocity, self.weights,
                                     self.weights_fp16, self.mask, self.packed,
                                     self.workspace, self.packed_fp16, self.send_scale,
                                     stream)

    def step_layer_groups(self, grads, groups: Sequence[Tuple[int, int]],
                          ready: Optional[Sequence[torch.cuda.Event]] = None,
                          stream=None) -> None:
        """One step with phase 1 streamed per layer group: `groups` lists
        layer ranges [first, end) in the order their gradients become ready
        (backprop: last layer first); before reducing group i the stream
        waits for ready[i], if given.  Results are the bits of step()."""
        spans = layer_group_spans(self.sizes, self.chunk, groups)
        s = stream if stream is not None else torch.cuda.current_stream()
        for i, (fb, fe) in enumerate(spans):
            if ready is not None:
                s.wait_event(ready[i])
            fc_step_reduce_span(grads, self.loss_scale, self.chunk, self.residual, self.a,
                                fb, fe, self.workspace, s)
        fc_step_select(self.N, self.chunk, self.k, self.norms, self.idx, self.mask,
                       self.threshold, self.workspace, s)
        fc_step_update(self.a, self.N, self.chunk, self.lr, self.momentum, self.residual,
                       self.velocity, self.weights, self.weights_fp16, self.mask, self.packed,
                       self.workspace, self.packed_fp16, self.send_scale, s)

    def status(self, stream=None) -> int:
        """FC_OK if the last step was applied, FC_ERR_TIMEOUT if not."""
        return fc_step_status(self.workspace, self.N, self.chunk, stream)

    def state_dict(self) -> dict:
        return {"residual": self.residual.clone(), "velocity": self.velocity.clone(),
                "weights": self.weights.clone()}

    def load_state_dict(self, sd: dict) -> None:
        self.residual.copy_(sd["residual"])
        self.velocity.copy_(sd["velocity"])
        self.weights.copy_(sd["weights"])
