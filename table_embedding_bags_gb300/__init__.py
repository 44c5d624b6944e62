"""Python binding of libtbe (table-batched embedding bags on GB300).

Argument marshalling only: every step of the operator runs in the CUDA
kernels of ``libtbe.so``; this module passes device pointers, sizes and the
current CUDA stream through ctypes.  There is no CPU fallback: if the
library is missing, loading it raises.

Function names mirror the C ABI in ``include/tbe.h``.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtbe.so")

TBE_OK, TBE_ERR_INVALID_ARG, TBE_ERR_UNSUPPORTED, TBE_ERR_CUDA, TBE_ERR_WORKSPACE = 0, 1, 2, 3, 4
TBE_DEV_BAD_INDEX, TBE_DEV_BAD_OFFSETS, TBE_DEV_TIMEOUT, TBE_DEV_CAPACITY = 1, 2, 4, 8
TBE_F32, TBE_F16, TBE_BF16 = 0, 1, 2
TBE_PATH_AUTO, TBE_PATH_GATHER, TBE_PATH_HISTOGRAM = 0, 1, 2
TBE_POOL_SUM, TBE_POOL_MEAN = 0, 1
TBE_MAX_TABLES = 4096
TBE_OPT_EXACT_SGD, TBE_OPT_EXACT_ROWWISE_ADAGRAD = 0, 1

# every symbol include/tbe.h declares
EXPORTED = [
    "tbe_plan_device_bytes", "tbe_plan_create", "tbe_plan_destroy", "tbe_forward", "tbe_forward_path",
    "tbe_histogram_counts", "tbe_backward_workspace_bytes", "tbe_backward", "tbe_get_tuning",
    "tbe_set_tuning", "tbe_trace_enable", "tbe_trace_read", "tbe_status_string", "tbe_version",
    "tbe_backward_static_workspace", "tbe_exact_update", "tbe_wait_selftest", "tbe_backward_update",
    "tbe_forward_i32", "tbe_backward_i32", "tbe_backward_update_i32", "tbe_backward_index", "tbe_backward_index_i32",
    "tbe_backward_reduce",
]
TBE_STATIC_WORKSPACE_BYTES = 32 << 20


class TBEError(RuntimeError):
    pass


class _Layout(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("table_row_base", ctypes.c_void_p), ("D_offsets", ctypes.c_void_p),
                ("weights_offsets", ctypes.c_void_p), ("weights_dtype", ctypes.c_void_p),
                ("table_weighted", ctypes.c_void_p), ("out_dtype", ctypes.c_int32), ("pooling", ctypes.c_int32)]


class Tuning(ctypes.Structure):
    _fields_ = [("long_run_threshold", ctypes.c_int32), ("long_chunk", ctypes.c_int32),
                ("fwd_unroll", ctypes.c_int32), ("fwd_blocks_per_sm", ctypes.c_int32),
                ("hist_min_mean_bag", ctypes.c_int32), ("short_item_lookups", ctypes.c_int32),
                ("fwd_lanes_per_row", ctypes.c_int32), ("red_unroll", ctypes.c_int32),
                ("fwd_ring", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class Optimizer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("learning_rate", ctypes.c_float), ("eps", ctypes.c_float)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libtbe.so (no fallback: raises when the CUDA library is absent)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise TBEError(f"libtbe.so not found at {path}: build it with table_embedding_bags_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.tbe_plan_device_bytes.restype = sz
    lib.tbe_plan_device_bytes.argtypes = [i32]
    lib.tbe_plan_create.restype = ctypes.c_int
    lib.tbe_plan_create.argtypes = [ctypes.POINTER(_Layout), P, sz, P, ctypes.POINTER(P)]
    lib.tbe_plan_destroy.restype = None
    lib.tbe_plan_destroy.argtypes = [P]
    lib.tbe_forward.restype = ctypes.c_int
    lib.tbe_forward.argtypes = [P, P, P, i64, P, i32, P, P, P, P]
    lib.tbe_forward_path.restype = ctypes.c_int
    lib.tbe_forward_path.argtypes = [P, P, P, i64, P, i32, P, P, P, P, i32]
    lib.tbe_histogram_counts.restype = ctypes.c_int
    lib.tbe_histogram_counts.argtypes = [P, P, i64, P, i32, P, P, P]
    lib.tbe_backward_workspace_bytes.restype = sz
    lib.tbe_backward_workspace_bytes.argtypes = [P, i32, i64]
    lib.tbe_backward.restype = ctypes.c_int
    lib.tbe_backward.argtypes = [P, P, P, i64, P, i32, P, P, P, P, P, i64, P, P, sz, P, P]
    lib.tbe_backward_static_workspace.restype = ctypes.c_int
    lib.tbe_backward_static_workspace.argtypes = [P, P, P, i64, P, i32, P, P, P, P, P, i64, P, P, P]
    lib.tbe_exact_update.restype = ctypes.c_int
    lib.tbe_exact_update.argtypes = [P, ctypes.POINTER(Optimizer), P, P, P, i64, P, i64, P, P, P]
    lib.tbe_get_tuning.restype = ctypes.c_int
    lib.tbe_get_tuning.argtypes = [ctypes.POINTER(Tuning)]
    lib.tbe_set_tuning.restype = ctypes.c_int
    lib.tbe_set_tuning.argtypes = [ctypes.POINTER(Tuning)]
    lib.tbe_trace_enable.restype = ctypes.c_int
    lib.tbe_trace_enable.argtypes = [i32]
    lib.tbe_trace_read.restype = ctypes.c_int
    lib.tbe_trace_read.argtypes = [P, P, i32]
    lib.tbe_status_string.restype = ctypes.c_char_p
    lib.tbe_status_string.argtypes = [i32]
    lib.tbe_version.restype = ctypes.c_char_p
    lib.tbe_version.argtypes = []
    lib.tbe_forward_i32.restype = ctypes.c_int
    lib.tbe_forward_i32.argtypes = [P, P, P, i64, P, i32, P, P, P, P, i32]
    lib.tbe_backward_i32.restype = ctypes.c_int
    lib.tbe_backward_i32.argtypes = [P, P, P, i64, P, i32, P, P, P, P, P, i64, P, P, sz, P, P]
    lib.tbe_backward_update.restype = ctypes.c_int
    lib.tbe_backward_update_i32.restype = ctypes.c_int
    lib.tbe_backward_update.argtypes = [P, ctypes.POINTER(Optimizer), P, P, P, P, i64, P, i32, P, P, P, P, P, P, sz,
                                        P, P]
    lib.tbe_backward_update_i32.argtypes = lib.tbe_backward_update.argtypes
    for name in ("tbe_backward_index", "tbe_backward_index_i32"):
        getattr(lib, name).restype = ctypes.c_int
        getattr(lib, name).argtypes = [P, P, i64, P, i32, P, P, P, P, i64, P, P, sz, P, P]
    lib.tbe_backward_reduce.restype = ctypes.c_int
    lib.tbe_backward_reduce.argtypes = [P, ctypes.POINTER(Optimizer), P, P, P, i64, i32, P, P, P, P, i64, P, P, sz, P,
                                        P]
    lib.tbe_wait_selftest.restype = ctypes.c_int
    lib.tbe_wait_selftest.argtypes = [i32, i32, P, P]
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != TBE_OK:
        msg = load_library().tbe_status_string(rc).decode()
        raise TBEError(f"{what} failed: {msg} ({rc})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtypes, numel, what, optional=False):
    """Checks a tensor argument before its pointer crosses the C ABI: a
    contiguous CUDA tensor of one of ``dtypes`` with at least ``numel``
    elements (the kernels read or write that many, so a smaller or host
    buffer would be accessed out of bounds)."""
    if t is None:
        if optional:
            return
        raise TBEError(f"{what} is required")
    if t.device.type != "cuda":
        raise TBEError(f"{what} must be a CUDA tensor (got {t.device})")
    if t.dtype not in dtypes:
        raise TBEError(f"{what} has dtype {t.dtype}; expected {' or '.join(str(d) for d in dtypes)}")
    if not t.is_contiguous():
        raise TBEError(f"{what} must be contiguous")
    if t.numel() < numel:
        raise TBEError(f"{what} has {t.numel()} elements; at least {numel} are read or written")


def _is_i32(plan, indices, offsets, B, allow_i32=True):
    """Checks the id and offset arrays; True for int32 (the *_i32 entry
    points).  Both arrays must have the same width."""
    import torch

    widths = (torch.int64, torch.int32) if allow_i32 else (torch.int64,)
    _need(indices, widths, 0, "indices")
    _need(offsets, (indices.dtype,), plan.T * int(B) + 1, "offsets")
    return indices.dtype == torch.int32


def _need_weights(plan, weights):
    import torch

    _need(weights, (torch.uint8, torch.int8, torch.float32, torch.float16, torch.bfloat16), 0, "weights")
    if weights.numel() * weights.element_size() < plan.weights_bytes:
        raise TBEError(f"weights holds {weights.numel() * weights.element_size()} bytes; the plan's tables "
                       f"need {plan.weights_bytes}")


def _stream(stream=None):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _np(a, dt):
    return np.ascontiguousarray(np.asarray(a), dtype=dt)


class Plan:
    """A validated table layout with its packed metadata on the device."""

    def __init__(self, T, table_row_base, D_offsets, weights_offsets, weights_dtype, out_dtype,
                 table_weighted=None, device="cuda", stream=None, pooling=TBE_POOL_SUM):
        import torch

        lib = load_library()
        self.T = int(T)
        self.table_row_base = _np(table_row_base, np.int64)
        self.D_offsets = _np(D_offsets, np.int32)
        self.weights_offsets = _np(weights_offsets, np.int64)
        self.weights_dtype = _np(weights_dtype, np.int32)
        self.table_weighted = None if table_weighted is None else _np(table_weighted, np.uint8)
        self.out_dtype = int(out_dtype)
        self.pooling = int(pooling)
        self.sumD = int(self.D_offsets[-1])
        self.D = np.diff(self.D_offsets).astype(np.int64)
        esz = np.array([{TBE_F32: 4, TBE_F16: 2, TBE_BF16: 2}.get(int(d), 4) for d in self.weights_dtype], np.int64)
        rows = np.diff(self.table_row_base)
        self.weights_bytes = int(np.max(self.weights_offsets[:self.T] + rows * self.D * esz)) if self.T else 0
        self.total_rows = int(self.table_row_base[self.T]) if self.T else 0
        nbytes = lib.tbe_plan_device_bytes(self.T)
        if nbytes == 0:
            raise TBEError("tbe_plan_device_bytes: T out of range")
        self.dev_meta = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        L = _Layout(self.T, self.table_row_base.ctypes.data, self.D_offsets.ctypes.data,
                    self.weights_offsets.ctypes.data, self.weights_dtype.ctypes.data,
                    None if self.table_weighted is None else self.table_weighted.ctypes.data,
                    self.out_dtype, self.pooling)
        h = ctypes.c_void_p()
        with torch.cuda.device(self.dev_meta.device):
            _check(lib.tbe_plan_create(ctypes.byref(L), _ptr(self.dev_meta), nbytes, _stream(stream),
                                       ctypes.byref(h)), "tbe_plan_create")
        self._h = h

    @classmethod
    def from_problem(cls, p, device="cuda"):
        lay = p.layout_arrays()
        return cls(lay["T"], lay["table_row_base"], lay["D_offsets"], lay["weights_offsets"],
                   lay["weights_dtype"], lay["out_dtype"], lay["table_weighted"], device=device,
                   pooling=lay.get("pooling", TBE_POOL_SUM))

    @property
    def handle(self):
        return self._h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.tbe_plan_destroy(h)
            self._h = None


def _out_torch_dtype(code):
    import torch

    return {TBE_F32: torch.float32, TBE_F16: torch.float16, TBE_BF16: torch.bfloat16}[code]


def tbe_forward(plan: Plan, weights, indices, offsets, B: int, per_sample_weights=None, out=None,
                dev_status=None, path: int = TBE_PATH_AUTO, stream=None):
    """Pooled forward; returns ``out`` [B, sum D] on the device."""
    import torch

    lib = load_library()
    if out is None:
        out = torch.empty((B, plan.sumD), dtype=_out_torch_dtype(plan.out_dtype), device=indices.device)
    N = int(indices.numel())
    i32 = _is_i32(plan, indices, offsets, B)
    _need_weights(plan, weights)
    _need(per_sample_weights, (torch.float32,), N, "per_sample_weights", optional=True)
    _need(out, (_out_torch_dtype(plan.out_dtype),), int(B) * plan.sumD, "out")
    _need(dev_status, (torch.int32,), 1, "dev_status", optional=True)
    fn = lib.tbe_forward_i32 if i32 else lib.tbe_forward_path
    rc = fn(plan.handle, _ptr(weights), _ptr(indices), N, _ptr(offsets), int(B), _ptr(per_sample_weights), _ptr(out),
            _ptr(dev_status), _stream(stream), int(path))
    _check(rc, "tbe_forward")
    return out


def tbe_histogram_counts(plan: Plan, indices, offsets, B: int, counts=None, dev_status=None, stream=None):
    """Per-bag id histograms of every table: a list of int32 [B, rows_t]
    views of one buffer of B * total_rows counts (``counts`` if given).
    int64 ids and offsets only."""
    import torch

    lib = load_library()
    base = plan.table_row_base
    _is_i32(plan, indices, offsets, B, allow_i32=False)
    if counts is None:
        counts = torch.empty(int(B) * int(base[plan.T]), dtype=torch.int32, device=indices.device)
    _need(counts, (torch.int32,), int(B) * plan.total_rows, "counts")
    _need(dev_status, (torch.int32,), 1, "dev_status", optional=True)
    rc = lib.tbe_histogram_counts(plan.handle, _ptr(indices), int(indices.numel()), _ptr(offsets), int(B),
                                  _ptr(counts), _ptr(dev_status), _stream(stream))
    _check(rc, "tbe_histogram_counts")
    return [counts[int(base[t]) * B:int(base[t + 1]) * B].view(B, int(base[t + 1] - base[t])) for t in range(plan.T)]


def tbe_backward_workspace_bytes(plan: Plan, B: int, N: int) -> int:
    return int(load_library().tbe_backward_workspace_bytes(plan.handle, int(B), int(N)))


class BackwardBuffers:
    """Preallocated outputs + workspace for one (B, N) capacity
    (with_workspace=False: outputs only, for tbe_backward_static_workspace)."""

    def __init__(self, plan: Plan, B: int, N: int, device="cuda", row_grads_capacity=None, with_workspace=True):
        import torch

        self.B, self.N = int(B), int(N)
        self.workspace = None
        if with_workspace:
            ws = tbe_backward_workspace_bytes(plan, B, N)
            self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=device)
        self.unique_rows = torch.empty(max(N, 1), dtype=torch.int64, device=device)
        self.run_starts = torch.empty(N + 1, dtype=torch.int32, device=device)
        self.sorted_positions = torch.empty(max(N, 1), dtype=torch.int32, device=device)
        if row_grads_capacity is None:
            total_rows = int(plan.table_row_base[-1])
            row_grads_capacity = min(N, total_rows) * int(plan.D.max()) if N else 0
        self.row_grads = torch.empty(max(int(row_grads_capacity), 1), dtype=torch.float32, device=device)
        self.row_grads_capacity = int(row_grads_capacity)
        self.unique_count = torch.empty(plan.T + 1, dtype=torch.int64, device=device)


def _need_backward(plan, grad_out, N, B, per_sample_weights, bufs, dev_status):
    import torch

    _need(grad_out, (torch.float32,), int(B) * plan.sumD, "grad_out")
    _need(per_sample_weights, (torch.float32,), N, "per_sample_weights", optional=True)
    _need(dev_status, (torch.int32,), 1, "dev_status", optional=True)
    if bufs.N < N:
        raise TBEError(f"bufs were sized for {bufs.N} lookups; this batch has {N}")
    _need(bufs.unique_count, (torch.int64,), plan.T + 1, "bufs.unique_count")


def tbe_backward(plan: Plan, grad_out, indices, offsets, B: int, per_sample_weights=None, bufs=None,
                 dev_status=None, want_run_starts=True, want_sorted_positions=True, stream=None):
    """Row gradients.  Returns the BackwardBuffers whose leading entries hold
    the results (U = unique_count[T], read it after a synchronisation)."""
    import torch

    lib = load_library()
    N = int(indices.numel())
    i32 = _is_i32(plan, indices, offsets, B)
    if bufs is None:
        bufs = BackwardBuffers(plan, B, N, device=indices.device)
    _need_backward(plan, grad_out, N, B, per_sample_weights, bufs, dev_status)
    _need(bufs.workspace, (torch.uint8,), 1, "bufs.workspace")
    fn = lib.tbe_backward_i32 if i32 else lib.tbe_backward
    rc = fn(plan.handle, _ptr(grad_out), _ptr(indices), N, _ptr(offsets), int(B),
                          _ptr(per_sample_weights), _ptr(bufs.unique_rows),
                          _ptr(bufs.run_starts) if want_run_starts else None,
                          _ptr(bufs.sorted_positions) if want_sorted_positions else None,
                          _ptr(bufs.row_grads), bufs.row_grads_capacity, _ptr(bufs.unique_count),
                          _ptr(bufs.workspace), bufs.workspace.numel(), _ptr(dev_status), _stream(stream))
    _check(rc, "tbe_backward")
    return bufs


def tbe_backward_static_workspace(plan: Plan, grad_out, indices, offsets, B: int, per_sample_weights=None,
                                  bufs=None, dev_status=None, stream=None):
    """Row gradients using the library's built-in scratch array instead of a
    workspace (for callers that cannot allocate device memory).  ``bufs``
    supplies the outputs; its workspace is not used."""
    lib = load_library()
    N = int(indices.numel())
    _is_i32(plan, indices, offsets, B, allow_i32=False)
    if bufs is None:
        bufs = BackwardBuffers(plan, B, N, device=indices.device, with_workspace=False)
    _need_backward(plan, grad_out, N, B, per_sample_weights, bufs, dev_status)
    rc = lib.tbe_backward_static_workspace(plan.handle, _ptr(grad_out), _ptr(indices), N, _ptr(offsets), int(B),
                                           _ptr(per_sample_weights), _ptr(bufs.unique_rows), _ptr(bufs.run_starts),
                                           _ptr(bufs.sorted_positions), _ptr(bufs.row_grads),
                                           bufs.row_grads_capacity, _ptr(bufs.unique_count), _ptr(dev_status),
                                           _stream(stream))
    _check(rc, "tbe_backward_static_workspace")
    return bufs


def tbe_exact_update(plan: Plan, weights, bufs: BackwardBuffers, kind: int, learning_rate: float, eps: float = 0.0,
                     momentum=None, dev_status=None, stream=None):
    """One exact optimizer step, in place on ``weights`` (and ``momentum``
    for row-wise Adagrad), from the outputs of a tbe_backward call that
    filled ``bufs`` on the same stream."""
    import torch

    _need_weights(plan, weights)
    _need(momentum, (torch.float32,), plan.total_rows, "momentum", optional=True)
    _need(bufs.unique_count, (torch.int64,), plan.T + 1, "bufs.unique_count")
    _need(dev_status, (torch.int32,), 1, "dev_status", optional=True)
    opt = Optimizer(int(kind), float(learning_rate), float(eps))
    rc = load_library().tbe_exact_update(plan.handle, ctypes.byref(opt), _ptr(weights), _ptr(momentum),
                                         _ptr(bufs.unique_rows), bufs.N, _ptr(bufs.row_grads),
                                         bufs.row_grads_capacity, _ptr(bufs.unique_count), _ptr(dev_status),
                                         _stream(stream))
    _check(rc, "tbe_exact_update")


def tbe_backward_update(plan: Plan, weights, kind: int, learning_rate: float, grad_out, indices, offsets, B: int,
                        per_sample_weights=None, eps: float = 0.0, momentum=None, bufs=None, dev_status=None,
                        want_run_starts=True, want_sorted_positions=True, stream=None):
    """Backward with the exact optimizer fused in: updates ``weights`` (and
    ``momentum`` for row-wise Adagrad) in place; ``bufs`` receives the
    indexing outputs (its row_grads are not written)."""
    import torch

    lib = load_library()
    N = int(indices.numel())
    i32 = _is_i32(plan, indices, offsets, B)
    if bufs is None:
        bufs = BackwardBuffers(plan, B, N, device=indices.device, row_grads_capacity=0)
    _need_weights(plan, weights)
    _need(momentum, (torch.float32,), plan.total_rows, "momentum", optional=True)
    _need_backward(plan, grad_out, N, B, per_sample_weights, bufs, dev_status)
    _need(bufs.workspace, (torch.uint8,), 1, "bufs.workspace")
    opt = Optimizer(int(kind), float(learning_rate), float(eps))
    fn = lib.tbe_backward_update_i32 if i32 else lib.tbe_backward_update
    rc = fn(plan.handle, ctypes.byref(opt), _ptr(weights), _ptr(momentum), _ptr(grad_out),
                                 _ptr(indices), N, _ptr(offsets), int(B), _ptr(per_sample_weights),
                                 _ptr(bufs.unique_rows), _ptr(bufs.run_starts) if want_run_starts else None,
                                 _ptr(bufs.sorted_positions) if want_sorted_positions else None,
                                 _ptr(bufs.unique_count), _ptr(bufs.workspace), bufs.workspace.numel(),
                                 _ptr(dev_status), _stream(stream))
    _check(rc, "tbe_backward_update")
    return bufs


def tbe_backward_index(plan: Plan, indices, offsets, B: int, per_sample_weights=None, bufs=None, dev_status=None,
                       fused=False, want_run_starts=True, want_sorted_positions=True, stream=None):
    """The index stages of the backward (everything before the reduction;
    no grad_out needed).  Returns the BackwardBuffers to pass to
    tbe_backward_reduce; ``fused`` when the reduction will apply an
    optimizer (no row gradients, so no capacity check)."""
    import torch

    lib = load_library()
    N = int(indices.numel())
    i32 = _is_i32(plan, indices, offsets, B)
    if bufs is None:
        bufs = BackwardBuffers(plan, B, N, device=indices.device, row_grads_capacity=0 if fused else None)
    _need(per_sample_weights, (torch.float32,), N, "per_sample_weights", optional=True)
    _need(dev_status, (torch.int32,), 1, "dev_status", optional=True)
    if bufs.N < N:
        raise TBEError(f"bufs were sized for {bufs.N} lookups; this batch has {N}")
    _need(bufs.unique_count, (torch.int64,), plan.T + 1, "bufs.unique_count")
    _need(bufs.workspace, (torch.uint8,), 1, "bufs.workspace")
    fn = lib.tbe_backward_index_i32 if i32 else lib.tbe_backward_index
    cap = (1 << 63) - 1 if fused else bufs.row_grads_capacity
    rc = fn(plan.handle, _ptr(indices), N, _ptr(offsets), int(B), _ptr(per_sample_weights), _ptr(bufs.unique_rows),
            _ptr(bufs.run_starts) if want_run_starts else None,
            _ptr(bufs.sorted_positions) if want_sorted_positions else None, cap, _ptr(bufs.unique_count),
            _ptr(bufs.workspace), bufs.workspace.numel(), _ptr(dev_status), _stream(stream))
    _check(rc, "tbe_backward_index")
    bufs._index_call = (N, int(B), per_sample_weights is not None, want_run_starts)
    return bufs


def tbe_backward_reduce(plan: Plan, grad_out, bufs: BackwardBuffers, kind: int = -1, learning_rate: float = 0.0,
                        weights=None, eps: float = 0.0, momentum=None, per_sample_weights=None, dev_status=None,
                        stream=None):
    """The reduction after tbe_backward_index on the same ``bufs``: row
    gradients into ``bufs.row_grads`` (kind < 0), or the exact optimizer
    ``kind`` applied in place on ``weights`` (and ``momentum``)."""
    import torch

    if getattr(bufs, "_index_call", None) is None:
        raise TBEError("tbe_backward_reduce needs the BackwardBuffers of a tbe_backward_index call")
    N, B, weighted, want_run_starts = bufs._index_call
    if weighted != (per_sample_weights is not None):
        raise TBEError("per_sample_weights must be given to both calls or to neither")
    lib = load_library()
    _need_backward(plan, grad_out, N, B, per_sample_weights, bufs, dev_status)
    opt = None
    if kind >= 0:
        _need_weights(plan, weights)
        _need(momentum, (torch.float32,), plan.total_rows, "momentum", optional=True)
        opt = ctypes.byref(Optimizer(int(kind), float(learning_rate), float(eps)))
    rc = lib.tbe_backward_reduce(plan.handle, opt, _ptr(weights), _ptr(momentum), _ptr(grad_out), N, B,
                                 _ptr(per_sample_weights), _ptr(bufs.unique_rows),
                                 _ptr(bufs.run_starts) if want_run_starts else None,
                                 None if kind >= 0 else _ptr(bufs.row_grads), 0 if kind >= 0 else bufs.row_grads_capacity,
                                 _ptr(bufs.unique_count), _ptr(bufs.workspace), bufs.workspace.numel(),
                                 _ptr(dev_status), _stream(stream))
    _check(rc, "tbe_backward_reduce")
    return bufs


def get_tuning() -> dict:
    t = Tuning()
    _check(load_library().tbe_get_tuning(ctypes.byref(t)), "tbe_get_tuning")
    return t.as_dict()


def set_tuning(**kw) -> dict:
    t = Tuning()
    lib = load_library()
    _check(lib.tbe_get_tuning(ctypes.byref(t)), "tbe_get_tuning")
    for k, v in kw.items():
        setattr(t, k, int(v))
    _check(lib.tbe_set_tuning(ctypes.byref(t)), "tbe_set_tuning")
    return t.as_dict()


def trace_enable(on: bool = True):
    _check(load_library().tbe_trace_enable(1 if on else 0), "tbe_trace_enable")


def trace_read(max_stages: int = 32):
    """[(stage_name, ms), ...] of the last traced call (waits for it)."""
    ms = (ctypes.c_float * max_stages)()
    names = (ctypes.c_char_p * max_stages)()
    n = load_library().tbe_trace_read(ms, names, max_stages)
    if n < 0:
        raise TBEError(f"tbe_trace_read failed ({-n})")
    return [(names[k].decode(), float(ms[k])) for k in range(n)]


def wait_selftest(kind: int, polls: int, dev_status, stream=None):
    """Runs one of the library's bounded waits on something that never
    completes (kind 0: a look-back word, 1: an mbarrier); it gives up after
    `polls` polls and sets TBE_DEV_TIMEOUT in dev_status."""
    _check(load_library().tbe_wait_selftest(int(kind), int(polls), _ptr(dev_status), _stream(stream)),
           "tbe_wait_selftest")


def version() -> str:
    return load_library().tbe_version().decode()
