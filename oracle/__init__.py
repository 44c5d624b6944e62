"""Oracle for table-batched embedding bags (TEST INFRASTRUCTURE ONLY).

A plain CPU statement of the operator (``tbe_oracle.c``, fp64 accumulation)
plus a thin ctypes wrapper.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package; the CUDA library and
its Python binding never do.

Functions take host numpy arrays in the packed-table layout described on
the page "FBTriton table-batched embeddings: the backward win is a threshold
moved from 32 to 256", section "A lookup table that is most of the model".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tbe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libtbe_oracle.so")

BAD_INDEX, BAD_OFFSETS, BAD_ARG = 1, 2, 4
F32, F16, BF16 = 0, 1, 2

_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc (IEEE double, no contraction into FMA)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-o", out, src, "-lm", *extra_flags]
    subprocess.check_call(cmd)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


def load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is None:
        if _lib is not None:
            return _lib
        if _needs_build():
            build()
        path = _LIB
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    lib.orc_decode_f16.restype = ctypes.c_double
    lib.orc_decode_f16.argtypes = [ctypes.c_uint16]
    lib.orc_decode_bf16.restype = ctypes.c_double
    lib.orc_decode_bf16.argtypes = [ctypes.c_uint16]
    lib.orc_encode_f16.restype = ctypes.c_uint16
    lib.orc_encode_f16.argtypes = [ctypes.c_double]
    lib.orc_encode_bf16.restype = ctypes.c_uint16
    lib.orc_encode_bf16.argtypes = [ctypes.c_double]
    lib.orc_round.restype = None
    lib.orc_round.argtypes = [P, i64, i32, P]
    lib.orc_check_offsets.restype = ctypes.c_int
    lib.orc_check_offsets.argtypes = [i32, i32, P, i64]
    lib.orc_forward.restype = ctypes.c_int
    lib.orc_forward.argtypes = [i32, i32, P, P, P, P, P, P, P, i64, P, P, P, i64, P, P, P, i32]
    lib.orc_histogram_counts.restype = ctypes.c_int
    lib.orc_histogram_counts.argtypes = [i32, i32, i32, i64, P, i64, P, P]
    lib.orc_counts_times_table.restype = None
    lib.orc_counts_times_table.argtypes = [i32, i64, i32, P, P, i64, i32, P]
    lib.orc_scale_by_bag_length.restype = None
    lib.orc_scale_by_bag_length.argtypes = [i32, i32, P, P, P]
    lib.orc_backward_indexing.restype = ctypes.c_int
    lib.orc_backward_indexing.argtypes = [i32, i32, P, P, i64, P, P, P, P, P, P]
    lib.orc_backward_values.restype = ctypes.c_int
    lib.orc_backward_values.argtypes = [i32, i32, P, P, P, P, i64, P, P, P, P, P, P, i64, P, P, P, i32]
    lib.orc_exact_update.restype = ctypes.c_int
    lib.orc_exact_update.argtypes = [i32, P, P, P, P, P, i32, ctypes.c_double, ctypes.c_double, P, i64, P, P,
                                     P, P, P]
    if path == _LIB:
        _lib = lib
    return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return None if a is None else np.ascontiguousarray(a, dtype=dt)


def _weights_np(weights):
    if hasattr(weights, "numpy"):  # torch tensor on the host
        weights = weights.numpy()
    return np.ascontiguousarray(weights, dtype=np.uint8)


# ----------------------------------------------------------------------------
# public helpers
# ----------------------------------------------------------------------------

def decode(bits, dtype: int, lib=None) -> np.ndarray:
    lib = lib or load()
    f = lib.orc_decode_f16 if dtype == F16 else lib.orc_decode_bf16
    return np.array([f(int(b)) for b in np.asarray(bits).ravel()], np.float64)


def round_to(x: np.ndarray, dtype: int, lib=None) -> np.ndarray:
    """Round fp64 values once (nearest-even) to fp32 / fp16 / bf16.

    Returns float32 values for fp32 and uint16 bit patterns otherwise."""
    lib = lib or load()
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.shape, np.float32 if dtype == F32 else np.uint16)
    lib.orc_round(_p(x), x.size, dtype, _p(out))
    return out


def forward(layout: dict, weights, indices, offsets, B: int, per_sample_weights=None,
            bags=None, nthreads: int = 0, lib=None):
    """Pooled sums.  Returns (status, out_sum, out_abs).

    With ``bags=None`` the outputs are [B, sum D] float64 arrays; otherwise a
    list of global bag ids g = t*B + b and flat outputs holding each listed
    bag's D_t values back to back (plus the start of each)."""
    lib = lib or load()
    T = int(layout["T"])
    trb = _c(layout["table_row_base"], np.int64)
    doff = _c(layout["D_offsets"], np.int32)
    woff = _c(layout["weights_offsets"], np.int64)
    wdt = _c(layout["weights_dtype"], np.int32)
    tw = _c(layout.get("table_weighted"), np.uint8)
    w = _weights_np(weights)
    ind = _c(indices, np.int64)
    off = _c(offsets, np.int64)
    psw = _c(per_sample_weights, np.float32)
    sumD = int(doff[T])
    D = np.diff(doff).astype(np.int64)
    if bags is None:
        bb, tt = np.meshgrid(np.arange(B, dtype=np.int64), np.arange(T, dtype=np.int64), indexing="ij")
        g = (tt * B + bb).ravel()
        pos = (bb * sumD + doff[tt].astype(np.int64)).ravel()
        n_out = B * sumD
    else:
        g = np.ascontiguousarray(bags, np.int64)
        widths = D[g // max(B, 1)] if g.size else np.zeros(0, np.int64)
        pos = np.concatenate([[0], np.cumsum(widths)[:-1]]).astype(np.int64) if g.size else np.zeros(0, np.int64)
        n_out = int(widths.sum())
    s = np.zeros(max(n_out, 1), np.float64)
    a = np.zeros(max(n_out, 1), np.float64)
    st = lib.orc_forward(T, B, _p(trb), _p(doff), _p(woff), _p(wdt), _p(tw), _p(w), _p(ind),
                         ind.shape[0], _p(off), _p(psw), _p(g), g.shape[0], _p(pos), _p(s), _p(a),
                         nthreads)
    s, a = s[:n_out], a[:n_out]
    mean = int(layout.get("pooling", POOL_SUM)) == POOL_MEAN
    if bags is None:
        s, a = s.reshape(B, sumD), a.reshape(B, sumD)
        if mean:
            s, a = scale_by_bag_length(T, B, doff, off, s, lib), scale_by_bag_length(T, B, doff, off, a, lib)
        return st, s, a
    if mean:  # scale each listed bag's block by its length
        lens = (off[g + 1] - off[g]).astype(np.float64)
        for k in range(g.size):
            if lens[k] > 0:
                w_k = int(D[g[k] // max(B, 1)])
                s[pos[k]:pos[k] + w_k] /= lens[k]
                a[pos[k]:pos[k] + w_k] /= lens[k]
    return st, s, a, pos


POOL_SUM, POOL_MEAN = 0, 1


def scale_by_bag_length(T, B, D_offsets, offsets, values, lib=None):
    """Mean pooling: each bag's block of a [B, sum D] float64 array divided by
    the bag's number of lookups (orc_scale_by_bag_length); returns a copy."""
    lib = lib or load()
    v = np.array(values, dtype=np.float64, order="C", copy=True)
    lib.orc_scale_by_bag_length(int(T), int(B), _p(_c(D_offsets, np.int32)), _p(_c(offsets, np.int64)), _p(v))
    return v


def histogram_counts(T, B, t, rows_t, indices, offsets, lib=None):
    lib = lib or load()
    ind = _c(indices, np.int64)
    off = _c(offsets, np.int64)
    cnt = np.zeros((B, rows_t), np.int32)
    st = lib.orc_histogram_counts(T, B, t, rows_t, _p(ind), ind.shape[0], _p(off), _p(cnt))
    return st, cnt


def counts_times_table(counts, weights, w_off, dtype, D, lib=None):
    lib = lib or load()
    cnt = _c(counts, np.int32)
    B, R = cnt.shape
    w = _weights_np(weights)
    out = np.zeros((B, D), np.float64)
    lib.orc_counts_times_table(B, R, D, _p(cnt), _p(w), int(w_off), int(dtype), _p(out))
    return out


def backward_indexing(layout: dict, indices, offsets, B: int, lib=None):
    """Returns dict(status, sorted_pos[N], unique_rows[U], run_starts[U+1], unique_count[T+1])."""
    lib = lib or load()
    T = int(layout["T"])
    trb = _c(layout["table_row_base"], np.int64)
    ind = _c(indices, np.int64)
    off = _c(offsets, np.int64)
    N = ind.shape[0]
    sp = np.zeros(max(N, 1), np.int32)
    ur = np.zeros(max(N, 1), np.int64)
    rs = np.zeros(N + 1, np.int32)
    uc = np.zeros(T + 1, np.int64)
    nu = np.zeros(1, np.int64)
    st = lib.orc_backward_indexing(T, B, _p(trb), _p(ind), N, _p(off), _p(sp), _p(ur), _p(rs),
                                   _p(uc), _p(nu))
    U = int(nu[0])
    return dict(status=st, sorted_pos=sp[:N], unique_rows=ur[:U], run_starts=rs[:U + 1],
                unique_count=uc, U=U)


def backward_values(layout: dict, offsets, B: int, grad_out, idx: dict, per_sample_weights=None,
                    runs=None, nthreads: int = 0, lib=None):
    """Row gradients of the listed runs (all runs if None).

    Returns (status, rg_sum, rg_abs, rg_pos): flat float64 arrays holding run
    k's D_t values at rg_pos[k].  With runs=None the flat layout is the
    table-major row-gradient layout (run after run, D_t floats each)."""
    lib = lib or load()
    T = int(layout["T"])
    trb = _c(layout["table_row_base"], np.int64)
    doff = _c(layout["D_offsets"], np.int32)
    tw = _c(layout.get("table_weighted"), np.uint8)
    off = _c(offsets, np.int64)
    psw = _c(per_sample_weights, np.float32)
    G = _c(np.asarray(grad_out, np.float32), np.float64)  # fp32 gradients, exactly in double
    if int(layout.get("pooling", POOL_SUM)) == POOL_MEAN:  # the mean's backward: the sum's on G / L
        G = scale_by_bag_length(T, B, doff, off, G, lib)
    ur = _c(idx["unique_rows"], np.int64)
    rs = _c(idx["run_starts"], np.int32)
    sp = _c(idx["sorted_pos"], np.int32)
    U = ur.shape[0]
    runs = np.arange(U, dtype=np.int64) if runs is None else _c(runs, np.int64)
    D = np.diff(doff).astype(np.int64)
    t_of = np.searchsorted(trb, ur, side="right") - 1 if U else np.zeros(0, np.int64)
    widths = D[t_of[runs]] if runs.size else np.zeros(0, np.int64)
    pos = np.concatenate([[0], np.cumsum(widths)[:-1]]).astype(np.int64) if runs.size else np.zeros(0, np.int64)
    n = int(widths.sum())
    s = np.zeros(max(n, 1), np.float64)
    a = np.zeros(max(n, 1), np.float64)
    N = int(off[-1]) if off.size else 0
    st = lib.orc_backward_values(T, B, _p(trb), _p(doff), _p(tw), _p(off), N, _p(psw), _p(G),
                                 _p(ur), _p(rs), _p(sp), _p(runs), runs.shape[0], _p(pos), _p(s),
                                 _p(a), nthreads)
    return st, s[:n], a[:n], pos


EXACT_SGD, EXACT_ROWWISE_ADAGRAD = 0, 1


def exact_update(layout: dict, weights, kind: int, lr: float, eps: float, rows, grads, g_pos=None,
                 momentum=None, lib=None):
    """One exact optimizer step on finished row gradients.

    ``rows``: global rows; ``grads``: flat float64 values, row k's D_t values
    at ``g_pos[k]`` (default: back to back in the order listed);
    ``momentum``: fp32 [total_rows] state before the step (Adagrad only).
    Returns (status, w_new, m_new): the updated weights in double, unrounded,
    at the same flat positions as ``grads``, and the new momentum of each
    listed row (zeros for SGD)."""
    lib = lib or load()
    T = int(layout["T"])
    trb = _c(layout["table_row_base"], np.int64)
    doff = _c(layout["D_offsets"], np.int32)
    woff = _c(layout["weights_offsets"], np.int64)
    wdt = _c(layout["weights_dtype"], np.int32)
    w = _weights_np(weights)
    r = _c(rows, np.int64)
    g = _c(grads, np.float64)
    if g_pos is None:
        D = np.diff(doff).astype(np.int64)
        t_of = np.searchsorted(trb, r, side="right") - 1 if r.size else np.zeros(0, np.int64)
        widths = D[np.clip(t_of, 0, T - 1)] if r.size else np.zeros(0, np.int64)
        g_pos = np.concatenate([[0], np.cumsum(widths)[:-1]]) if r.size else np.zeros(0, np.int64)
    gp = _c(g_pos, np.int64)
    m = _c(momentum, np.float32)
    if kind == EXACT_ROWWISE_ADAGRAD and m is None:
        raise ValueError("row-wise Adagrad needs the momentum state")
    w_new = np.zeros(max(g.size, 1), np.float64)
    m_new = np.zeros(max(r.size, 1), np.float64)
    st = lib.orc_exact_update(T, _p(trb), _p(doff), _p(woff), _p(wdt), _p(w), int(kind), float(lr), float(eps),
                              _p(m), r.size, _p(r), _p(g), _p(gp), _p(w_new), _p(m_new))
    return st, w_new[:g.size], m_new[:r.size]


def problem_forward(p, weights_host, bags=None, nthreads=0, lib=None):
    """Convenience: forward of a tbe_inputs.TBEProblem."""
    return forward(p.layout_arrays(), weights_host, p.indices, p.offsets, p.B,
                   p.per_sample_weights, bags=bags, nthreads=nthreads, lib=lib)


def problem_backward(p, runs=None, nthreads=0, lib=None):
    """Convenience: indexing + row gradients of a tbe_inputs.TBEProblem."""
    lay = p.layout_arrays()
    idx = backward_indexing(lay, p.indices, p.offsets, p.B, lib=lib)
    st, s, a, pos = backward_values(lay, p.offsets, p.B, p.grad_out, idx, p.per_sample_weights,
                                    runs=runs, nthreads=nthreads, lib=lib)
    return idx, st, s, a, pos


if __name__ == "__main__":  # pragma: no cover
    print(build(), file=sys.stderr)
