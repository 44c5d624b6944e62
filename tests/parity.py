"""Comparison helpers for GPU-vs-oracle parity tests.

Tolerances (the operator's stated accuracy, read per element):
* fp32 tables, and every backward row gradient:
      |gpu - oracle| <= 1e-5 * sum|terms|  (+ half an output ulp when the
      forward output is stored as fp16/bf16: rounding the FP32 sum to the
      output format is part of the operator)
* fp16 / bf16 tables:
      |gpu - oracle| <= max(2 * ulp_h(oracle), 1e-5 * sum|terms| + ulp_out(oracle) / 2)
  where ulp_h is the spacing of the table's half format at |oracle|
  (floored at its smallest subnormal spacing) and ulp_out the spacing of the
  output format.  The second clause covers cancellation, where FP32
  accumulation cannot promise 2 half-ulps of a result near zero; how many
  elements pass only by it is reported.
* an element whose sum of |terms| is 0 (empty bag, no valid lookups) must
  be exactly 0.
"""

from __future__ import annotations

import numpy as np

import oracle
from tbe_inputs import DT_BF16, DT_F16, DT_F32, materialize_weights

HOST_GEN_LIMIT = 1 << 30  # bytes: below this the tables are generated on the host too


def ulp(x: np.ndarray, dt: int) -> np.ndarray:
    a = np.abs(x)
    if dt == DT_F32:
        mant, emin, sub = 23, -126, 2.0 ** -149
    elif dt == DT_F16:
        mant, emin, sub = 10, -14, 2.0 ** -24
    else:
        mant, emin, sub = 7, -126, 2.0 ** -133
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.where(a >= 2.0 ** emin, 2.0 ** (e - mant), sub)


def tolerance(ref, abs_sum, table_dt, out_dt):
    """Per-element bound; the stored output adds at most half an output ulp
    (taken at the largest magnitude the FP32 sum can have)."""
    fp = 1e-5 * abs_sum
    store = ulp(np.abs(ref) + fp, out_dt) / 2 if out_dt != DT_F32 else 0.0
    if table_dt == DT_F32:
        return fp + store, np.zeros(ref.shape, bool)
    half = 2 * ulp(ref, table_dt)
    alt = fp + ulp(np.abs(ref) + fp, out_dt) / 2
    return np.maximum(half, alt), alt > half


def weights_pair(p, device="cuda"):
    """(device buffer, host buffer) of the packed tables, both from the generator."""
    import torch

    if p.weights_bytes <= HOST_GEN_LIMIT:
        w_host = materialize_weights(p, device="cpu")
        return w_host.to(device), w_host
    w_dev = materialize_weights(p, device=device)
    torch.cuda.synchronize()
    return w_dev, w_dev.cpu()


def to_f64(out):
    import torch

    return out.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def compare_forward(p, got: np.ndarray, ref: np.ndarray, ref_abs: np.ndarray, cols=None):
    """Element-wise check of a forward output.  ``cols`` maps each column of
    ``got`` to its table (defaults to the full [B, sumD] layout).  Returns
    the number of elements that passed only through the cancellation clause."""
    doff = p.D_offsets
    if cols is None:
        cols = np.repeat(np.arange(p.T), np.diff(doff))
    tdt = p.weights_dtype[cols]
    only_second = 0
    for dt in np.unique(tdt):
        m = np.broadcast_to(tdt == dt, got.shape)
        g, r, a = got[m], ref[m], ref_abs[m]
        tol, alt = tolerance(r, a, int(dt), p.out_dtype)
        err = np.abs(g - r)
        zero = a == 0
        bad = (err > tol) | (zero & (g != 0))
        if bad.any():
            k = np.nonzero(bad)[0][:10]
            raise AssertionError(f"forward mismatch ({int(bad.sum())} of {g.size}, table dtype {dt}): "
                                 f"got {g[k]} want {r[k]} tol {tol[k]} abs {a[k]}")
        only_second += int(np.sum(alt & (err > 2 * ulp(r, int(dt))) & ~zero))
    return only_second


def compare_rowgrads(got: np.ndarray, ref: np.ndarray, ref_abs: np.ndarray):
    tol = 1e-5 * ref_abs
    err = np.abs(got - ref)
    bad = (err > tol) | ((ref_abs == 0) & (got != 0))
    if bad.any():
        k = np.nonzero(bad)[0][:10]
        raise AssertionError(f"row_grads mismatch ({int(bad.sum())} of {got.size}): got {got[k]} "
                             f"want {ref[k]} tol {tol[k]}")


def upload(p, device="cuda"):
    import torch

    d = dict(indices=torch.from_numpy(p.indices).to(device), offsets=torch.from_numpy(p.offsets).to(device))
    d["psw"] = None if p.per_sample_weights is None else torch.from_numpy(p.per_sample_weights).to(device)
    d["grad"] = None if p.grad_out is None else torch.from_numpy(p.grad_out).to(device)
    return d
