"""Exact optimizer step (SGD, row-wise Adagrad): the CUDA update kernel after
the CUDA backward, against the oracle's backward + update (GPU).

The oracle works from the original inputs only (tables, batch, output
gradient, momentum before the step); the library's intermediate results are
never fed to it.  Tolerance per element follows the arithmetic: the row
gradient may differ from the exact sum by 1e-5 * sum|terms| (the backward's
bound); that difference is carried through the update (for Adagrad also
through the mean square, the square root and the division, each adding its
FP32 rounding); the fused multiply-add that forms w - step * g rounds once
to FP32 (half an FP32 unit in the last place), and fp16 / bf16 tables round
that once more (half a unit of their format).
"""

import numpy as np
import pytest

import oracle
import parity
from tbe_inputs import DT_BF16, DT_F16, DT_F32, make_config, make_problem

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

U32 = 2.0 ** -24  # unit roundoff of FP32


@pytest.fixture(scope="module")
def tbe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import table_embedding_bags_gb300 as m

    m.load_library()
    return m


def _rows_f64(p, w_bytes: np.ndarray, rows: np.ndarray):
    """Values of the listed global rows, decoded from a packed table buffer,
    back to back (float64)."""
    out = []
    t_of = np.searchsorted(p.table_row_base, rows, side="right") - 1
    for r, t in zip(rows, t_of):
        D, dt = int(p.D[t]), int(p.weights_dtype[t])
        eb = 4 if dt == DT_F32 else 2
        start = int(p.weights_offsets[t]) + (int(r) - int(p.table_row_base[t])) * D * eb
        raw = w_bytes[start:start + D * eb]
        if dt == DT_F32:
            out.append(raw.view(np.float32).astype(np.float64))
        elif dt == DT_F16:
            out.append(raw.view(np.float16).astype(np.float64))
        else:
            out.append((raw.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    return np.concatenate(out) if out else np.zeros(0)


def _table_dtype_per_elem(p, rows):
    t_of = np.searchsorted(p.table_row_base, rows, side="right") - 1
    return np.repeat(p.weights_dtype[t_of].astype(np.int64), p.D[t_of].astype(np.int64))


def _tolerances(kind, lr, eps, g, g_abs, widths, m0_rows, y, tdt):
    """Per-element bound on |stored - exact| and per-row bound on the momentum."""
    tg = 1e-5 * g_abs
    n = widths.size
    starts = np.concatenate([[0], np.cumsum(widths)[:-1]]).astype(np.int64)
    step = np.full(n, lr)
    dstep = np.zeros(n)
    dm = np.zeros(n)
    if kind == oracle.EXACT_ROWWISE_ADAGRAD:
        ss = np.add.reduceat(g * g, starts) if n else np.zeros(0)
        dss_data = np.add.reduceat(2 * np.abs(g) * tg + tg * tg, starts) if n else np.zeros(0)
        dss = dss_data + (widths + 2) * U32 * (ss + dss_data)
        m = m0_rows + ss / widths
        dm = dss / widths + 2 * U32 * (m + dss / widths)
        sq = np.sqrt(m)
        dsq = dm / (sq + np.sqrt(np.maximum(m - dm, 0.0))) + U32 * sq
        den = sq + eps
        dden = dsq + U32 * (den + dsq)
        step = lr / den
        # where the denominator's own uncertainty is not small against it
        # (a gradient that cancels to almost nothing on a row without
        # momentum), allow the step to be off by its whole size
        ok = den > 2 * dden
        dstep = np.where(ok, lr * dden / (den * np.where(ok, den - dden, 1.0)) + 2 * U32 * step, step)
    step_e = np.repeat(step, widths)
    dstep_e = np.repeat(dstep, widths)
    pre = step_e * tg + dstep_e * (np.abs(g) + tg)
    # the kernel's w - step * g is one fused multiply-add (one FP32 rounding),
    # then fp16 / bf16 tables round that once more to their format
    a = np.abs(y) + pre
    r32 = parity.ulp(a, DT_F32) / 2
    a = a + r32
    half = np.where(tdt == DT_F16, parity.ulp(a, DT_F16) / 2,
                    np.where(tdt == DT_BF16, parity.ulp(a, DT_BF16) / 2, 0.0))
    return pre + r32 + half, dm


def momentum_before(p, seed):
    """Seeded momentum state: uniform in [0, 2), about 30 % of rows at 0."""
    total = int(p.table_row_base[-1])
    rng = np.random.default_rng(seed)
    m0 = (rng.random(total) * 2.0).astype(np.float32)
    m0[rng.random(total) < 0.3] = 0.0
    return m0


def _step_and_check(tbe, p, kind, lr, eps, seed, row_grads_capacity=None, expect_bwd_status=0):
    w_dev, w_host = parity.weights_pair(p)
    w_before = w_host.numpy().copy()
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    m0 = momentum_before(p, seed)
    mom = torch.from_numpy(m0).cuda() if kind == tbe.TBE_OPT_EXACT_ROWWISE_ADAGRAD else None
    bufs = tbe.BackwardBuffers(plan, p.B, p.N, row_grads_capacity=row_grads_capacity)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, d["psw"], bufs=bufs, dev_status=st)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    tbe.tbe_exact_update(plan, w_dev, bufs, kind, lr, eps, momentum=mom, dev_status=st2)
    torch.cuda.synchronize()
    bwd_status, upd_status = int(st.item()), int(st2.item())
    w_after = w_dev.cpu().numpy()
    m_after = mom.cpu().numpy() if mom is not None else None
    del w_dev, d, bufs, mom
    return check_step(p, kind, lr, eps, w_before, w_after, m0, m_after, bwd_status, upd_status,
                      row_grads_capacity, expect_bwd_status)


def check_step(p, kind, lr, eps, w_before, w_after, m0, m_after, bwd_status, upd_status,
               row_grads_capacity=None, expect_bwd_status=0):
    """Compares the tables (and momentum) after one backward + update with
    the oracle's, element by element; returns the number of distinct rows."""
    TBE_DEV_CAPACITY = 8
    idx, ost, rg, rabs, pos = oracle.problem_backward(p)
    assert (bwd_status & ~TBE_DEV_CAPACITY) == expect_bwd_status
    total = int(p.table_row_base[-1])
    lr32, eps32 = float(np.float32(lr)), float(np.float32(eps))
    rows = idx["unique_rows"]
    t_of = np.searchsorted(p.table_row_base, rows, side="right") - 1
    widths = p.D[t_of].astype(np.int64)
    if row_grads_capacity is not None:  # runs whose gradient did not fit are left alone
        fits = pos + widths <= row_grads_capacity
        assert not fits.all() and (bwd_status & TBE_DEV_CAPACITY) and (upd_status & TBE_DEV_CAPACITY)
    else:
        fits = np.ones(rows.size, bool)
        assert upd_status == 0
    sel = np.nonzero(fits)[0]
    g = np.concatenate([rg[pos[k]:pos[k] + widths[k]] for k in sel]) if sel.size else np.zeros(0)
    ga = np.concatenate([rabs[pos[k]:pos[k] + widths[k]] for k in sel]) if sel.size else np.zeros(0)
    ost2, y, m_new = oracle.exact_update(p.layout_arrays(), w_before, kind, lr32, eps32, rows[sel], g,
                                         momentum=m0)
    assert ost2 == 0
    got = _rows_f64(p, w_after, rows[sel])
    tdt = _table_dtype_per_elem(p, rows[sel])
    tol, dm = _tolerances(kind, lr32, eps32, g, ga, widths[sel], m0[rows[sel]].astype(np.float64), y, tdt)
    err = np.abs(got - y)
    bad = err > tol
    if bad.any():
        k = np.nonzero(bad)[0][:8]
        raise AssertionError(f"weights mismatch ({int(bad.sum())} of {got.size}): got {got[k]} want {y[k]} "
                             f"tol {tol[k]}")
    # every other row, and every byte outside the tables' updated rows, is untouched
    untouched = np.ones(w_before.size, bool)
    for r, t in zip(rows[sel], t_of[sel]):
        D, eb = int(p.D[t]), (4 if p.weights_dtype[t] == DT_F32 else 2)
        s0 = int(p.weights_offsets[t]) + (int(r) - int(p.table_row_base[t])) * D * eb
        untouched[s0:s0 + D * eb] = False
    np.testing.assert_array_equal(w_after[untouched], w_before[untouched])
    if m_after is not None:
        np.testing.assert_array_less(np.abs(m_after[rows[sel]] - m_new), dm + 1e-30)
        keep = np.ones(total, bool)
        keep[rows[sel]] = False
        np.testing.assert_array_equal(m_after[keep], m0[keep])
    return rows.size


KINDS = [(0, "sgd", 0.05, 0.0), (1, "adagrad", 0.3, 1e-4)]


def mixed_problem(kind, weighted):
    """fp32 / fp16 / bf16 tables from one 16-byte chunk per row to column
    counts above a warp's 128, repeated rows, empty bags, ragged batch."""
    rng = np.random.default_rng(500 + 2 * kind + weighted)
    specs = [(DT_F32, 4), (DT_F32, 12), (DT_F32, 128), (DT_F32, 520), (DT_F16, 8), (DT_F16, 136),
             (DT_BF16, 64), (DT_BF16, 256), (DT_F16, 1024)]
    T, B = len(specs), 41
    rows = rng.integers(1, 400, size=T)
    lens = rng.integers(0, 60, size=(T, B))
    lens[:, 2] = 0
    lens[0, 9] = 300  # a long run on a one-chunk table
    ids = [rng.integers(0, rows[t], size=int(lens[t].sum())) for t in range(T)]
    N = int(lens.sum())
    psw = rng.random(N).astype(np.float32) if weighted else None
    tw = (np.arange(T) % 2).astype(np.uint8) if weighted else None
    D = [dd for _, dd in specs]
    G = rng.standard_normal((B, sum(D))).astype(np.float32)
    return make_problem(T, B, rows=rows, D=D, weights_dtype=[s for s, _ in specs], out_dtype=DT_F32,
                        lengths=lens, ids=ids, psw=psw, grad_out=G, table_weighted=tw, seed=77)


def bad_ids_problem():
    G = np.random.default_rng(8).standard_normal((4, 24)).astype(np.float32)
    return make_problem(2, 4, rows=[50, 60], D=[16, 8], weights_dtype=[DT_F32, DT_F16], out_dtype=DT_F32,
                        lengths=[[3, 2, 0, 1], [1, 1, 4, 0]],
                        ids=[[1, 50, 3, -2, 7, 9], [59, 60, 1, 2, -1, 99999]], grad_out=G, seed=4)


@pytest.mark.parametrize("kind,name,lr,eps", KINDS, ids=[k[1] for k in KINDS])
@pytest.mark.parametrize("weighted", [False, True])
def test_mixed_dtypes_and_widths(tbe, kind, name, lr, eps, weighted):
    assert _step_and_check(tbe, mixed_problem(kind, weighted), kind, lr, eps, seed=3) > 0


@pytest.mark.parametrize("kind,name,lr,eps", KINDS, ids=[k[1] for k in KINDS])
@pytest.mark.parametrize("cfg,B,rows_scale", [("tiny", None, 1.0), ("mixed", 300, 0.01), ("bwd_skew", 257, 0.02)])
def test_configs_reduced(tbe, kind, name, lr, eps, cfg, B, rows_scale):
    p = make_config(cfg, B=B, rows_scale=rows_scale)
    _step_and_check(tbe, p, kind, lr, eps, seed=11)


def test_mid_skewed_full_size_adagrad(tbe):
    """The workload the benchmark times, in its launch configuration."""
    p = make_config("mid_skewed")
    assert _step_and_check(tbe, p, tbe.TBE_OPT_EXACT_ROWWISE_ADAGRAD, 0.01, 1e-8, seed=5) > 50000


def test_bad_ids_skipped(tbe):
    _step_and_check(tbe, bad_ids_problem(), tbe.TBE_OPT_EXACT_ROWWISE_ADAGRAD, 0.5, 1e-3, seed=2,
                    expect_bwd_status=tbe.TBE_DEV_BAD_INDEX)


def test_capacity_shortfall_leaves_rows_alone(tbe):
    p = make_config("mixed", B=64, rows_scale=0.005)
    _step_and_check(tbe, p, tbe.TBE_OPT_EXACT_SGD, 0.1, 0.0, seed=9, row_grads_capacity=4096)


def test_empty_batch_is_a_no_op(tbe):
    p = make_problem(2, 8, rows=[5, 7], D=[8, 4], weights_dtype=[DT_F16, DT_F32], out_dtype=DT_F32,
                     lengths=np.zeros((2, 8)), ids=[[], []], grad_out=np.ones((8, 12), np.float32))
    w_dev, w_host = parity.weights_pair(p)
    plan = tbe.Plan.from_problem(p)
    d = parity.upload(p)
    bufs = tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B)
    mom = torch.ones(int(p.table_row_base[-1]), device="cuda")
    tbe.tbe_exact_update(plan, w_dev, bufs, tbe.TBE_OPT_EXACT_ROWWISE_ADAGRAD, 1.0, 0.0, momentum=mom)
    torch.cuda.synchronize()
    assert torch.equal(w_dev.cpu(), w_host) and torch.equal(mom.cpu(), torch.ones_like(mom.cpu()))


def test_host_argument_errors(tbe):
    p = make_config("tiny")
    w_dev, _ = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    bufs = tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B)
    torch.cuda.synchronize()
    with pytest.raises(tbe.TBEError):  # unknown kind
        tbe.tbe_exact_update(plan, w_dev, bufs, 7, 0.1)
    with pytest.raises(tbe.TBEError):  # Adagrad without momentum
        tbe.tbe_exact_update(plan, w_dev, bufs, tbe.TBE_OPT_EXACT_ROWWISE_ADAGRAD, 0.1, 1e-8)
    with pytest.raises(tbe.TBEError):  # negative eps
        tbe.tbe_exact_update(plan, w_dev, bufs, tbe.TBE_OPT_EXACT_SGD, 0.1, -1.0)
    with pytest.raises(tbe.TBEError):  # non-finite learning rate
        tbe.tbe_exact_update(plan, w_dev, bufs, tbe.TBE_OPT_EXACT_SGD, float("nan"))
    with pytest.raises(tbe.TBEError):  # weights not 16-byte aligned
        tbe.tbe_exact_update(plan, w_dev[4:], bufs, tbe.TBE_OPT_EXACT_SGD, 0.1)
