"""32-bit ids and offsets (tbe_forward_i32, tbe_backward_i32) (GPU).

The int32 entry points read the same values through half-width arrays, so
every output must be bit-identical to the int64 entry points': the pooled
forward output of every gather kernel and of the histogram path, and all
backward outputs (distinct rows, run starts, sorted positions, per-table
counts, row gradients).  The int64 results are themselves checked against
the oracle by the other GPU tests.
"""

import numpy as np
import pytest

import parity
from tbe_inputs import DT_F32, make_config, make_problem

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tbe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import table_embedding_bags_gb300 as m

    m.load_library()
    return m


@pytest.fixture
def tuned(tbe):
    old = tbe.get_tuning()
    yield tbe.set_tuning
    tbe.set_tuning(**old)


def _both_widths(p):
    d = parity.upload(p)
    d32 = dict(d, indices=d["indices"].to(torch.int32), offsets=d["offsets"].to(torch.int32))
    return d, d32


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


CONFIGS = [("tiny", None, 1.0), ("mid_skewed", None, 1.0), ("mixed", 300, 0.01), ("small_table", 500, 1.0),
           ("bwd_skew", 301, 0.02)]


@pytest.mark.parametrize("name,B,rows_scale", CONFIGS)
@pytest.mark.parametrize("mode", [3, 2, 1, 0], ids=["auto", "stream", "ring", "registers"])
def test_forward_matches_int64(tbe, tuned, name, B, rows_scale, mode):
    tuned(fwd_ring=mode)
    p = make_config(name, B=B, rows_scale=rows_scale)
    w_dev, _ = parity.weights_pair(p)
    d, d32 = _both_widths(p)
    plan = tbe.Plan.from_problem(p)
    paths = [tbe.TBE_PATH_GATHER] + ([tbe.TBE_PATH_HISTOGRAM] if name == "small_table" else [])
    for path in paths:
        st, st32 = (torch.zeros(1, dtype=torch.int32, device="cuda") for _ in range(2))
        a = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, d["psw"], dev_status=st, path=path)
        b = tbe.tbe_forward(plan, w_dev, d32["indices"], d32["offsets"], p.B, d32["psw"], dev_status=st32, path=path)
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and int(st32.item()) == 0
        assert torch.equal(_bits(a), _bits(b)), f"path {path}"


@pytest.mark.parametrize("name,B,rows_scale", CONFIGS)
def test_backward_matches_int64(tbe, name, B, rows_scale):
    p = make_config(name, B=B, rows_scale=rows_scale)
    d, d32 = _both_widths(p)
    plan = tbe.Plan.from_problem(p)
    st, st32 = (torch.zeros(1, dtype=torch.int32, device="cuda") for _ in range(2))
    a = tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, d["psw"], dev_status=st)
    b = tbe.tbe_backward(plan, d32["grad"], d32["indices"], d32["offsets"], p.B, d32["psw"], dev_status=st32)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st32.item()) == 0
    U = int(a.unique_count[-1].item())
    assert torch.equal(a.unique_count, b.unique_count)
    assert torch.equal(a.unique_rows[:U], b.unique_rows[:U])
    assert torch.equal(a.run_starts[:U + 1], b.run_starts[:U + 1])
    assert torch.equal(a.sorted_positions[:p.N], b.sorted_positions[:p.N])
    n = int(np.sum(np.diff(a.unique_count.cpu().numpy()) * p.D))
    assert torch.equal(_bits(a.row_grads[:n]), _bits(b.row_grads[:n]))


def test_bad_ids_and_offsets_reported(tbe):
    G = np.ones((4, 24), np.float32)
    p = make_problem(2, 4, rows=[50, 60], D=[16, 8], weights_dtype=[DT_F32, DT_F32], out_dtype=DT_F32,
                     lengths=[[3, 2, 0, 1], [1, 1, 4, 0]],
                     ids=[[1, 50, 3, -2, 7, 9], [59, 60, 1, 2, -1, 99999]], grad_out=G, seed=4)
    w_dev, _ = parity.weights_pair(p)
    d, d32 = _both_widths(p)
    plan = tbe.Plan.from_problem(p)
    st, st32 = (torch.zeros(1, dtype=torch.int32, device="cuda") for _ in range(2))
    a = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, dev_status=st)
    b = tbe.tbe_forward(plan, w_dev, d32["indices"], d32["offsets"], p.B, dev_status=st32)
    ba = tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, dev_status=st)
    bb = tbe.tbe_backward(plan, d32["grad"], d32["indices"], d32["offsets"], p.B, dev_status=st32)
    torch.cuda.synchronize()
    assert int(st.item()) == int(st32.item()) == tbe.TBE_DEV_BAD_INDEX
    assert torch.equal(a, b)
    U = int(ba.unique_count[-1].item())
    assert torch.equal(ba.unique_rows[:U], bb.unique_rows[:U])
    assert torch.equal(ba.sorted_positions[:p.N], bb.sorted_positions[:p.N])
    st32.zero_()
    broken = torch.tensor([0, 4, 2, 5, 5, 6, 7, 11, 12], dtype=torch.int32, device="cuda")
    tbe.tbe_forward(plan, w_dev, d32["indices"], broken, p.B, dev_status=st32)
    torch.cuda.synchronize()
    assert int(st32.item()) & tbe.TBE_DEV_BAD_OFFSETS


def test_mixed_widths_rejected(tbe):
    p = make_config("tiny")
    w_dev, _ = parity.weights_pair(p)
    d, d32 = _both_widths(p)
    plan = tbe.Plan.from_problem(p)
    with pytest.raises(tbe.TBEError):
        tbe.tbe_forward(plan, w_dev, d32["indices"], d["offsets"], p.B)


@pytest.mark.parametrize("kind", [0, 1], ids=["sgd", "adagrad"])
def test_fused_update_matches_int64(tbe, kind):
    p = make_config("mid_skewed", B=300)
    w_a, _ = parity.weights_pair(p)
    w_b = w_a.clone()
    d, d32 = _both_widths(p)
    plan = tbe.Plan.from_problem(p)
    m_a = torch.rand(plan.total_rows, device="cuda") if kind == 1 else None
    m_b = m_a.clone() if kind == 1 else None
    a = tbe.tbe_backward_update(plan, w_a, kind, 0.05, d["grad"], d["indices"], d["offsets"], p.B, eps=1e-6,
                                momentum=m_a)
    b = tbe.tbe_backward_update(plan, w_b, kind, 0.05, d32["grad"], d32["indices"], d32["offsets"], p.B, eps=1e-6,
                                momentum=m_b)
    torch.cuda.synchronize()
    U = int(a.unique_count[-1].item())
    assert torch.equal(a.unique_rows[:U], b.unique_rows[:U])
    assert torch.equal(w_a, w_b)
    if kind == 1:
        assert torch.equal(m_a.view(torch.int32), m_b.view(torch.int32))


def test_wrappers_reject_arrays_the_kernels_would_overrun(tbe):
    """A wrong dtype, a short buffer or a host tensor is refused before any
    pointer reaches the library (the kernels would read or write past it)."""
    p = make_config("tiny")
    w_dev, _ = parity.weights_pair(p)
    d, d32 = _both_widths(p)
    plan = tbe.Plan.from_problem(p)
    fwd = lambda **kw: tbe.tbe_forward(plan, kw.get("w", w_dev), kw.get("ind", d["indices"]),  # noqa: E731
                                       kw.get("off", d["offsets"]), p.B, kw.get("psw"), out=kw.get("out"))
    bad = [dict(ind=d["indices"].to(torch.int16), off=d["offsets"].to(torch.int16)),
           dict(off=d["offsets"][:-1]),
           dict(ind=d["indices"].cpu(), off=d["offsets"].cpu()),
           dict(w=w_dev[: plan.weights_bytes - 1]),
           dict(psw=torch.ones(p.N, dtype=torch.float16, device="cuda")),
           dict(psw=torch.ones(p.N - 1, device="cuda")),
           dict(out=torch.empty((p.B, plan.sumD), dtype=torch.float16, device="cuda")),
           dict(out=torch.empty((p.B - 1, plan.sumD), device="cuda"))]
    for kw in bad:
        with pytest.raises(tbe.TBEError):
            fwd(**kw)
    with pytest.raises(tbe.TBEError):
        tbe.tbe_backward(plan, d["grad"].half(), d["indices"], d["offsets"], p.B)
    with pytest.raises(tbe.TBEError):
        tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B,
                         bufs=tbe.BackwardBuffers(plan, p.B, p.N - 1))
    with pytest.raises(tbe.TBEError):  # int64-only entry points
        tbe.tbe_backward_static_workspace(plan, d["grad"], d32["indices"], d32["offsets"], p.B)
    with pytest.raises(tbe.TBEError):
        tbe.tbe_histogram_counts(plan, d32["indices"], d32["offsets"], p.B)
    with pytest.raises(tbe.TBEError):  # momentum shorter than the tables' rows
        tbe.tbe_backward_update(plan, w_dev, 1, 0.1, d["grad"], d["indices"], d["offsets"], p.B,
                                momentum=torch.zeros(plan.total_rows - 1, device="cuda"))
    torch.cuda.synchronize()
