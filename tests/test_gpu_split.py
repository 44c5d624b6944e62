"""The backward in two calls: tbe_backward_index, then tbe_backward_reduce (GPU).

The pair must give exactly what one tbe_backward (or tbe_backward_update)
call gives -- the same distinct rows, run starts, sorted positions, counts,
row gradients or updated tables, bit for bit -- whether the index stages run
on the same stream or on a second stream beside a forward.  The one-call
results are themselves checked against the oracle by the other GPU tests.
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


CONFIGS = [("tiny", None, 1.0), ("mid_skewed", 400, 1.0), ("mixed", 300, 0.01), ("small_table", 200, 1.0),
           ("bwd_skew", 257, 0.02)]


def _same_indexing(p, a, b):
    U = int(a.unique_count[-1].item())
    assert torch.equal(a.unique_count, b.unique_count)
    assert torch.equal(a.unique_rows[:U], b.unique_rows[:U])
    assert torch.equal(a.run_starts[:U + 1], b.run_starts[:U + 1])
    assert torch.equal(a.sorted_positions[:p.N], b.sorted_positions[:p.N])
    return U


@pytest.mark.parametrize("name,B,rows_scale", CONFIGS)
@pytest.mark.parametrize("width", [64, 32])
def test_split_equals_one_call(tbe, name, B, rows_scale, width):
    p = make_config(name, B=B, rows_scale=rows_scale)
    d = parity.upload(p)
    if width == 32:
        d = dict(d, indices=d["indices"].to(torch.int32), offsets=d["offsets"].to(torch.int32))
    plan = tbe.Plan.from_problem(p)
    st1, st2 = (torch.zeros(1, dtype=torch.int32, device="cuda") for _ in range(2))
    one = tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, d["psw"], dev_status=st1)
    two = tbe.tbe_backward_index(plan, d["indices"], d["offsets"], p.B, d["psw"], dev_status=st2)
    tbe.tbe_backward_reduce(plan, d["grad"], two, per_sample_weights=d["psw"], dev_status=st2)
    torch.cuda.synchronize()
    assert int(st1.item()) == int(st2.item()) == 0
    _same_indexing(p, one, two)
    n = int(np.sum(np.diff(one.unique_count.cpu().numpy()) * p.D))
    assert torch.equal(one.row_grads[:n].view(torch.int32), two.row_grads[:n].view(torch.int32))


def test_index_on_a_second_stream_beside_the_forward(tbe):
    """The index stages on a side stream while the forward runs, the
    reduction after both; repeated over rotated batches."""
    for batch in range(3):
        p = make_config("mid_skewed", batch=batch)
        w_dev, _ = parity.weights_pair(p)
        d = parity.upload(p)
        plan = tbe.Plan.from_problem(p)
        one = tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B)
        ref_out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B)
        torch.cuda.synchronize()
        main, side = torch.cuda.current_stream(), torch.cuda.Stream()
        side.wait_stream(main)
        bufs = tbe.BackwardBuffers(plan, p.B, p.N)
        with torch.cuda.stream(side):
            tbe.tbe_backward_index(plan, d["indices"], d["offsets"], p.B, bufs=bufs, stream=side)
        out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, stream=main)
        main.wait_stream(side)
        tbe.tbe_backward_reduce(plan, d["grad"], bufs, stream=main)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out)
        _same_indexing(p, one, bufs)
        n = int(np.sum(np.diff(one.unique_count.cpu().numpy()) * p.D))
        assert torch.equal(one.row_grads[:n].view(torch.int32), bufs.row_grads[:n].view(torch.int32))


@pytest.mark.parametrize("kind", [0, 1], ids=["sgd", "adagrad"])
def test_split_with_the_fused_update(tbe, kind):
    p = make_config("mid_skewed", B=500)
    w_a, _ = parity.weights_pair(p)
    w_b = w_a.clone()
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    m_a = torch.rand(plan.total_rows, device="cuda") if kind == 1 else None
    m_b = m_a.clone() if kind == 1 else None
    tbe.tbe_backward_update(plan, w_a, kind, 0.05, d["grad"], d["indices"], d["offsets"], p.B, eps=1e-6, momentum=m_a)
    bufs = tbe.tbe_backward_index(plan, d["indices"], d["offsets"], p.B, fused=True)
    tbe.tbe_backward_reduce(plan, d["grad"], bufs, kind=kind, learning_rate=0.05, weights=w_b, eps=1e-6, momentum=m_b)
    torch.cuda.synchronize()
    assert torch.equal(w_a, w_b)
    if kind == 1:
        assert torch.equal(m_a.view(torch.int32), m_b.view(torch.int32))


def test_split_misuse_is_refused(tbe):
    p = make_config("tiny")
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    with pytest.raises(tbe.TBEError):  # no index call on these buffers
        tbe.tbe_backward_reduce(plan, d["grad"], tbe.BackwardBuffers(plan, p.B, p.N))
    bufs = tbe.tbe_backward_index(plan, d["indices"], d["offsets"], p.B)
    with pytest.raises(tbe.TBEError):  # weights given to one call only
        tbe.tbe_backward_reduce(plan, d["grad"], bufs, per_sample_weights=torch.ones(p.N, device="cuda"))
    torch.cuda.synchronize()


def test_split_with_no_lookups(tbe):
    """Every bag empty (N = 0): the index call clears the counts and the
    reduction has nothing to do."""
    p = make_problem(2, 3, rows=[5, 7], D=[4, 8], weights_dtype=[DT_F32, DT_F32], out_dtype=DT_F32,
                     lengths=[[0, 0, 0], [0, 0, 0]], ids=[[], []], grad_out=np.ones((3, 12), np.float32))
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bufs = tbe.tbe_backward_index(plan, d["indices"], d["offsets"], p.B, dev_status=st)
    tbe.tbe_backward_reduce(plan, d["grad"], bufs, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert bufs.unique_count.cpu().tolist() == [0, 0, 0]
