"""Mean pooling (TBE_POOL_MEAN) against the oracle (GPU).

Every forward kernel (stream, per-bag ring, registers, histogram) divides a
bag's fp32 sum by its number of lookups; the backward gives each lookup
(w_i / L_b) * grad_out[b].  Outputs and row gradients are compared element
by element with the oracle's mean (the sum's output, and the sum's backward
on grad_out, scaled per bag), with the usual tolerances taken on the scaled
absolute sums; indexing outputs must be bit-exact.
"""

import numpy as np
import pytest

import oracle
import parity
from tbe_inputs import DT_BF16, DT_F16, DT_F32, make_config, make_problem
from test_gpu_backward import check_backward
from test_gpu_forward import check_full

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tbe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import table_embedding_bags_gb300 as m

    m.load_library()
    return m


@pytest.fixture(params=[3, 2, 1, 0], ids=["auto", "stream", "ring", "registers"])
def gather_mode(tbe, request):
    old = tbe.get_tuning()
    tbe.set_tuning(fwd_ring=request.param)
    yield request.param
    tbe.set_tuning(**old)


CONFIGS = [("tiny", None, 1.0), ("mid_skewed", 500, 1.0), ("mixed", 300, 0.01), ("bwd_skew", 301, 0.02)]


def _mean(p):
    p.pooling = 1
    return p


@pytest.mark.parametrize("name,B,rows_scale", CONFIGS)
def test_forward_every_gather_kernel(tbe, gather_mode, name, B, rows_scale):
    check_full(tbe, _mean(make_config(name, B=B, rows_scale=rows_scale)), path=tbe.TBE_PATH_GATHER)


@pytest.mark.parametrize("weighted", [False, True])
def test_forward_histogram_path(tbe, weighted):
    """fp16 and bf16 tables (one weighted or not), histogram path and gather
    path, bags of 0..300 lookups."""
    rng = np.random.default_rng(17 + weighted)
    specs = [(64, 128, DT_F16), (20, 64, DT_BF16), (33, 256, DT_F16)]
    T, B = len(specs), 260
    lens = rng.integers(0, 301, size=(T, B))
    lens[:, 3] = 0
    ids = [rng.integers(0, specs[t][0], size=int(lens[t].sum())) for t in range(T)]
    psw = rng.standard_normal(int(lens.sum())).astype(np.float32) if weighted else None
    p = make_problem(T, B, rows=[s[0] for s in specs], D=[s[1] for s in specs], weights_dtype=[s[2] for s in specs],
                     out_dtype=DT_F32, lengths=lens, ids=ids, psw=psw, table_weighted=[1, 0, 1] if weighted else None,
                     seed=5, pooling=1)
    check_full(tbe, p, path=tbe.TBE_PATH_HISTOGRAM)
    check_full(tbe, p, path=tbe.TBE_PATH_GATHER)


def test_forward_small_table_full_size(tbe):
    """Config 4 at full size on the histogram path (sampled against the oracle)."""
    p = _mean(make_config("small_table"))
    w_dev, w_host = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bags = np.random.default_rng(3).choice(p.B, size=500, replace=False).astype(np.int64)
    ost, ref, ref_abs, pos = oracle.problem_forward(p, w_host, bags=bags)
    assert ost == 0
    got = parity.to_f64(out)[bags]
    parity.compare_forward(p, got, ref.reshape(len(bags), -1), ref_abs.reshape(len(bags), -1))


@pytest.mark.parametrize("name,B,rows_scale", CONFIGS + [("small_table", 300, 1.0)])
def test_backward(tbe, name, B, rows_scale):
    check_backward(tbe, _mean(make_config(name, B=B, rows_scale=rows_scale)))


def test_backward_weighted_tables(tbe):
    rng = np.random.default_rng(23)
    T, B = 3, 97
    lens = rng.integers(0, 40, size=(T, B))
    ids = [rng.integers(0, 50, size=int(lens[t].sum())) for t in range(T)]
    psw = rng.random(int(lens.sum())).astype(np.float32)
    G = rng.standard_normal((B, 3 * 32)).astype(np.float32)
    p = make_problem(T, B, rows=[50] * 3, D=[32] * 3, weights_dtype=[DT_F32, DT_F16, DT_BF16], out_dtype=DT_F32,
                     lengths=lens, ids=ids, psw=psw, grad_out=G, table_weighted=[1, 0, 1], seed=6, pooling=1)
    check_backward(tbe, p)


@pytest.mark.parametrize("kind", [0, 1], ids=["sgd", "adagrad"])
def test_fused_update_equals_separate(tbe, kind):
    p = _mean(make_config("mid_skewed", B=400))
    w_a, _ = parity.weights_pair(p)
    w_b = w_a.clone()
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    m_a = torch.rand(plan.total_rows, device="cuda") if kind == 1 else None
    m_b = m_a.clone() if kind == 1 else None
    bufs = tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B)
    tbe.tbe_exact_update(plan, w_a, bufs, kind, 0.05, 1e-6, momentum=m_a)
    tbe.tbe_backward_update(plan, w_b, kind, 0.05, d["grad"], d["indices"], d["offsets"], p.B, eps=1e-6, momentum=m_b)
    torch.cuda.synchronize()
    assert torch.equal(w_a, w_b)
    if kind == 1:
        assert torch.equal(m_a.view(torch.int32), m_b.view(torch.int32))


def test_mean_is_the_sum_over_the_length(tbe):
    """The same batch pooled both ways: mean * L reproduces the sum (within
    the rounding of one division), and empty bags are zero in both."""
    p = make_config("mid_skewed", B=300)
    w_dev, _ = parity.weights_pair(p)
    d = parity.upload(p)
    s = tbe.tbe_forward(tbe.Plan.from_problem(p), w_dev, d["indices"], d["offsets"], p.B).float()
    m = tbe.tbe_forward(tbe.Plan.from_problem(_mean(p)), w_dev, d["indices"], d["offsets"], p.B).float()
    torch.cuda.synchronize()
    L = torch.from_numpy(np.diff(p.offsets).reshape(p.T, p.B).T.astype(np.float32)).cuda()  # [B, T]
    Lc = L.repeat_interleave(int(p.D[0]), dim=1)
    assert torch.all(m[Lc == 0] == 0) and torch.all(s[Lc == 0] == 0)
    nz = Lc > 0
    assert torch.allclose((m * Lc)[nz], s[nz], rtol=2e-3, atol=1e-3)  # fp16 output rounding


def test_all_bags_empty(tbe):
    """Mean of no lookups is 0 on every path, and the backward has no rows."""
    p = make_problem(2, 4, rows=[5, 7], D=[16, 32], weights_dtype=[DT_F16, DT_BF16], out_dtype=DT_F32,
                     lengths=[[0] * 4, [0] * 4], ids=[[], []], grad_out=np.ones((4, 48), np.float32), pooling=1)
    w_dev, _ = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    for path in (tbe.TBE_PATH_GATHER, tbe.TBE_PATH_HISTOGRAM):
        out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, path=path)
        torch.cuda.synchronize()
        assert torch.count_nonzero(out) == 0
    bufs = tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B)
    torch.cuda.synchronize()
    assert bufs.unique_count.cpu().tolist() == [0, 0, 0]
