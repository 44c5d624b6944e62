"""Small-table histogram path (counts x table on tcgen05) against the oracle (GPU).

Counts must match the oracle's histogram bit for bit; pooled outputs must
meet the forward tolerance against the oracle and agree with the gather
kernel (both are the same sum, one as a gather, one as counts x table).
"""

import numpy as np
import pytest

import oracle
import parity
from tbe_inputs import DT_BF16, DT_F16, DT_F32, make_config, make_problem

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tbe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import table_embedding_bags_gb300 as m

    m.load_library()
    return m


def _small_problem(rows, D, B, lo, hi, out_dt=DT_F32, seed=0, std=0.02):
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=(1, B))
    ids = [rng.integers(0, rows, size=int(lens.sum()))]
    w = torch.from_numpy((rng.standard_normal((rows, D)) * std).astype(np.float32).astype(np.float16))
    return make_problem(1, B, rows=[rows], D=[D], weights_dtype=[DT_F16], out_dtype=out_dt, lengths=lens,
                        ids=ids, host_tables={0: w})


def check(tbe, p, compare_gather=True):
    w_dev, w_host = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cnt = tbe.tbe_histogram_counts(plan, d["indices"], d["offsets"], p.B, dev_status=st)
    out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, dev_status=st, path=tbe.TBE_PATH_HISTOGRAM)
    gat = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, dev_status=st, path=tbe.TBE_PATH_GATHER)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ost, ref_cnt = oracle.histogram_counts(1, p.B, 0, int(p.rows[0]), p.indices, p.offsets)
    assert ost == 0
    np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
    ost, ref, ref_abs = oracle.problem_forward(p, w_host)
    assert ost == 0
    parity.compare_forward(p, parity.to_f64(out), ref, ref_abs)
    if compare_gather:
        parity.compare_forward(p, parity.to_f64(gat), ref, ref_abs)
        # the two kernels compute the same sums; both sit within the tolerance of
        # the exact result, so they agree to twice that tolerance
        tol, _ = parity.tolerance(ref, ref_abs, DT_F16, p.out_dtype)
        assert np.all(np.abs(parity.to_f64(out) - parity.to_f64(gat)) <= 2 * tol)
    return out


def test_small_table_config_reduced(tbe):
    check(tbe, make_config("small_table", B=1000))


@pytest.mark.parametrize("rows,D", [(1, 16), (7, 48), (16, 64), (33, 128), (64, 128), (64, 256), (50, 80)])
def test_shapes(tbe, rows, D):
    check(tbe, _small_problem(rows, D, B=300, lo=0, hi=200, seed=rows * 1000 + D))


@pytest.mark.parametrize("out_dt", [DT_F16, DT_BF16])
def test_output_types(tbe, out_dt):
    check(tbe, _small_problem(64, 128, B=257, lo=60, hi=300, out_dt=out_dt, seed=out_dt))


def test_bags_longer_than_exact_fp16_counts(tbe):
    # a bag of 5000 ids over 3 rows has counts > 2048: recounted exactly
    rng = np.random.default_rng(4)
    lens = np.array([[5000, 0, 3, 2100, 1]])
    ids = [rng.integers(0, 3, size=int(lens.sum()))]
    w = torch.from_numpy((rng.standard_normal((3, 32)) * 0.02).astype(np.float32).astype(np.float16))
    p = make_problem(1, 5, rows=[3], D=[32], weights_dtype=[DT_F16], out_dtype=DT_F32, lengths=lens, ids=ids,
                     host_tables={0: w})
    check(tbe, p)


def test_auto_path_picks_histogram_for_long_bags(tbe):
    p = make_config("small_table", B=512)
    w_dev, _ = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    tbe.trace_enable(True)
    tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B)
    stages = tbe.trace_read()
    tbe.trace_enable(False)
    assert [n for n, _ in stages] == ["fwd_histogram"]


def test_bad_ids_and_offsets(tbe):
    p = _small_problem(16, 64, B=130, lo=1, hi=40, seed=9)
    p.indices[5] = 16
    p.indices[7] = -3
    w_dev, w_host = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, dev_status=st, path=tbe.TBE_PATH_HISTOGRAM)
    torch.cuda.synchronize()
    assert int(st.item()) == tbe.TBE_DEV_BAD_INDEX
    ost, ref, ref_abs = oracle.problem_forward(p, w_host)
    assert ost == oracle.BAD_INDEX
    parity.compare_forward(p, parity.to_f64(out), ref, ref_abs)
    bad = d["offsets"].clone()
    bad[3] = bad[4] + 1
    st.zero_()
    tbe.tbe_forward(plan, w_dev, d["indices"], bad, p.B, dev_status=st, path=tbe.TBE_PATH_HISTOGRAM)
    torch.cuda.synchronize()
    assert int(st.item()) & tbe.TBE_DEV_BAD_OFFSETS


def test_ineligible_layouts_refused(tbe):
    p = make_config("tiny")
    w_dev, _ = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    with pytest.raises(tbe.TBEError):
        tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, path=tbe.TBE_PATH_HISTOGRAM)
    q = _small_problem(65, 64, B=10, lo=1, hi=5)  # 65 rows: above the tile
    with pytest.raises(tbe.TBEError):
        tbe.tbe_histogram_counts(tbe.Plan.from_problem(q), parity.upload(q)["indices"],
                                 parity.upload(q)["offsets"], q.B)
