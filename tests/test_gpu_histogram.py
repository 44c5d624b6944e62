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


def _problem(specs, B, lo, hi, out_dt=DT_F32, seed=0, weighted=None, psw_scale=1.0):
    """Tables given as (rows, D, dtype); bag lengths U{lo..hi}, uniform ids;
    per-sample weights (signed, of magnitude about psw_scale) when
    ``weighted`` (one flag per table) is given."""
    rng = np.random.default_rng(seed)
    T = len(specs)
    lens = rng.integers(lo, hi + 1, size=(T, B))
    ids = [rng.integers(0, specs[t][0], size=int(lens[t].sum())) for t in range(T)]
    psw = None
    if weighted is not None:
        psw = (rng.standard_normal(int(lens.sum())) * psw_scale).astype(np.float32)
    return make_problem(T, B, rows=[s[0] for s in specs], D=[s[1] for s in specs],
                        weights_dtype=[s[2] for s in specs], out_dtype=out_dt, lengths=lens, ids=ids, psw=psw,
                        table_weighted=weighted, seed=seed + 17)


def _column_tolerance(p, ref, ref_abs):
    cols = np.repeat(np.arange(p.T), np.diff(p.D_offsets))
    tol = np.zeros(ref.shape)
    for dt in np.unique(p.weights_dtype):
        m = np.broadcast_to(p.weights_dtype[cols] == dt, ref.shape)
        tol[m] = parity.tolerance(ref[m], ref_abs[m], int(dt), p.out_dtype)[0]
    return tol


def check(tbe, p, compare_gather=True):
    w_dev, w_host = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cnt = tbe.tbe_histogram_counts(plan, d["indices"], d["offsets"], p.B, dev_status=st)
    out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, d["psw"], dev_status=st,
                          path=tbe.TBE_PATH_HISTOGRAM)
    gat = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, d["psw"], dev_status=st,
                          path=tbe.TBE_PATH_GATHER)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for t in range(p.T):
        ost, ref_cnt = oracle.histogram_counts(p.T, p.B, t, int(p.rows[t]), p.indices, p.offsets)
        assert ost == 0
        np.testing.assert_array_equal(cnt[t].cpu().numpy(), ref_cnt)
    ost, ref, ref_abs = oracle.problem_forward(p, w_host)
    assert ost == 0
    parity.compare_forward(p, parity.to_f64(out), ref, ref_abs)
    if compare_gather:
        parity.compare_forward(p, parity.to_f64(gat), ref, ref_abs)
        # the two kernels compute the same sums; both sit within the tolerance of
        # the exact result, so they agree to twice that tolerance
        tol = _column_tolerance(p, ref, ref_abs)
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


MULTI = [(64, 128, DT_F16), (20, 64, DT_BF16), (1, 16, DT_F16), (50, 80, DT_BF16), (33, 256, DT_F16)]


@pytest.mark.parametrize("out_dt", [DT_F32, DT_F16, DT_BF16])
def test_several_tables_one_launch(tbe, out_dt):
    """fp16 and bf16 tables of different rows and widths, one launch; a
    ragged last tile (B = 300)."""
    check(tbe, _problem(MULTI, B=300, lo=0, hi=200, out_dt=out_dt, seed=31 + out_dt))


@pytest.mark.parametrize("rows,D", [(1, 16), (3, 128), (17, 48), (64, 256)])
def test_bf16_counts_split_at_256(tbe, rows, D):
    """bf16 counts are exact only to 256: bags of 300..1500 ids over a few rows
    put most counts above it (the lo / hi split), one bag of 5000 ids over the
    recount limit."""
    rng = np.random.default_rng(rows * 7 + D)
    lens = rng.integers(300, 1501, size=(1, 40))
    lens[0, 3] = 5000
    lens[0, 5] = 0
    ids = [rng.integers(0, min(rows, 4), size=int(lens.sum()))]
    p = make_problem(1, 40, rows=[rows], D=[D], weights_dtype=[DT_BF16], out_dtype=DT_F32, lengths=lens, ids=ids,
                     seed=rows)
    _, cnt = oracle.histogram_counts(1, 40, 0, rows, p.indices, p.offsets)
    assert (cnt > 256).sum() >= 30 and lens.max() > 2048  # lo / hi split, and a recounted bag
    check(tbe, p)


@pytest.mark.parametrize("psw_scale", [1.0, 1e-4, 300.0])
def test_weighted_tables(tbe, psw_scale):
    """Per-sample weights summed per (bag, row) and split into two tf32 terms;
    table 1 is not weighted (its lookups count 1), fp16 and bf16 mixed."""
    specs = [(64, 128, DT_F16), (40, 64, DT_BF16), (7, 32, DT_BF16), (64, 256, DT_F16)]
    check(tbe, _problem(specs, B=260, lo=0, hi=300, seed=5, weighted=[1, 0, 1, 1], psw_scale=psw_scale))


def test_weighted_is_deterministic_and_matches_int32(tbe):
    p = _problem(MULTI, B=400, lo=20, hi=400, out_dt=DT_F16, seed=12, weighted=[1] * len(MULTI))
    w_dev, _ = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    runs = [tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, d["psw"], path=tbe.TBE_PATH_HISTOGRAM)
            for _ in range(3)]
    i32 = tbe.tbe_forward(plan, w_dev, d["indices"].to(torch.int32), d["offsets"].to(torch.int32), p.B, d["psw"],
                          path=tbe.TBE_PATH_HISTOGRAM)
    torch.cuda.synchronize()
    for r in runs[1:] + [i32]:
        assert torch.equal(r.view(torch.int16), runs[0].view(torch.int16))


def test_weighted_long_bags_and_bad_ids(tbe):
    """Weighted bags of up to 5000 ids (fp32 sums need no recount) and ids out
    of range, which are skipped and reported."""
    rng = np.random.default_rng(21)
    lens = np.array([[5000, 0, 3, 2100, 1, 700]])
    ids = rng.integers(0, 5, size=int(lens.sum()))
    ids[10], ids[5003] = 5, -1
    psw = rng.random(int(lens.sum())).astype(np.float32)
    p = make_problem(1, 6, rows=[5], D=[64], weights_dtype=[DT_BF16], out_dtype=DT_F32, lengths=lens, ids=[ids],
                     psw=psw, seed=3)
    w_dev, w_host = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, d["psw"], dev_status=st,
                          path=tbe.TBE_PATH_HISTOGRAM)
    torch.cuda.synchronize()
    assert int(st.item()) == tbe.TBE_DEV_BAD_INDEX
    ost, ref, ref_abs = oracle.problem_forward(p, w_host)
    assert ost == oracle.BAD_INDEX
    parity.compare_forward(p, parity.to_f64(out), ref, ref_abs)


def test_layouts_with_one_ineligible_table_use_the_gather(tbe):
    for specs in ([(64, 128, DT_F16), (10, 64, DT_F32)], [(64, 128, DT_F16), (10, 24, DT_BF16)],
                  [(64, 128, DT_F16), (65, 64, DT_F16)]):
        p = _problem(specs, B=64, lo=100, hi=200, seed=2)
        w_dev, _ = parity.weights_pair(p)
        d = parity.upload(p)
        plan = tbe.Plan.from_problem(p)
        with pytest.raises(tbe.TBEError):
            tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, path=tbe.TBE_PATH_HISTOGRAM)
        tbe.trace_enable(True)
        tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B)
        stages = tbe.trace_read()
        tbe.trace_enable(False)
        assert [n for n, _ in stages] == ["fwd_gather"]


def test_auto_path_several_tables(tbe):
    p = _problem([(32, 128, DT_BF16), (16, 64, DT_F16)], B=256, lo=60, hi=200, seed=8, weighted=[1, 1])
    w_dev, _ = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    tbe.trace_enable(True)
    tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, d["psw"])
    stages = tbe.trace_read()
    tbe.trace_enable(False)
    assert [n for n, _ in stages] == ["fwd_histogram"]
