"""Backward parity: sort + segment + short/long-run reduce against the oracle (GPU).

Indexing outputs (sorted positions, unique rows, run starts, per-table run
counts) must match bit for bit; row gradients within 1e-5 * sum|terms|.
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


@pytest.fixture
def tuned(tbe):
    old = tbe.get_tuning()
    yield tbe.set_tuning
    tbe.set_tuning(**old)


def run_backward(tbe, p, capacity=None):
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bufs = tbe.BackwardBuffers(plan, p.B, p.N, row_grads_capacity=capacity)
    tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, d["psw"], bufs=bufs, dev_status=st)
    torch.cuda.synchronize()
    return bufs, int(st.item())


def check_backward(tbe, p, expect_status=0):
    bufs, st = run_backward(tbe, p)
    assert st == expect_status
    lay = p.layout_arrays()
    idx = oracle.backward_indexing(lay, p.indices, p.offsets, p.B)
    U = int(bufs.unique_count[-1].item())
    assert U == idx["U"]
    np.testing.assert_array_equal(bufs.unique_count.cpu().numpy(), idx["unique_count"])
    np.testing.assert_array_equal(bufs.unique_rows[:U].cpu().numpy(), idx["unique_rows"])
    np.testing.assert_array_equal(bufs.run_starts[:U + 1].cpu().numpy(), idx["run_starts"])
    np.testing.assert_array_equal(bufs.sorted_positions[:p.N].cpu().numpy(), idx["sorted_pos"])
    ost, rg, rabs, _ = oracle.backward_values(lay, p.offsets, p.B, p.grad_out, idx, p.per_sample_weights)
    assert ost == 0
    got = bufs.row_grads[:rg.size].cpu().numpy().astype(np.float64)
    parity.compare_rowgrads(got, rg, rabs)
    return bufs, idx


@pytest.mark.parametrize("name,B,rows_scale", [
    ("tiny", None, 1.0),
    ("mid_skewed", None, 1.0),
    ("mixed", 400, 0.01),
    ("small_table", 300, 1.0),
    ("bwd_skew", 400, 0.05),
])
def test_configs_reduced(tbe, name, B, rows_scale):
    check_backward(tbe, make_config(name, B=B, rows_scale=rows_scale))


@pytest.mark.parametrize("tau,chunk", [(1, 32), (2, 64), (32, 32), (33, 256), (256, 256), (4096, 256),
                                       (1 << 20, 1024)])
def test_tiers_and_thresholds(tbe, tuned, tau, chunk):
    """Every run short, every run long with tiny chunks (deep combine trees),
    and the thresholds in between all give the same rows and sums."""
    tuned(long_run_threshold=tau, long_chunk=chunk)
    check_backward(tbe, make_config("small_table", B=200))
    check_backward(tbe, make_config("mid_skewed", B=256))


@pytest.mark.parametrize("unroll", [4, 8])
@pytest.mark.parametrize("item", [32, 40, 64, 1000])
def test_reduce_variants(tbe, tuned, unroll, item):
    """Both reduction kernels (4 or 8 slices in flight per lane) and short-run
    work items from one part per batch to many, weighted and unweighted."""
    tuned(red_unroll=unroll, short_item_lookups=item)
    check_backward(tbe, make_config("mixed", B=200, rows_scale=0.01))
    check_backward(tbe, make_config("mid_skewed", B=300))


def test_deterministic_bits(tbe, tuned):
    tuned(long_run_threshold=16, long_chunk=32)
    p = make_config("bwd_skew", B=300, rows_scale=0.01)
    a, _ = run_backward(tbe, p)
    U = int(a.unique_count[-1].item())
    n = U * 128  # every table of this workload has D = 128
    ra = a.row_grads[:n].clone()
    b, _ = run_backward(tbe, p)
    assert torch.equal(ra.view(torch.int32), b.row_grads[:n].view(torch.int32))
    assert torch.equal(a.unique_rows[:U], b.unique_rows[:U])


@pytest.mark.parametrize("weighted", [False, True])
def test_widths_and_dtypes(tbe, weighted):
    rng = np.random.default_rng(7 + weighted)
    specs = [(DT_F32, 4), (DT_F32, 12), (DT_F16, 128), (DT_F32, 256), (DT_BF16, 136), (DT_F32, 520)]
    T, B = len(specs), 45
    rows = rng.integers(1, 400, size=T)
    lens = rng.integers(0, 70, size=(T, B))
    ids = [rng.integers(0, rows[t], size=int(lens[t].sum())) for t in range(T)]
    N = int(lens.sum())
    psw = rng.random(N).astype(np.float32) if weighted else None
    tw = (np.arange(T) % 2).astype(np.uint8) if weighted else None
    G = rng.standard_normal((B, sum(d for _, d in specs))).astype(np.float32)
    p = make_problem(T, B, rows=rows, D=[d for _, d in specs], weights_dtype=[s for s, _ in specs],
                     out_dtype=DT_F32, lengths=lens, ids=ids, psw=psw, grad_out=G, table_weighted=tw)
    check_backward(tbe, p)


def test_weighted_pairing_with_permuted_duplicates(tbe, tuned):
    """Many lookups of one row with distinct weights: each weight must meet
    its own bag's gradient (one stable order carries both)."""
    tuned(long_run_threshold=64, long_chunk=32)
    rng = np.random.default_rng(3)
    T, B = 2, 500
    lens = rng.integers(1, 6, size=(T, B))
    ids = [rng.choice([0, 1, 2], size=int(lens[t].sum())) for t in range(T)]
    N = int(lens.sum())
    psw = (rng.permutation(N).astype(np.float32) + 1) / N
    G = rng.standard_normal((B, 8)).astype(np.float32)
    p = make_problem(T, B, rows=[3, 3], D=[4, 4], weights_dtype=[DT_F32, DT_F32], out_dtype=DT_F32,
                     lengths=lens, ids=ids, psw=psw, grad_out=G)
    check_backward(tbe, p)


def test_bad_ids_excluded(tbe):
    G = np.ones((3, 8), np.float32)
    p = make_problem(2, 3, rows=[5, 7], D=[4, 4], weights_dtype=[DT_F32, DT_F32], out_dtype=DT_F32,
                     lengths=[[2, 1, 3], [2, 0, 1]], ids=[[1, 5, 2, -1, 4, 1], [6, 7, 99]], grad_out=G)
    check_backward(tbe, p, expect_status=tbe.TBE_DEV_BAD_INDEX)


@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("bad", [False, True])
def test_segmented_sort(tbe, weighted, bad):
    """Few tables of at most 2^18 rows with more than 2^16 rows in total: the
    radix sort runs over ids within each table (two passes); ids outside
    their table must still end up behind every valid lookup, in position
    order, exactly as the global sort with its sentinel puts them."""
    rng = np.random.default_rng(71 + 2 * weighted + bad)
    rows = [70000, 50000, 100, 3000, 200000]
    T, B = len(rows), 700
    lens = rng.integers(0, 40, size=(T, B))
    lens[2, :] = rng.integers(0, 3, size=B)
    ids = []
    for t in range(T):
        n = int(lens[t].sum())
        x = (rng.zipf(1.3, size=n) * 7919) % rows[t]
        if bad:  # ids outside the table: negative and too large
            k = rng.choice(n, size=max(1, n // 50), replace=False)
            x[k[::2]] = -3
            x[k[1::2]] = rows[t] + 5
        ids.append(x)
    N = int(lens.sum())
    psw = rng.random(N).astype(np.float32) if weighted else None
    tw = np.array([1, 0, 1, 1, 0], np.uint8) if weighted else None
    D = [64, 32, 128, 16, 64]
    G = rng.standard_normal((B, sum(D))).astype(np.float32)
    p = make_problem(T, B, rows=rows, D=D, weights_dtype=[DT_F32] * T, out_dtype=DT_F32, lengths=lens, ids=ids,
                     psw=psw, table_weighted=tw, grad_out=G)
    check_backward(tbe, p, expect_status=tbe.TBE_DEV_BAD_INDEX if bad else 0)


def test_empty_batches(tbe):
    p = make_problem(2, 8, rows=[5, 7], D=[4, 8], weights_dtype=[DT_F32, DT_F16], out_dtype=DT_F32,
                     lengths=np.zeros((2, 8)), ids=[[], []], grad_out=np.ones((8, 12), np.float32))
    bufs, st = run_backward(tbe, p)
    assert st == 0 and bufs.unique_count.cpu().tolist() == [0, 0, 0]
    q = make_problem(2, 8, rows=[5, 7], D=[4, 8], weights_dtype=[DT_F32, DT_F16], out_dtype=DT_F32,
                     lengths=np.array([[0] * 7 + [1], [0] * 8]), ids=[[3], []],
                     grad_out=np.ones((8, 12), np.float32))
    check_backward(tbe, q)


def test_capacity_reported(tbe):
    p = make_config("tiny")
    bufs, st = run_backward(tbe, p, capacity=8)
    assert st & tbe.TBE_DEV_CAPACITY


def test_bad_offsets_reported(tbe):
    p = make_problem(1, 3, rows=[50], D=[16], weights_dtype=[DT_F32], out_dtype=DT_F32,
                     lengths=[[2, 2, 1]], ids=[[1, 2, 3, 4, 5]], grad_out=np.ones((3, 16), np.float32))
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bufs = tbe.BackwardBuffers(plan, 3, 5)
    tbe.tbe_backward(plan, torch.from_numpy(p.grad_out).cuda(), torch.from_numpy(p.indices).cuda(),
                     torch.tensor([0, 4, 2, 5], device="cuda"), 3, bufs=bufs, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tbe.TBE_DEV_BAD_OFFSETS


def test_workspace_too_small(tbe):
    p = make_config("tiny")
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    bufs = tbe.BackwardBuffers(plan, p.B, p.N)
    bufs.workspace = bufs.workspace[:256]
    with pytest.raises(tbe.TBEError):
        tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, bufs=bufs)
