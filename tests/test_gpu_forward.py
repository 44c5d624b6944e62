"""Forward parity: the CUDA gather kernel against the oracle (GPU)."""

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


def run_forward(tbe, p, path=None, psw=True, status=None):
    w_dev, w_host = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    kw = {} if path is None else dict(path=path)
    out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, d["psw"] if psw else None,
                          dev_status=st, **kw)
    torch.cuda.synchronize()
    return out, int(st.item()), w_host


def check_full(tbe, p, path=None):
    out, st, w_host = run_forward(tbe, p, path)
    assert st == 0
    ost, ref, ref_abs = oracle.problem_forward(p, w_host)
    assert ost == 0
    return parity.compare_forward(p, parity.to_f64(out), ref, ref_abs)


@pytest.fixture(params=[2, 1, 0], ids=["stream", "ring", "registers"])
def gather_mode(tbe, request):
    """Runs a test with each gather kernel: the stream kernel (2, rows of at
    most 512 bytes through a cp.async ring, bags of a task back to back), the
    per-bag shared-memory ring (1) and rows loaded into registers (0)."""
    old = tbe.get_tuning()
    tbe.set_tuning(fwd_ring=request.param)
    yield request.param
    tbe.set_tuning(**old)


@pytest.mark.parametrize("name,B,rows_scale", [
    ("tiny", None, 1.0),
    ("mid_skewed", None, 1.0),
    ("mixed", 300, 0.01),
    ("small_table", 777, 1.0),
    ("bwd_skew", 301, 0.02),
])
def test_configs_reduced(tbe, gather_mode, name, B, rows_scale):
    p = make_config(name, B=B, rows_scale=rows_scale)
    check_full(tbe, p, path=tbe.TBE_PATH_GATHER)


@pytest.mark.parametrize("out_dt", [DT_F32, DT_F16, DT_BF16])
@pytest.mark.parametrize("weighted", [False, True])
def test_shapes_and_dtypes(tbe, out_dt, weighted):
    """Row widths from one 16-byte chunk to column-blocked rows, all dtypes,
    bags spanning several 32-id groups and a ragged batch."""
    rng = np.random.default_rng(100 + out_dt * 2 + weighted)
    specs = [(DT_F32, 4), (DT_F32, 12), (DT_F32, 128), (DT_F32, 256), (DT_F32, 520),
             (DT_F16, 8), (DT_F16, 24), (DT_F16, 136), (DT_BF16, 64), (DT_BF16, 256), (DT_BF16, 1024)]
    T, B = len(specs), 37
    rows = rng.integers(1, 3000, size=T)
    lens = rng.integers(0, 90, size=(T, B))
    lens[:, 3] = 0
    lens[2, 5] = 200
    ids = [rng.integers(0, rows[t], size=int(lens[t].sum())) for t in range(T)]
    N = int(lens.sum())
    psw = rng.random(N).astype(np.float32) if weighted else None
    tw = (np.arange(T) % 2).astype(np.uint8) if weighted else None
    p = make_problem(T, B, rows=rows, D=[d for _, d in specs], weights_dtype=[s for s, _ in specs],
                     out_dtype=out_dt, lengths=lens, ids=ids, psw=psw, table_weighted=tw, seed=99)
    check_full(tbe, p, path=tbe.TBE_PATH_GATHER)


@pytest.mark.parametrize("out_dt", [DT_F32, DT_F16, DT_BF16])
@pytest.mark.parametrize("weighted", [False, True])
def test_narrow_rows_long_bags(tbe, gather_mode, out_dt, weighted):
    """Rows of 16..512 bytes in every dtype, a row width that is not a power
    of two chunks, bags longer than several id windows, empty bags."""
    rng = np.random.default_rng(300 + out_dt * 2 + weighted)
    specs = [(DT_F32, 4), (DT_F32, 16), (DT_F32, 128), (DT_F16, 8), (DT_F16, 24), (DT_F16, 256),
             (DT_BF16, 64), (DT_BF16, 128), (DT_BF16, 256), (DT_F32, 36)]
    T, B = len(specs), 45
    rows = rng.integers(1, 2000, size=T)
    lens = rng.integers(0, 70, size=(T, B))
    lens[:, 7] = 0
    lens[1, 3] = 300
    lens[5, 44] = 97
    lens[2, 9] = 1500  # fp32 bags far past the ~160-add depth a single serial fp32 sum guarantees
    lens[0, 11] = 700
    lens[9, 20] = 2000
    ids = [rng.integers(0, rows[t], size=int(lens[t].sum())) for t in range(T)]
    N = int(lens.sum())
    psw = rng.random(N).astype(np.float32) if weighted else None
    tw = (np.arange(T) % 3 != 0).astype(np.uint8) if weighted else None
    p = make_problem(T, B, rows=rows, D=[d for _, d in specs], weights_dtype=[s for s, _ in specs],
                     out_dtype=out_dt, lengths=lens, ids=ids, psw=psw, table_weighted=tw, seed=98)
    check_full(tbe, p, path=tbe.TBE_PATH_GATHER)


def split_bags(T, B, N, grid):
    """Bags per block with which the stream kernel splits its tasks (0: it
    does not): the fewest that fit every table's runs in one wave, at most
    32, with 32 positions per warp on average at least."""
    nbb = max(1, -(-T * B // grid))
    while nbb <= 32 and T * -(-B // nbb) > grid:
        nbb += 1
    runs = T * -(-B // nbb)
    return nbb if nbb <= 32 and N >= 32 * 4 * runs else 0


@pytest.mark.parametrize("dt,D", [(DT_F16, 128), (DT_BF16, 64), (DT_F32, 64), (DT_F16, 8), (DT_F32, 4)])
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("pooling", [0, 1])
def test_split_tasks(tbe, dt, D, weighted, pooling):
    """The stream kernel's split tasks: a block pools one run of bags in four
    equal parts of its padded stream, so bags are cut by part boundaries --
    one bag longer than the rest of its run, runs of empty bags, bags of one
    lookup -- and the pieces are added after a block barrier."""
    rng = np.random.default_rng(31 + D + 2 * weighted + pooling)
    T, B, rows = 3, 96, 300
    lens = rng.poisson(40, size=(T, B))
    lens[0, 5] = 3000
    lens[1, ::7] = 0
    lens[2, 10:20] = 1
    lens[1, 40:48] = 0
    N = int(lens.sum())
    assert split_bags(T, B, N, -(-T * B // 4)) > 0
    ids = [rng.integers(0, rows, size=int(lens[t].sum())) for t in range(T)]
    psw = rng.standard_normal(N).astype(np.float32) if weighted else None
    p = make_problem(T, B, rows=[rows] * T, D=[D] * T, weights_dtype=[dt] * T, out_dtype=DT_F32, lengths=lens,
                     ids=ids, psw=psw, table_weighted=[1] * T if weighted else None, seed=7, pooling=pooling)
    old = tbe.get_tuning()
    tbe.set_tuning(fwd_ring=2)
    try:
        check_full(tbe, p, path=tbe.TBE_PATH_GATHER)
    finally:
        tbe.set_tuning(**old)


def test_split_tasks_idle_blocks_and_short_last_run(tbe):
    """A batch whose runs do not fill the grid (blocks without a run) and
    whose tables end in a run shorter than the others."""
    rng = np.random.default_rng(41)
    T, B, rows, D = 5, 97, 500, 64
    lens = rng.poisson(40, size=(T, B))
    lens[3, -2:] = [700, 0]
    ids = [rng.integers(0, rows, size=int(lens[t].sum())) for t in range(T)]
    p = make_problem(T, B, rows=[rows] * T, D=[D] * T, weights_dtype=[DT_F16] * T, out_dtype=DT_F16, lengths=lens,
                     ids=ids, seed=9)
    grid = -(-T * B // 4)
    nbb = split_bags(T, B, p.N, grid)
    assert nbb > 0 and T * -(-B // nbb) < grid and B % nbb != 0
    old = tbe.get_tuning()
    tbe.set_tuning(fwd_ring=2)
    try:
        check_full(tbe, p, path=tbe.TBE_PATH_GATHER)
    finally:
        tbe.set_tuning(**old)


def test_split_tasks_bad_id_in_a_cut_bag(tbe):
    """A bad id inside the bag that spans the parts is reported and adds
    nothing; every other output still matches."""
    T, B, rows, D = 2, 64, 100, 32
    lens = np.full((T, B), 40)
    lens[0, 3] = 2000
    ids = [np.arange(int(lens[t].sum())) % rows for t in range(T)]
    ids[0][int(lens[0, :3].sum()) + 1500] = rows + 5
    p = make_problem(T, B, rows=[rows] * T, D=[D] * T, weights_dtype=[DT_F16] * T, out_dtype=DT_F32, lengths=lens,
                     ids=ids, seed=3)
    assert split_bags(T, B, p.N, -(-T * B // 4)) > 0
    old = tbe.get_tuning()
    tbe.set_tuning(fwd_ring=2)
    try:
        out, st, w_host = run_forward(tbe, p, tbe.TBE_PATH_GATHER)
    finally:
        tbe.set_tuning(**old)
    assert st == tbe.TBE_DEV_BAD_INDEX
    ost, ref, ref_abs = oracle.problem_forward(p, w_host)
    assert ost == oracle.BAD_INDEX
    parity.compare_forward(p, parity.to_f64(out), ref, ref_abs)


def test_repeated_ids_and_empty(tbe, gather_mode):
    p = make_problem(2, 3, rows=[5, 7], D=[8, 4], weights_dtype=[DT_F16, DT_F32], out_dtype=DT_F32,
                     lengths=[[0, 40, 1], [3, 0, 0]], ids=[[2] * 40 + [4], [6, 6, 0]])
    check_full(tbe, p)


def test_all_empty_and_zero_batch(tbe):
    p = make_problem(3, 16, rows=[5, 7, 9], D=[8, 4, 16], weights_dtype=[DT_F16, DT_F32, DT_BF16],
                     out_dtype=DT_F16, lengths=np.zeros((3, 16)), ids=[[], [], []])
    out, st, _ = run_forward(tbe, p)
    assert st == 0 and torch.count_nonzero(out).item() == 0
    q = make_problem(1, 0, rows=[5], D=[8], weights_dtype=[DT_F32], out_dtype=DT_F32,
                     lengths=np.zeros((1, 0)), ids=[[]])
    out, st, _ = run_forward(tbe, q)
    assert out.shape == (0, 8) and st == 0


def test_bad_ids_reported_and_skipped(tbe, gather_mode):
    p = make_problem(2, 4, rows=[50, 60], D=[16, 8], weights_dtype=[DT_F32, DT_F16], out_dtype=DT_F32,
                     lengths=[[3, 2, 0, 1], [1, 1, 4, 0]], ids=[[1, 50, 3, -2, 7, 9], [59, 60, 1, 2, -1, 99999]])
    out, st, w_host = run_forward(tbe, p)
    assert st == tbe.TBE_DEV_BAD_INDEX
    ost, ref, ref_abs = oracle.problem_forward(p, w_host)
    assert ost == oracle.BAD_INDEX
    parity.compare_forward(p, parity.to_f64(out), ref, ref_abs)


@pytest.mark.parametrize("bad", [[1, 2, 4, 5], [0, 2, 4, 4], [0, 4, 2, 5], [0, 2, 4, 9]])
def test_bad_offsets_reported(tbe, gather_mode, bad):
    p = make_problem(1, 3, rows=[50], D=[16], weights_dtype=[DT_F32], out_dtype=DT_F32,
                     lengths=[[2, 2, 1]], ids=[[1, 2, 3, 4, 5]])
    w_dev, _ = parity.weights_pair(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tbe.tbe_forward(plan, w_dev, torch.from_numpy(p.indices).cuda(), torch.tensor(bad, device="cuda"), 3,
                    dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tbe.TBE_DEV_BAD_OFFSETS


def test_deterministic(tbe, gather_mode):
    p = make_config("mid_skewed")
    w_dev, _ = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    a = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B)
    b = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("unroll,lpr,per_sm", [(4, 8, 0), (8, 8, 0), (8, 4, 0), (8, 16, 0), (4, 32, 0), (8, 1, 0),
                                            (4, 2, 0), (4, 16, 4), (4, 8, 4)])
def test_unroll_variants(tbe, unroll, lpr, per_sm):
    old = tbe.get_tuning()
    try:
        tbe.set_tuning(fwd_unroll=unroll, fwd_lanes_per_row=lpr, fwd_blocks_per_sm=per_sm, fwd_ring=0)
        p = make_config("mixed", B=64, rows_scale=0.005)
        check_full(tbe, p, path=tbe.TBE_PATH_GATHER)
    finally:
        tbe.set_tuning(**old)


@pytest.mark.parametrize("lpr", [1, 4, 8, 32])
def test_ring_lanes_per_row(tbe, lpr):
    """The ring gather with one bag per warp up to 32 bags per warp (two
    chunks per lane where the row is wider than the lanes)."""
    old = tbe.get_tuning()
    try:
        tbe.set_tuning(fwd_lanes_per_row=lpr, fwd_ring=1)
        check_full(tbe, make_config("mixed", B=64, rows_scale=0.005), path=tbe.TBE_PATH_GATHER)
        check_full(tbe, make_config("mid_skewed", B=128, rows_scale=0.1), path=tbe.TBE_PATH_GATHER)
    finally:
        tbe.set_tuning(**old)


def test_host_argument_errors(tbe):
    p = make_config("tiny")
    w_dev, _ = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    out = torch.empty((p.B, p.total_D), dtype=torch.float32, device="cuda")
    with pytest.raises(tbe.TBEError):  # negative batch size
        tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], -1, out=out)
    with pytest.raises(tbe.TBEError):  # histogram path needs one small fp16 table
        tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, path=tbe.TBE_PATH_HISTOGRAM)
    with pytest.raises(tbe.TBEError):  # rows that are not a multiple of 16 bytes
        tbe.Plan(1, [0, 10], [0, 3], [0], [DT_F32], DT_F32)
