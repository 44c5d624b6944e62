"""Backward with the exact optimizer fused in (tbe_backward_update) (GPU).

The fused step must leave the tables and the momentum exactly as the
separate path does -- tbe_backward, then tbe_exact_update on its row
gradients -- bit for bit (the reducer applies the same FP32 operations in
the same order where each row's gradient is finished), and it is checked
against the oracle's backward + update like the separate step.
"""

import numpy as np
import pytest

import parity
from tbe_inputs import DT_BF16, DT_F16, DT_F32, make_config, make_problem
from test_gpu_optimizer import check_step, momentum_before

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

KINDS = [(0, "sgd", 0.05, 0.0), (1, "adagrad", 0.3, 1e-4)]


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


def narrow_problem(kind, weighted):
    """fp32 / fp16 / bf16 tables of 4..128 columns, repeated rows (a run of
    hundreds of lookups takes the chunked tier), empty bags, ragged batch."""
    rng = np.random.default_rng(900 + 2 * kind + weighted)
    specs = [(DT_F32, 4), (DT_F32, 12), (DT_F32, 128), (DT_F16, 8), (DT_F16, 128), (DT_BF16, 64), (DT_BF16, 128)]
    T, B = len(specs), 53
    rows = rng.integers(1, 300, size=T)
    lens = rng.integers(0, 50, size=(T, B))
    lens[:, 4] = 0
    ids = [rng.integers(0, rows[t], size=int(lens[t].sum())) for t in range(T)]
    ids[2][: len(ids[2]) // 2] = 7  # half of table 2's lookups on one row: a long run
    N = int(lens.sum())
    psw = rng.random(N).astype(np.float32) if weighted else None
    tw = (np.arange(T) % 2).astype(np.uint8) if weighted else None
    D = [d for _, d in specs]
    G = rng.standard_normal((B, sum(D))).astype(np.float32)
    return make_problem(T, B, rows=rows, D=D, weights_dtype=[s for s, _ in specs], out_dtype=DT_F32,
                        lengths=lens, ids=ids, psw=psw, grad_out=G, table_weighted=tw, seed=91)


def fused_vs_separate(tbe, p, kind, lr, eps, seed=5):
    """Runs both paths from the same tables and momentum; asserts equal bytes
    and equal indexing outputs; returns what the oracle check needs."""
    w_a, w_host = parity.weights_pair(p)
    w_b = w_a.clone()
    w_before = w_host.numpy().copy()
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    m0 = momentum_before(p, seed)
    adagrad = kind == tbe.TBE_OPT_EXACT_ROWWISE_ADAGRAD
    m_a = torch.from_numpy(m0).cuda() if adagrad else None
    m_b = torch.from_numpy(m0).cuda() if adagrad else None
    st_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_u = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    bufs = tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, d["psw"], dev_status=st_a)
    tbe.tbe_exact_update(plan, w_a, bufs, kind, lr, eps, momentum=m_a, dev_status=st_u)
    fb = tbe.tbe_backward_update(plan, w_b, kind, lr, d["grad"], d["indices"], d["offsets"], p.B, d["psw"],
                                 eps=eps, momentum=m_b, dev_status=st_b)
    torch.cuda.synchronize()
    assert int(st_b.item()) == int(st_a.item())
    U = int(bufs.unique_count[-1].item())
    assert int(fb.unique_count[-1].item()) == U
    assert torch.equal(fb.unique_rows[:U], bufs.unique_rows[:U])
    assert torch.equal(fb.run_starts[:U + 1], bufs.run_starts[:U + 1])
    assert torch.equal(fb.sorted_positions[:p.N], bufs.sorted_positions[:p.N])
    assert torch.equal(w_b, w_a), "fused weights differ from the separate step"
    if adagrad:
        assert torch.equal(m_b.view(torch.int32), m_a.view(torch.int32)), "fused momentum differs"
    return (w_before, w_b.cpu().numpy(), m0, m_b.cpu().numpy() if adagrad else None, int(st_b.item()),
            int(st_u.item()))


@pytest.mark.parametrize("kind,name,lr,eps", KINDS, ids=[k[1] for k in KINDS])
@pytest.mark.parametrize("weighted", [False, True])
def test_narrow_tables_match_separate_step_and_oracle(tbe, kind, name, lr, eps, weighted):
    p = narrow_problem(kind, weighted)
    w_before, w_after, m0, m_after, st, st_u = fused_vs_separate(tbe, p, kind, lr, eps)
    check_step(p, kind, lr, eps, w_before, w_after, m0, m_after, st, st_u)


@pytest.mark.parametrize("kind,name,lr,eps", KINDS, ids=[k[1] for k in KINDS])
@pytest.mark.parametrize("cfg,B,rows_scale", [("tiny", None, 1.0), ("mid_skewed", 300, 1.0),
                                              ("bwd_skew", 257, 0.02), ("small_table", 150, 1.0)])
def test_configs_reduced(tbe, kind, name, lr, eps, cfg, B, rows_scale):
    p = make_config(cfg, B=B, rows_scale=rows_scale)
    w_before, w_after, m0, m_after, st, st_u = fused_vs_separate(tbe, p, kind, lr, eps)
    check_step(p, kind, lr, eps, w_before, w_after, m0, m_after, st, st_u)


@pytest.mark.parametrize("tau,chunk", [(1, 32), (16, 32), (1 << 20, 256)])
def test_every_tier(tbe, tuned, tau, chunk):
    """All runs long with 32-lookup chunks (deep combine trees), mixed, and all
    runs short (the pending-row buffer is flushed many times)."""
    tuned(long_run_threshold=tau, long_chunk=chunk)
    for cfg, B in [("small_table", 120), ("mid_skewed", 256)]:
        p = make_config(cfg, B=B)
        fused_vs_separate(tbe, p, tbe.TBE_OPT_EXACT_ROWWISE_ADAGRAD, 0.3, 1e-4)


def test_mid_skewed_full_size(tbe):
    p = make_config("mid_skewed")
    fused_vs_separate(tbe, p, tbe.TBE_OPT_EXACT_ROWWISE_ADAGRAD, 0.01, 1e-8)


def test_bad_ids_are_skipped(tbe):
    G = np.random.default_rng(8).standard_normal((4, 24)).astype(np.float32)
    p = make_problem(2, 4, rows=[50, 60], D=[16, 8], weights_dtype=[DT_F32, DT_F16], out_dtype=DT_F32,
                     lengths=[[3, 2, 0, 1], [1, 1, 4, 0]],
                     ids=[[1, 50, 3, -2, 7, 9], [59, 60, 1, 2, -1, 99999]], grad_out=G, seed=4)
    w_before, w_after, m0, m_after, st, st_u = fused_vs_separate(tbe, p, 1, 0.3, 1e-4)
    assert st == tbe.TBE_DEV_BAD_INDEX
    check_step(p, 1, 0.3, 1e-4, w_before, w_after, m0, m_after, st, st_u, expect_bwd_status=tbe.TBE_DEV_BAD_INDEX)


def test_host_argument_errors(tbe):
    p = make_config("tiny")
    w_dev, _ = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    with pytest.raises(tbe.TBEError):  # unknown optimizer kind
        tbe.tbe_backward_update(plan, w_dev, 7, 0.1, d["grad"], d["indices"], d["offsets"], p.B)
    with pytest.raises(tbe.TBEError):  # Adagrad needs a momentum buffer
        tbe.tbe_backward_update(plan, w_dev, 1, 0.1, d["grad"], d["indices"], d["offsets"], p.B)
    q = make_problem(1, 2, rows=[5], D=[256], weights_dtype=[DT_F32], out_dtype=DT_F32, lengths=[[1, 1]],
                     ids=[[0, 1]], grad_out=np.ones((2, 256), np.float32))
    wq, _ = parity.weights_pair(q)
    dq = parity.upload(q)
    with pytest.raises(tbe.TBEError):  # rows wider than 128 columns: use tbe_backward + tbe_exact_update
        tbe.tbe_backward_update(tbe.Plan.from_problem(q), wq, 0, 0.1, dq["grad"], dq["indices"], dq["offsets"], 2)
