"""Parity at the workloads' full sizes, in the launch configuration the
benchmark uses (default tuning, one call per batch), on sampled outputs (GPU).

Forward: a seeded sample of bags (plus the longest and some empty ones) is
recomputed by the oracle.  Backward: the indexing outputs (sorted positions,
unique rows, run starts, per-table counts) are compared in full and bit for
bit; row gradients of a sample of runs (plus the longest runs, which take the
chunked tier) are recomputed by the oracle.
"""

import gc

import numpy as np
import pytest

import oracle
import parity
from tbe_inputs import make_config, materialize_weights

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")

N_SAMPLE = 3000


@pytest.fixture(scope="module")
def tbe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import table_embedding_bags_gb300 as m

    m.load_library()
    return m


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _sample_bags(p, rng):
    lens = np.diff(p.offsets)
    nb = p.T * p.B
    pick = set(rng.choice(nb, size=min(N_SAMPLE, nb), replace=False).tolist())
    pick.update(np.argsort(lens)[-20:].tolist())          # longest bags
    pick.update(np.nonzero(lens == 0)[0][:20].tolist())   # some empty bags
    return np.array(sorted(pick), np.int64)


@pytest.mark.parametrize("name", ["mixed", "small_table", "bwd_skew"])
def test_forward_full_size_sampled(tbe, name):
    p = make_config(name, with_grad=False)
    w_dev = materialize_weights(p, device="cuda")
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, d["psw"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got_all = out.float().cpu().numpy().astype(np.float64)
    w_host = w_dev.cpu()
    del w_dev, d, out
    _free()
    rng = np.random.default_rng(7)
    bags = _sample_bags(p, rng)
    ost, ref, ref_abs, pos = oracle.forward(p.layout_arrays(), w_host, p.indices, p.offsets, p.B,
                                            p.per_sample_weights, bags=bags)
    assert ost == 0
    doff = p.D_offsets
    got, cols = [], []
    for g in bags:
        t, b = int(g // p.B), int(g % p.B)
        got.append(got_all[b, doff[t]:doff[t + 1]])
        cols.append(np.full(int(p.D[t]), t))
    got = np.concatenate(got)[None, :]
    parity.compare_forward(p, got, ref[None, :], ref_abs[None, :], cols=np.concatenate(cols))


def auto_chunk(N):
    """Lookups per long-run chunk the library picks for a batch of N lookups
    with the default tuning: N / (128 x SMs) rounded down to 32, in 64..256."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return min(256, max(64, N // (4 * 32 * sms) // 32 * 32))


@pytest.mark.parametrize("name", ["mixed", "small_table", "bwd_skew"])
def test_backward_full_size(tbe, name):
    p = make_config(name)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bufs = tbe.BackwardBuffers(plan, p.B, p.N)
    tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, d["psw"], bufs=bufs, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    lay = p.layout_arrays()
    idx = oracle.backward_indexing(lay, p.indices, p.offsets, p.B)
    assert idx["status"] == 0
    U = int(bufs.unique_count[-1].item())
    assert U == idx["U"]
    np.testing.assert_array_equal(bufs.unique_count.cpu().numpy(), idx["unique_count"])
    np.testing.assert_array_equal(bufs.unique_rows[:U].cpu().numpy(), idx["unique_rows"])
    np.testing.assert_array_equal(bufs.run_starts[:U + 1].cpu().numpy(), idx["run_starts"])
    np.testing.assert_array_equal(bufs.sorted_positions[:p.N].cpu().numpy(), idx["sorted_pos"])
    # row gradients of sampled runs: the longest (chunked tier) and a random sample
    lens = np.diff(idx["run_starts"])
    rng = np.random.default_rng(11)
    runs = set(np.argsort(lens)[-64:].tolist())
    runs.update(rng.choice(U, size=min(N_SAMPLE, U), replace=False).tolist())
    runs = np.array(sorted(runs), np.int64)
    ost, rg, rabs, rpos = oracle.backward_values(lay, p.offsets, p.B, p.grad_out, idx, p.per_sample_weights,
                                                 runs=runs, nthreads=0)
    assert ost == 0
    # where the library put each sampled run (table-major blocks)
    uc = idx["unique_count"]
    D = p.D.astype(np.int64)
    gofs = np.concatenate([[0], np.cumsum(np.diff(uc) * D)])
    t_of = np.searchsorted(p.table_row_base, idx["unique_rows"][runs], side="right") - 1
    starts = gofs[t_of] + (runs - uc[t_of]) * D[t_of]
    rg_all = bufs.row_grads
    got = np.concatenate([rg_all[int(s):int(s) + int(D[t])].cpu().numpy() for s, t in zip(starts, t_of)])
    parity.compare_rowgrads(got.astype(np.float64), rg, rabs)
    assert lens.max() >= 256  # the workload exercises the chunked long-run tier
    if name == "small_table":
        # 18.9 M lookups on 64 rows: runs of ~295 K lookups are cut into more
        # than 32 x 32 chunks, so the fan-in-32 combine tree has three levels
        assert -(-int(lens.max()) // auto_chunk(p.N)) > 32 * 32
    del d, bufs
    _free()
