"""The seeded input generators: shapes, ranges and reproducibility (CPU only)."""

import numpy as np
import pytest
import torch

from tbe_inputs import DT_F16, config_names, make_config, materialize_weights, table_rows


@pytest.mark.parametrize("name", config_names())
def test_config_shapes(name):
    p = make_config(name, B=64, rows_scale=0.01 if name in ("mixed", "bwd_skew") else 1.0)
    assert p.offsets.shape == (p.T * p.B + 1,)
    assert p.offsets[0] == 0 and p.offsets[-1] == p.N and np.all(np.diff(p.offsets) >= 0)
    for t in range(p.T):
        seg = p.indices[p.offsets[t * p.B]: p.offsets[(t + 1) * p.B]]
        assert np.all((seg >= 0) & (seg < p.rows[t]))
    assert p.grad_out.shape == (p.B, p.total_D) and p.grad_out.dtype == np.float32
    assert np.all(p.weights_offsets % 256 == 0)
    if name in ("tiny", "mid_skewed", "mid_uniform", "mid_identity"):
        assert (np.diff(p.offsets) == 0).any()
    if name == "mixed":
        assert p.per_sample_weights is not None and int(p.table_weighted.sum()) == 20
    # same seed, same batch -> identical draws; another batch -> other ids
    q = make_config(name, B=64, rows_scale=0.01 if name in ("mixed", "bwd_skew") else 1.0)
    assert np.array_equal(p.indices, q.indices) and np.array_equal(p.grad_out, q.grad_out)
    r = make_config(name, B=64, rows_scale=0.01 if name in ("mixed", "bwd_skew") else 1.0, batch=1)
    assert not np.array_equal(p.indices, r.indices) or p.N == 0


def test_table_rows_regenerate_buffer():
    p = make_config("mixed", B=8, rows_scale=0.002)
    w = materialize_weights(p)
    rng = np.random.default_rng(0)
    for t in range(p.T):
        R, D = int(p.rows[t]), int(p.D[t])
        ids = rng.integers(0, R, size=5)
        got = table_rows(p, t, ids)
        eb = got.element_size()
        off = int(p.weights_offsets[t])
        view = w[off: off + R * D * eb].view(got.dtype).view(R, D)
        assert torch.equal(view[torch.as_tensor(ids)], got)
        assert float(got.float().abs().max()) <= 0.0505  # U(-0.05, 0.05) after rounding


def test_zipf_is_skewed():
    p = make_config("mid_skewed", B=2048)
    seg = p.indices[p.offsets[0]: p.offsets[p.B]]
    counts = np.bincount(seg, minlength=int(p.rows[0]))
    top = np.sort(counts)[::-1]
    assert top[0] > 0.05 * seg.size  # hottest row takes several percent of lookups
    assert int(p.weights_dtype[0]) == DT_F16


def test_bench_byte_counts_on_the_hand_example():
    """The benchmark's byte accounting, counted by hand on the two-table
    example: T=2, B=2, fp32 tables of widths 2 and 1, fp32 output, 4 + 3
    lookups, 3 + 2 distinct rows, 5 offsets."""
    import bench
    from oracle_pins import _hand_problem

    _, p = _hand_problem(False)
    U = [3, 2]
    # effective: lookups 4*(2*4 + 8) + 3*(1*4 + 8) = 100; offsets 40; output 2*3*4 = 24
    # backward: lookups 4*(4*2 + 8) + 3*(4*1 + 8) = 100; offsets 40; rows 3*(8+8) + 2*(8+4) = 72
    assert bench.effective_bytes(p, U) == (164, 212)
    # compulsory: rows 3*2*4 + 2*1*4 = 32; ids 7*8 = 56; offsets 40; output 24 -> 152
    # backward: ids 56; offsets 40; G once 4*2*3 = 24; rows 72 -> 192
    assert bench.compulsory_bytes(p, U) == (152, 192)
    # Adagrad step: per row 8 + 4*D + 2*4*D + 8 -> 40 for D=2, 28 for D=1; plus (T+1)*8
    assert bench.optimizer_bytes(p, U) == 3 * 40 + 2 * 28 + 24


def test_uniform_control_matches_the_skewed_workload():
    """Same tables and bag lengths as the mid-size skewed batch, ids spread
    evenly: many more distinct rows, no row far above the mean."""
    a, b = make_config("mid_skewed"), make_config("mid_uniform")
    assert np.array_equal(a.offsets, b.offsets) and np.array_equal(a.grad_out, b.grad_out)
    assert np.array_equal(a.rows, b.rows) and np.array_equal(a.weights_offsets, b.weights_offsets)
    ua = sum(len(np.unique(a.indices[a.offsets[t * a.B]: a.offsets[(t + 1) * a.B]])) for t in range(a.T))
    ub = sum(len(np.unique(b.indices[b.offsets[t * b.B]: b.offsets[(t + 1) * b.B]])) for t in range(b.T))
    assert ub > 2 * ua
    seg = b.indices[b.offsets[0]: b.offsets[b.B]]
    assert np.bincount(seg, minlength=int(b.rows[0])).max() < 12


@pytest.mark.parametrize("name", ["band_short", "band_mid", "band_long"])
def test_run_length_bands(name):
    """Every distinct row of a band workload is read a number of times inside
    its band (one run per table may fall short: the remainder), and the three
    bands share their bag lengths."""
    from tbe_inputs import RUN_BANDS

    lo, hi = RUN_BANDS[name]
    p = make_config(name, B=512, with_grad=False)
    q = make_config("band_mid", B=512, with_grad=False)
    assert np.array_equal(p.offsets, q.offsets)
    for t in range(p.T):
        seg = p.indices[p.offsets[t * p.B]: p.offsets[(t + 1) * p.B]]
        assert np.all((seg >= 0) & (seg < p.rows[t]))
        _, counts = np.unique(seg, return_counts=True)
        outside = counts[(counts < lo) | (counts > hi)]
        assert outside.size <= 1 and np.all(outside < lo), (t, outside)
        assert counts[(counts >= lo) & (counts <= hi)].sum() >= 0.9 * seg.size or seg.size < 2 * hi


def test_identity_case_keeps_the_skew_but_not_the_permutation():
    a, c = make_config("mid_skewed"), make_config("mid_identity")
    assert np.array_equal(a.offsets, c.offsets)
    seg_a = a.indices[a.offsets[0]: a.offsets[a.B]]
    seg_c = c.indices[c.offsets[0]: c.offsets[c.B]]
    # the most frequent id is rank 1: id 0 without the permutation
    assert np.bincount(seg_c).argmax() == 0
    # same number of distinct rows up to sampling noise (the permutation only renames rows)
    assert abs(len(np.unique(seg_a)) - len(np.unique(seg_c))) < 0.05 * len(np.unique(seg_a))
