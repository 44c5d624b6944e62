"""Pins for the oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an oracle library handle (so a deliberately
broken build of the oracle can be run through the same checks) and raises
AssertionError on a mismatch.  What pins what:

* ``pin_hand_example``  -- values worked by hand (tests/golden/hand_example.json)
  from the page's semantics: empty bag = 0, repeated id counted twice,
  column offsets, row gradient = sum of bag gradients, stable key order.
* ``pin_dense_onehot``  -- the textbook form: with A_t[b, r] = sum of the
  weights of the lookups of bag (t, b) that name row r, the forward is the
  matrix product A_t @ W_t and the table gradient is A_t^T @ G_t (numpy
  float64 matmul, a library routine).
* ``pin_invariants``    -- column sums, adjoint identity, lookup count,
  histogram form == gather form bit for bit (exact fp64 sums of fp16).
* ``pin_sort_vs_numpy`` -- sorted positions equal numpy's stable argsort.
* ``pin_formats``       -- fp16/bf16 decoding over all 65536 codes and
  nearest-even rounding against numpy and against a brute-force nearest
  search.
* ``pin_special_cases`` -- all-empty batch, single-id bags, one id repeated
  n times, out-of-range ids, broken offsets.
* ``pin_mean_hand``     -- mean pooling worked by hand: each bag's mean of its
  rows, an empty bag 0, and a lookup of bag b receiving grad_out[b] / L_b.
* ``pin_mean_dense``    -- mean pooling in the textbook form: with M_t =
  diag(1 / L_b) A_t (empty bags: a zero row), the forward is M_t @ W_t and
  the table gradient M_t^T @ G_t (numpy float64 matmul).
* ``pin_optimizer_hand`` -- exact SGD and row-wise Adagrad steps worked by
  hand (tests/golden/optimizer_example.json), with momentum carried over
  from an earlier step and with and without eps.
* ``pin_optimizer_invariants`` -- properties the update must have whatever
  the data: a first Adagrad step from zero momentum (eps 0) moves each row
  by exactly lr * sqrt(D_t) in Euclidean norm and is unchanged when the
  gradient is scaled; duplicating every column leaves momentum and update
  unchanged (a mean, not a sum); SGD is linear in the gradient; Adagrad
  whose denominator sqrt(m) + eps equals 1 is SGD; rows outside every
  table are reported.
"""

from __future__ import annotations

import json
import os

import numpy as np

import oracle
from tbe_inputs import DT_BF16, DT_F16, DT_F32, make_problem, materialize_weights

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _hand_problem(weighted: bool):
    import torch

    g = json.load(open(os.path.join(GOLDEN, "hand_example.json")))
    T, B = g["T"], g["B"]
    offs = np.array(g["offsets"])
    lens = np.diff(offs).reshape(T, B)
    ind = np.array(g["indices"])
    ids = [ind[offs[t * B]: offs[(t + 1) * B]] for t in range(T)]
    tables = {t: torch.tensor(g["tables"][t], dtype=torch.float32) for t in range(T)}
    p = make_problem(T, B, rows=[3, 2], D=[2, 1], weights_dtype=[DT_F32, DT_F32], out_dtype=DT_F32,
                     lengths=lens, ids=ids, grad_out=np.array(g["grad_out"], np.float32),
                     psw=np.array(g["per_sample_weights"], np.float32) if weighted else None,
                     host_tables=tables)
    return g, p


def pin_hand_example(lib):
    for weighted in (False, True):
        g, p = _hand_problem(weighted)
        w = materialize_weights(p)
        st, out, _ = oracle.problem_forward(p, w, lib=lib)
        assert st == 0
        exp = g["expected"]["weighted_out" if weighted else "out"]
        np.testing.assert_array_equal(out, np.array(exp, np.float64))
        idx, st2, rg, _, pos = oracle.problem_backward(p, lib=lib)
        assert st2 == 0 and idx["status"] == 0
        np.testing.assert_array_equal(idx["sorted_pos"], g["expected"]["sorted_pos"])
        np.testing.assert_array_equal(idx["unique_rows"], g["expected"]["unique_rows"])
        np.testing.assert_array_equal(idx["run_starts"], g["expected"]["run_starts"])
        np.testing.assert_array_equal(idx["unique_count"], g["expected"]["unique_count"])
        exp_rg = g["expected"]["weighted_row_grads" if weighted else "row_grads"]
        np.testing.assert_array_equal(rg, np.concatenate([np.array(r, np.float64) for r in exp_rg]))
        # the fp32 output rounding of small integers is exact
        np.testing.assert_array_equal(oracle.round_to(out, DT_F32, lib=lib), np.array(exp, np.float32))


def _random_problem(rng, T, B, dtypes, weighted, max_len=7, max_rows=9):
    rows = rng.integers(1, max_rows + 1, size=T)
    D = rng.choice([1, 2, 3, 4, 8], size=T)
    lens = rng.integers(0, max_len + 1, size=(T, B))
    ids = [rng.integers(0, rows[t], size=int(lens[t].sum())) for t in range(T)]
    G = rng.standard_normal((B, int(D.sum()))).astype(np.float32)
    N = int(lens.sum())
    psw = rng.random(N).astype(np.float32) * 2 - 0.5 if weighted else None
    tw = None
    if weighted:
        tw = (rng.random(T) < 0.6).astype(np.uint8)
    p = make_problem(T, B, rows=rows, D=D, weights_dtype=[dtypes[t % len(dtypes)] for t in range(T)],
                     out_dtype=DT_F32, lengths=lens, ids=ids, psw=psw, grad_out=G,
                     table_weighted=tw, seed=int(rng.integers(1 << 30)))
    return p


def _table_f64(p, w, t):
    """Decode table t of the packed buffer with numpy's own format support."""
    import torch

    code = int(p.weights_dtype[t])
    R, D = int(p.rows[t]), int(p.D[t])
    off = int(p.weights_offsets[t])
    eb = 4 if code == DT_F32 else 2
    raw = w[off: off + R * D * eb]
    if code == DT_F32:
        return raw.view(torch.float32).numpy().astype(np.float64).reshape(R, D)
    if code == DT_F16:
        return raw.view(torch.float16).numpy().astype(np.float64).reshape(R, D)
    bits = raw.view(torch.int16).numpy().astype(np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64).reshape(R, D)


def pin_dense_onehot(lib, trials=40, seed=5):
    rng = np.random.default_rng(seed)
    for k in range(trials):
        T = int(rng.integers(1, 5))
        B = int(rng.integers(1, 6))
        weighted = bool(k % 2)
        p = _random_problem(rng, T, B, [DT_F32, DT_F16, DT_BF16], weighted)
        w = materialize_weights(p)
        st, out, _ = oracle.problem_forward(p, w, lib=lib)
        assert st == 0
        idx, st2, rg, _, rpos = oracle.problem_backward(p, lib=lib)
        assert st2 == 0
        doff = p.D_offsets
        trb = p.table_row_base
        for t in range(T):
            R = int(p.rows[t])
            A = np.zeros((B, R), np.float64)
            for b in range(B):
                g = t * B + b
                for i in range(int(p.offsets[g]), int(p.offsets[g + 1])):
                    wi = 1.0
                    if p.per_sample_weights is not None and p.table_weighted[t]:
                        wi = float(p.per_sample_weights[i])
                    A[b, p.indices[i]] += wi
            Wt = _table_f64(p, w, t)
            exp = A @ Wt
            np.testing.assert_allclose(out[:, doff[t]: doff[t + 1]], exp, rtol=1e-12, atol=1e-12)
            Gt = p.grad_out[:, doff[t]: doff[t + 1]].astype(np.float64)
            dense = A.T @ Gt  # [R, D_t]
            occurring = np.nonzero(np.bincount(p.indices[p.offsets[t * B]: p.offsets[(t + 1) * B]],
                                               minlength=R))[0]
            uc = idx["unique_count"]
            ours_rows = idx["unique_rows"][uc[t]: uc[t + 1]] - trb[t]
            np.testing.assert_array_equal(ours_rows, occurring)
            Dt = int(p.D[t])
            for j, u in enumerate(range(int(uc[t]), int(uc[t + 1]))):
                got = rg[rpos[u]: rpos[u] + Dt]
                np.testing.assert_allclose(got, dense[occurring[j]], rtol=1e-12, atol=1e-12)


def pin_mean_hand(lib):
    """T=1, three rows of D=2, table [[1,2],[3,4],[5,6]] (fp32); bags [0,2],
    [1,1,2] and []; grad_out rows (1,1), (3,3), (7,7).  By hand: outputs
    (3,4), (11/3, 14/3), (0,0); row gradients row0 = (1,1)/2 = (0.5,0.5),
    row1 = 2*(3,3)/3 = (2,2), row2 = (1,1)/2 + (3,3)/3 = (1.5,1.5)."""
    import torch

    table = torch.tensor([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]], dtype=torch.float32)
    G = np.array([[1.0, 1.0], [3.0, 3.0], [7.0, 7.0]], np.float32)
    p = make_problem(1, 3, rows=[3], D=[2], weights_dtype=[DT_F32], out_dtype=DT_F32, lengths=[[2, 3, 0]],
                     ids=[[0, 2, 1, 1, 2]], grad_out=G, host_tables={0: table}, pooling=1)
    w = materialize_weights(p)
    st, out, _ = oracle.problem_forward(p, w, lib=lib)
    assert st == 0
    np.testing.assert_allclose(out, [[3.0, 4.0], [11 / 3, 14 / 3], [0.0, 0.0]], rtol=1e-15)
    idx, st2, rg, _, rpos = oracle.problem_backward(p, lib=lib)
    assert st2 == 0
    np.testing.assert_array_equal(idx["unique_rows"], [0, 1, 2])
    np.testing.assert_allclose(rg.reshape(3, 2), [[0.5, 0.5], [2.0, 2.0], [1.5, 1.5]], rtol=1e-15)


def pin_mean_dense(lib, trials=30, seed=13):
    rng = np.random.default_rng(seed)
    for k in range(trials):
        T = int(rng.integers(1, 5))
        B = int(rng.integers(1, 6))
        p = _random_problem(rng, T, B, [DT_F32, DT_F16, DT_BF16], bool(k % 2))
        p.pooling = 1
        w = materialize_weights(p)
        st, out, _ = oracle.problem_forward(p, w, lib=lib)
        idx, st2, rg, _, rpos = oracle.problem_backward(p, lib=lib)
        assert st == 0 and st2 == 0
        doff, trb, uc = p.D_offsets, p.table_row_base, idx["unique_count"]
        for t in range(T):
            R = int(p.rows[t])
            M = np.zeros((B, R), np.float64)
            for b in range(B):
                g = t * B + b
                L = int(p.offsets[g + 1] - p.offsets[g])
                for i in range(int(p.offsets[g]), int(p.offsets[g + 1])):
                    wi = 1.0
                    if p.per_sample_weights is not None and p.table_weighted[t]:
                        wi = float(p.per_sample_weights[i])
                    M[b, p.indices[i]] += wi / L
            np.testing.assert_allclose(out[:, doff[t]: doff[t + 1]], M @ _table_f64(p, w, t), rtol=1e-12, atol=1e-12)
            dense = M.T @ p.grad_out[:, doff[t]: doff[t + 1]].astype(np.float64)
            Dt = int(p.D[t])
            for u in range(int(uc[t]), int(uc[t + 1])):
                r = int(idx["unique_rows"][u] - trb[t])
                np.testing.assert_allclose(rg[rpos[u]: rpos[u] + Dt], dense[r], rtol=1e-12, atol=1e-12)


def pin_invariants(lib, trials=30, seed=11):
    rng = np.random.default_rng(seed)
    for k in range(trials):
        T = int(rng.integers(1, 5))
        B = int(rng.integers(1, 7))
        weighted = bool(k % 3 == 0)
        p = _random_problem(rng, T, B, [DT_F16, DT_F32, DT_BF16], weighted, max_len=12, max_rows=20)
        w = materialize_weights(p)
        st, out, oabs = oracle.problem_forward(p, w, lib=lib)
        idx, st2, rg, rabs, rpos = oracle.problem_backward(p, lib=lib)
        assert st == 0 and st2 == 0
        # I3: lookup count, strictly increasing rows inside their tables
        rs = idx["run_starts"]
        assert rs[0] == 0 and rs[-1] == p.N and np.all(np.diff(rs) > 0)
        ur = idx["unique_rows"]
        assert np.all(np.diff(ur) > 0)
        trb = p.table_row_base
        uc = idx["unique_count"]
        for t in range(T):
            seg = ur[uc[t]: uc[t + 1]]
            assert np.all((seg >= trb[t]) & (seg < trb[t + 1]))
        assert sorted(idx["sorted_pos"].tolist()) == list(range(p.N))
        # I1: per table, sum of row gradients = sum_b (sum of bag weights) * G[b, cols_t]
        doff = p.D_offsets
        for t in range(T):
            Dt = int(p.D[t])
            tot = np.zeros(Dt)
            for u in range(int(uc[t]), int(uc[t + 1])):
                tot += rg[rpos[u]: rpos[u] + Dt]
            exp = np.zeros(Dt)
            for b in range(B):
                g = t * B + b
                lo, hi = int(p.offsets[g]), int(p.offsets[g + 1])
                if p.per_sample_weights is not None and p.table_weighted[t]:
                    wsum = float(np.sum(p.per_sample_weights[lo:hi].astype(np.float64)))
                else:
                    wsum = float(hi - lo)
                exp += wsum * p.grad_out[b, doff[t]: doff[t + 1]].astype(np.float64)
            np.testing.assert_allclose(tot, exp, rtol=1e-11, atol=1e-11)
        # I2: adjoint <out, G> = sum_u <row_grad_u, W[row_u]>
        lhs = float(np.sum(out * p.grad_out.astype(np.float64)))
        rhs = 0.0
        for t in range(T):
            Wt = _table_f64(p, w, t)
            Dt = int(p.D[t])
            for u in range(int(uc[t]), int(uc[t + 1])):
                rhs += float(np.dot(rg[rpos[u]: rpos[u] + Dt], Wt[ur[u] - trb[t]]))
        assert abs(lhs - rhs) <= 1e-10 * (1 + abs(lhs))
        # |terms| sums bound the sums
        assert np.all(np.abs(out) <= oabs + 1e-15) and np.all(np.abs(rg) <= rabs + 1e-15)
        # I4: histogram form == gather form, bit for bit, for unweighted fp16 tables
        for t in range(T):
            if int(p.weights_dtype[t]) != DT_F16:
                continue
            if p.per_sample_weights is not None and p.table_weighted[t]:
                continue
            st3, cnt = oracle.histogram_counts(T, B, t, int(p.rows[t]), p.indices, p.offsets, lib=lib)
            assert st3 == 0
            assert np.array_equal(cnt.sum(axis=1), np.diff(p.offsets)[t * B:(t + 1) * B])
            hist = oracle.counts_times_table(cnt, w, p.weights_offsets[t], DT_F16, int(p.D[t]), lib=lib)
            assert np.array_equal(hist, out[:, doff[t]: doff[t + 1]])


def pin_sort_vs_numpy(lib, seed=3):
    rng = np.random.default_rng(seed)
    for _ in range(5):
        T, B = 3, 50
        p = _random_problem(rng, T, B, [DT_F32], False, max_len=30, max_rows=15)
        idx = oracle.backward_indexing(p.layout_arrays(), p.indices, p.offsets, p.B, lib=lib)
        t_of = np.repeat(np.arange(T * B) // B, np.diff(p.offsets))
        keys = p.table_row_base[t_of] + p.indices
        np.testing.assert_array_equal(idx["sorted_pos"], np.argsort(keys, kind="stable"))
        sk = keys[np.argsort(keys, kind="stable")]
        starts = np.nonzero(np.concatenate([[True], sk[1:] != sk[:-1]]))[0]
        np.testing.assert_array_equal(idx["run_starts"][:-1], starts)
        np.testing.assert_array_equal(idx["unique_rows"], sk[starts])


def _nearest_even_codes(x: np.ndarray, pos_codes: np.ndarray, pos_vals: np.ndarray) -> np.ndarray:
    """Nearest representable magnitude by search over the sorted value list;
    ties go to the even code."""
    a = np.abs(x)
    hi = np.clip(np.searchsorted(pos_vals, a), 1, pos_vals.size - 1)
    lo = hi - 1
    dlo, dhi = a - pos_vals[lo], pos_vals[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(pos_codes[lo] % 2 == 0, lo, hi)))
    out = pos_codes[pick].astype(np.uint16)
    return np.where(x < 0, out | 0x8000, out).astype(np.uint16)


def pin_formats(lib, seed=17):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    # decoding: fp16 against numpy's float16, bf16 against the upper half of float32
    f16 = codes.view(np.float16).astype(np.float64)
    dec16 = oracle.decode(codes, oracle.F16, lib=lib)
    fin = np.isfinite(f16)
    np.testing.assert_array_equal(dec16[fin], f16[fin])
    assert np.all(np.isnan(dec16[np.isnan(f16)]))
    with np.errstate(invalid="ignore"):  # NaN codes widen to NaN
        bf = (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    decb = oracle.decode(codes, oracle.BF16, lib=lib)
    finb = np.isfinite(bf)
    np.testing.assert_array_equal(decb[finb], bf[finb])
    # rounding to fp16: exact values, midpoints and random doubles against numpy
    pos16 = np.unique(np.abs(f16[fin]))
    mids = (pos16[1:] + pos16[:-1]) / 2
    rng = np.random.default_rng(seed)
    rnd = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
                          np.nextafter(mids, 0), np.nextafter(mids, 1)])
    xs = np.concatenate([pos16, -pos16, mids, -mids, rnd, [70000.0, 65519.0, 65520.0, -1e-9, 0.0]])
    ours = oracle.round_to(xs, oracle.F16, lib=lib)
    with np.errstate(over="ignore"):  # values past the largest fp16 round to infinity
        ref = xs.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    # rounding to bf16: brute-force nearest representable, ties to even code
    posb = np.unique(np.abs(bf[finb]))
    midb = (posb[1:] + posb[:-1]) / 2
    sel = rng.choice(midb.size, 3000, replace=False)
    xb = np.concatenate([posb[rng.choice(posb.size, 2000, replace=False)], midb[sel],
                         rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)])
    oursb = oracle.round_to(xb, oracle.BF16, lib=lib)
    pos_codes = codes[(codes < 0x7F80)]
    pos_vals = bf[pos_codes.astype(np.int64)]
    want = _nearest_even_codes(xb, pos_codes, pos_vals)
    np.testing.assert_array_equal(oursb, want)
    # rounding to fp32: the nearest fp32 value by exact rational distance among
    # the cast's neighbours, ties to the even code; midpoints of adjacent fp32
    # values (exact in fp64), their neighbours, subnormals and random doubles
    from fractions import Fraction

    f32 = (rng.integers(0, 0x7F7FFFFF, 3000, dtype=np.uint32)).view(np.float32).astype(np.float64)
    nxt = np.nextafter(f32.astype(np.float32), np.float32(np.inf)).astype(np.float64)
    mid32 = (f32 + nxt) / 2
    x32 = np.concatenate([mid32, -mid32, np.nextafter(mid32, 0), np.nextafter(mid32, np.inf), f32,
                          rng.standard_normal(3000) * 10.0 ** rng.integers(-44, 38, 3000),
                          [1.5 * 2.0 ** -149, 2.0 ** -150, 0.0, -0.0]])
    ours32 = oracle.round_to(x32, oracle.F32, lib=lib)
    for x, got in zip(x32, ours32):
        c = np.float32(x)
        cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
        cands = [v for v in cands if np.isfinite(v)]
        dist = [abs(Fraction(float(v)) - Fraction(float(x))) for v in cands]
        best = min(dist)
        near = [v for v, dd in zip(cands, dist) if dd == best]
        want32 = near[0] if len(near) == 1 else [v for v in near if (int(np.float32(v).view(np.uint32)) & 1) == 0][0]
        assert float(got) == float(want32) and (got == 0 or np.signbit(got) == np.signbit(x)), (x, got, want32)
    # past the largest fp32 by half an ulp or more: infinity (ties go to the even code, 2^128)
    big = float(np.finfo(np.float32).max)
    np.testing.assert_array_equal(oracle.round_to(np.array([big + 2.0 ** 103, -(big + 2.0 ** 104)]), oracle.F32, lib=lib),
                                  np.array([np.inf, -np.inf], np.float32))


def pin_special_cases(lib):
    import torch

    # all bags empty: output 0, no runs
    p = make_problem(2, 3, rows=[4, 5], D=[4, 8], weights_dtype=[DT_F32, DT_F16], out_dtype=DT_F32,
                     lengths=np.zeros((2, 3)), ids=[[], []], grad_out=np.ones((3, 12), np.float32))
    w = materialize_weights(p)
    st, out, _ = oracle.problem_forward(p, w, lib=lib)
    assert st == 0 and np.all(out == 0)
    idx, st2, rg, _, _ = oracle.problem_backward(p, lib=lib)
    assert idx["U"] == 0 and rg.size == 0 and list(idx["run_starts"]) == [0]
    # each bag [k]: output rows are copies of W[k]; one id repeated n times gives n*W[k]
    T, B = 1, 5
    tbl = torch.tensor(np.arange(6 * 4, dtype=np.float32).reshape(6, 4) / 8)
    p = make_problem(T, B, rows=[6], D=[4], weights_dtype=[DT_F32], out_dtype=DT_F32,
                     lengths=[[1, 1, 3, 5, 1]], ids=[[2, 0, 4, 4, 4, 1, 1, 1, 1, 1, 5]],
                     grad_out=np.ones((5, 4), np.float32), host_tables={0: tbl})
    w = materialize_weights(p)
    st, out, _ = oracle.problem_forward(p, w, lib=lib)
    W = tbl.numpy().astype(np.float64)
    np.testing.assert_array_equal(out, np.stack([W[2], W[0], 3 * W[4], 5 * W[1], W[5]]))
    # out-of-range and negative ids: reported, contribute nothing
    p = make_problem(1, 2, rows=[6], D=[4], weights_dtype=[DT_F32], out_dtype=DT_F32,
                     lengths=[[3, 2]], ids=[[1, 6, 2, -1, 3]], grad_out=np.ones((2, 4), np.float32),
                     host_tables={0: tbl})
    w = materialize_weights(p)
    st, out, _ = oracle.problem_forward(p, w, lib=lib)
    assert st == oracle.BAD_INDEX
    np.testing.assert_array_equal(out, np.stack([W[1] + W[2], W[3]]))
    idx, st2, rg, _, _ = oracle.problem_backward(p, lib=lib)
    assert idx["status"] == oracle.BAD_INDEX
    np.testing.assert_array_equal(idx["unique_rows"], [1, 2, 3])
    np.testing.assert_array_equal(idx["run_starts"], [0, 1, 2, 3])
    np.testing.assert_array_equal(idx["sorted_pos"], [0, 2, 4, 1, 3])
    # broken offsets are reported: not starting at 0, not ending at N, decreasing
    p = make_problem(1, 3, rows=[6], D=[4], weights_dtype=[DT_F32], out_dtype=DT_F32,
                     lengths=[[2, 2, 1]], ids=[[1, 2, 3, 4, 5]], grad_out=np.ones((3, 4), np.float32),
                     host_tables={0: tbl})
    lay = p.layout_arrays()
    for bad in ([1, 2, 4, 5], [0, 2, 4, 4], [0, 4, 2, 5]):
        st = oracle.forward(lay, w, p.indices, np.array(bad), 3, lib=lib)[0]
        assert st == oracle.BAD_OFFSETS, bad
        st = oracle.backward_indexing(lay, p.indices, np.array(bad), 3, lib=lib)["status"]
        assert st == oracle.BAD_OFFSETS, bad


def _flat_tables(tables):
    return np.array([v for t in tables for row in t for v in row], np.float64)


def pin_optimizer_hand(lib):
    g = json.load(open(os.path.join(GOLDEN, "optimizer_example.json")))
    _, p = _hand_problem(False)
    w = materialize_weights(p)
    lay = p.layout_arrays()
    rows = np.array(g["rows"], np.int64)
    grads = np.array([v for r in g["row_grads"] for v in r], np.float64)
    st, w_new, _ = oracle.exact_update(lay, w, oracle.EXACT_SGD, g["sgd"]["lr"], 0.0, rows, grads, lib=lib)
    assert st == 0
    np.testing.assert_allclose(w_new, _flat_tables(g["sgd"]["expected_tables"]), rtol=1e-15, atol=0)
    for case in ("adagrad", "adagrad_eps"):
        c = g[case]
        mom = np.array(c["momentum_before"], np.float32)
        st, w_new, m_new = oracle.exact_update(lay, w, oracle.EXACT_ROWWISE_ADAGRAD, c["lr"], c["eps"], rows,
                                               grads, momentum=mom, lib=lib)
        assert st == 0
        np.testing.assert_array_equal(m_new, c["expected_momentum"])
        np.testing.assert_allclose(w_new, _flat_tables(c["expected_tables"]), rtol=1e-15, atol=1e-15)


def _opt_problem(rng, T=5, dtypes=(DT_F32, DT_F16, DT_BF16)):
    p = _random_problem(rng, T, 3, list(dtypes), False, max_rows=12)
    w = materialize_weights(p)
    lay = p.layout_arrays()
    total = int(p.table_row_base[-1])
    rows = np.sort(rng.choice(total, size=min(total, 9), replace=False)).astype(np.int64)
    D = p.D.astype(np.int64)
    t_of = np.searchsorted(p.table_row_base, rows, side="right") - 1
    widths = D[t_of]
    grads = rng.standard_normal(int(widths.sum()))
    pos = np.concatenate([[0], np.cumsum(widths)[:-1]]).astype(np.int64)
    return p, w, lay, rows, grads, widths, pos


def pin_optimizer_invariants(lib, trials=20, seed=23):
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        p, w, lay, rows, grads, widths, pos = _opt_problem(rng)
        total = int(p.table_row_base[-1])
        zero = np.zeros(total, np.float32)
        lr = float(rng.uniform(0.01, 2.0))
        st, w0, _ = oracle.exact_update(lay, w, oracle.EXACT_SGD, 0.0, 0.0, rows, grads, lib=lib)
        assert st == 0  # lr 0: the table as stored, in double
        # first Adagrad step from zero momentum, eps 0: |dW_row| = lr * sqrt(D_t), scale-free in g
        st, w1, m1 = oracle.exact_update(lay, w, oracle.EXACT_ROWWISE_ADAGRAD, lr, 0.0, rows, grads,
                                         momentum=zero, lib=lib)
        assert st == 0
        st, w1s, m1s = oracle.exact_update(lay, w, oracle.EXACT_ROWWISE_ADAGRAD, lr, 0.0, rows, 3.5 * grads,
                                           momentum=zero, lib=lib)
        np.testing.assert_allclose(w1s, w1, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(m1s, 12.25 * m1, rtol=1e-13)
        for k, (s0, n) in enumerate(zip(pos, widths)):
            step = np.linalg.norm(w1[s0:s0 + n] - w0[s0:s0 + n])
            np.testing.assert_allclose(step, lr * np.sqrt(n), rtol=1e-12)
        # SGD is linear in the gradient
        g2 = rng.standard_normal(grads.size)
        st, wa, _ = oracle.exact_update(lay, w, oracle.EXACT_SGD, lr, 0.0, rows, grads, lib=lib)
        st, wb, _ = oracle.exact_update(lay, w, oracle.EXACT_SGD, lr, 0.0, rows, g2, lib=lib)
        st, wab, _ = oracle.exact_update(lay, w, oracle.EXACT_SGD, lr, 0.0, rows, grads + g2, lib=lib)
        np.testing.assert_allclose(wab - w0, (wa - w0) + (wb - w0), rtol=1e-12, atol=1e-12)
        assert np.all((wa != w0) == (grads != 0))
        # Adagrad whose denominator sqrt(m) + eps is 1 takes the SGD step (one row at a time;
        # a gradient of 0.5 everywhere has mean square 0.25)
        for k in range(min(3, rows.size)):
            s0, n = int(pos[k]), int(widths[k])
            gk = np.zeros(n) + 0.5  # mean square 0.25
            mom = zero.copy()
            mom[rows[k]] = 0.75  # m after the step = 1.0 -> sqrt = 1, eps 0 -> factor lr
            st, wad, mad = oracle.exact_update(lay, w, oracle.EXACT_ROWWISE_ADAGRAD, lr, 0.0, rows[k:k + 1], gk,
                                               momentum=mom, lib=lib)
            st, wsg, _ = oracle.exact_update(lay, w, oracle.EXACT_SGD, lr, 0.0, rows[k:k + 1], gk, lib=lib)
            assert mad[0] == 1.0
            np.testing.assert_array_equal(wad, wsg)
            mom[rows[k]] = 0.0  # m after = 0.25 -> sqrt 0.5; eps 0.5 makes the denominator 1 again
            st, wad2, _ = oracle.exact_update(lay, w, oracle.EXACT_ROWWISE_ADAGRAD, lr, 0.5, rows[k:k + 1], gk,
                                              momentum=mom, lib=lib)
            np.testing.assert_array_equal(wad2, wsg)
    # duplicating every column (W -> [W, W], g -> [g, g]) keeps momentum and update
    import torch

    tbl = rng.standard_normal((4, 3)).astype(np.float32)
    one = make_problem(1, 1, rows=[4], D=[3], weights_dtype=[DT_F32], out_dtype=DT_F32, lengths=[[0]], ids=[[]],
                       host_tables={0: torch.from_numpy(tbl)})
    two = make_problem(1, 1, rows=[4], D=[6], weights_dtype=[DT_F32], out_dtype=DT_F32, lengths=[[0]], ids=[[]],
                       host_tables={0: torch.from_numpy(np.concatenate([tbl, tbl], axis=1))})
    g = rng.standard_normal(3)
    mom = np.array([0.3, 1.7, 0.0, 2.5], np.float32)
    st, wo, mo = oracle.exact_update(one.layout_arrays(), materialize_weights(one), oracle.EXACT_ROWWISE_ADAGRAD,
                                     0.7, 1e-3, [2], g, momentum=mom, lib=lib)
    st, wt, mt = oracle.exact_update(two.layout_arrays(), materialize_weights(two), oracle.EXACT_ROWWISE_ADAGRAD,
                                     0.7, 1e-3, [2], np.concatenate([g, g]), momentum=mom, lib=lib)
    np.testing.assert_allclose(mt, mo, rtol=1e-15)
    np.testing.assert_allclose(wt, np.concatenate([wo, wo]), rtol=1e-15)
    # a row outside every table is reported
    st, _, _ = oracle.exact_update(one.layout_arrays(), materialize_weights(one), oracle.EXACT_SGD, 1.0, 0.0,
                                   [4], np.ones(3), lib=lib)
    assert st == oracle.BAD_INDEX


ALL_PINS = [pin_hand_example, pin_dense_onehot, pin_invariants, pin_sort_vs_numpy, pin_formats,
            pin_special_cases, pin_mean_hand, pin_mean_dense, pin_optimizer_hand, pin_optimizer_invariants]
