"""Property tests of the oracle (CPU only, hypothesis): random small layouts,
batches and dtypes, checked against statements that do not go through the
oracle's own loops.

* forward == A_t @ W_t per table, where A_t[b, r] is the summed weight of the
  lookups of bag (t, b) that name row r (numpy float64 matmul);
* row gradients == rows of A_t^T @ G_t for the rows that occur;
* sorted positions == numpy's stable argsort of the keys, unique rows ==
  numpy.unique of the keys, run lengths == their counts;
* one exact SGD step with learning rate lr moves every listed row by exactly
  -lr * g, and a row-wise Adagrad step from zero momentum with eps 0 moves
  each row by lr * sqrt(D_t) in Euclidean norm.
"""

import numpy as np
import pytest

import oracle
from tbe_inputs import DT_BF16, DT_F16, DT_F32, make_problem, materialize_weights

hyp = pytest.importorskip("hypothesis")
st = hyp.strategies
given, settings = hyp.given, hyp.settings


@st.composite
def problems(draw):
    T = draw(st.integers(1, 4))
    B = draw(st.integers(1, 6))
    rows = draw(st.lists(st.integers(1, 7), min_size=T, max_size=T))
    D = draw(st.lists(st.sampled_from([1, 2, 3, 4, 8]), min_size=T, max_size=T))
    dts = draw(st.lists(st.sampled_from([DT_F32, DT_F16, DT_BF16]), min_size=T, max_size=T))
    lens = [[draw(st.integers(0, 5)) for _ in range(B)] for _ in range(T)]
    ids = [[draw(st.integers(0, rows[t] - 1)) for _ in range(sum(lens[t]))] for t in range(T)]
    N = sum(sum(x) for x in lens)
    weighted = draw(st.booleans()) and N > 0
    psw = np.array([draw(st.floats(-2, 2, width=32)) for _ in range(N)], np.float32) if weighted else None
    tw = np.array([draw(st.integers(0, 1)) for _ in range(T)], np.uint8) if weighted else None
    seed = draw(st.integers(0, 1 << 20))
    G = np.random.default_rng(seed).standard_normal((B, sum(D))).astype(np.float32)
    return make_problem(T, B, rows=rows, D=D, weights_dtype=dts, out_dtype=DT_F32, lengths=lens, ids=ids,
                        psw=psw, grad_out=G, table_weighted=tw, seed=seed)


def _table(p, w, t):
    """Table t decoded with numpy's own formats (float64)."""
    R, D, off = int(p.rows[t]), int(p.D[t]), int(p.weights_offsets[t])
    dt = int(p.weights_dtype[t])
    raw = np.asarray(w)[off: off + R * D * (4 if dt == DT_F32 else 2)]
    if dt == DT_F32:
        return raw.view(np.float32).astype(np.float64).reshape(R, D)
    if dt == DT_F16:
        return raw.view(np.float16).astype(np.float64).reshape(R, D)
    return (raw.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(R, D)


def _onehot(p, t):
    A = np.zeros((p.B, int(p.rows[t])))
    weighted = p.per_sample_weights is not None and bool(p.table_weighted[t])
    for b in range(p.B):
        g = t * p.B + b
        for i in range(int(p.offsets[g]), int(p.offsets[g + 1])):
            A[b, int(p.indices[i])] += float(p.per_sample_weights[i]) if weighted else 1.0
    return A


@settings(max_examples=60, deadline=None)
@given(problems())
def test_forward_and_backward_are_the_dense_products(p):
    w = materialize_weights(p).numpy()
    st_, out, _ = oracle.problem_forward(p, w)
    assert st_ == 0
    idx, st2, rg, _, pos = oracle.problem_backward(p)
    assert st2 == 0
    doff = p.D_offsets
    G = p.grad_out.astype(np.float64)
    ur = idx["unique_rows"]
    for t in range(p.T):
        A = _onehot(p, t)
        W = _table(p, w, t)
        np.testing.assert_allclose(out[:, doff[t]:doff[t + 1]], A @ W, rtol=1e-12, atol=1e-12)
        full = A.T @ G[:, doff[t]:doff[t + 1]]
        base = int(p.table_row_base[t])
        for k in np.nonzero((ur >= base) & (ur < base + int(p.rows[t])))[0]:
            r = int(ur[k]) - base
            np.testing.assert_allclose(rg[pos[k]: pos[k] + int(p.D[t])], full[r], rtol=1e-12, atol=1e-12)


@settings(max_examples=60, deadline=None)
@given(problems())
def test_indexing_is_the_stable_sort(p):
    idx = oracle.backward_indexing(p.layout_arrays(), p.indices, p.offsets, p.B)
    keys = np.empty(p.N, np.int64)
    for t in range(p.T):
        a, b = int(p.offsets[t * p.B]), int(p.offsets[(t + 1) * p.B])
        keys[a:b] = p.indices[a:b] + int(p.table_row_base[t])
    np.testing.assert_array_equal(idx["sorted_pos"], np.argsort(keys, kind="stable"))
    u, c = np.unique(keys, return_counts=True)
    np.testing.assert_array_equal(idx["unique_rows"], u)
    np.testing.assert_array_equal(np.diff(idx["run_starts"]), c)
    np.testing.assert_array_equal(idx["unique_count"], np.searchsorted(u, p.table_row_base))


@settings(max_examples=40, deadline=None)
@given(problems(), st.floats(0.01, 4.0))
def test_update_steps(p, lr):
    w = materialize_weights(p).numpy()
    lay = p.layout_arrays()
    total = int(p.table_row_base[-1])
    rows = np.arange(total, dtype=np.int64)
    t_of = np.searchsorted(p.table_row_base, rows, side="right") - 1
    widths = p.D[t_of].astype(np.int64)
    g = np.random.default_rng(total).standard_normal(int(widths.sum())) + 0.1
    _, w0, _ = oracle.exact_update(lay, w, oracle.EXACT_SGD, 0.0, 0.0, rows, g)
    _, w1, _ = oracle.exact_update(lay, w, oracle.EXACT_SGD, lr, 0.0, rows, g)
    np.testing.assert_allclose(w1 - w0, -lr * g, rtol=1e-12, atol=1e-12)
    _, w2, m2 = oracle.exact_update(lay, w, oracle.EXACT_ROWWISE_ADAGRAD, lr, 0.0, rows, g,
                                    momentum=np.zeros(total, np.float32))
    starts = np.concatenate([[0], np.cumsum(widths)[:-1]])
    for s0, n in zip(starts, widths):
        np.testing.assert_allclose(np.linalg.norm(w2[s0:s0 + n] - w0[s0:s0 + n]), lr * np.sqrt(n), rtol=1e-12)
