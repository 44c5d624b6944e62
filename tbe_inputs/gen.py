"""Seeded generators for the five synthetic TBE workloads.

Nothing here computes the operator: the module draws layouts, ids, bag
lengths, per-sample weights, output gradients and table contents.  Table
contents come from a counter-based hash so that any row can be regenerated
bit-identically on the CPU or on a GPU (integer arithmetic only, then one
IEEE fp32 multiply and one round-to-nearest-even cast to the table dtype).

Counter hash: ``lowbias32`` from Chris Wellons' "hash-prospector" (2018):
``x ^= x >> 16; x *= 0x7feb352d; x ^= x >> 15; x *= 0x846ca68b; x ^= x >> 16``
on 32-bit unsigned words.  It is evaluated in int64 tensors with the
multiplications split into 16-bit halves so that no intermediate exceeds
2**49 (no signed overflow on any device).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

DT_F32, DT_F16, DT_BF16 = 0, 1, 2
DTYPE_NAMES = {DT_F32: "f32", DT_F16: "f16", DT_BF16: "bf16"}
ELEM_BYTES = {DT_F32: 4, DT_F16: 2, DT_BF16: 2}
TABLE_ALIGN = 256

_MASK32 = 0xFFFFFFFF


@dataclass
class TBEProblem:
    """One batch of a TBE workload (host arrays) plus how to make its tables."""

    name: str
    T: int
    B: int
    rows: np.ndarray            # int64 [T]
    D: np.ndarray               # int32 [T]
    weights_dtype: np.ndarray   # int32 [T]  (0 fp32, 1 fp16, 2 bf16)
    out_dtype: int
    table_weighted: np.ndarray  # uint8 [T]
    indices: np.ndarray         # int64 [N]
    offsets: np.ndarray         # int64 [T*B + 1]
    per_sample_weights: np.ndarray | None  # float32 [N]
    grad_out: np.ndarray | None  # float32 [B, sum D]
    weight_seed: int
    weight_dist: list = field(default_factory=list)  # per table: ("usym", a) or ("normal", std)
    host_tables: dict = field(default_factory=dict)  # t -> raw table bytes made on the host
    recipe: str = ""
    pooling: int = 0  # 0 sum, 1 mean (each bag's sum divided by its number of lookups)

    # ---- derived layout -------------------------------------------------
    @property
    def N(self) -> int:
        return int(self.indices.shape[0])

    @property
    def table_row_base(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.rows)]).astype(np.int64)

    @property
    def D_offsets(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.D)]).astype(np.int32)

    @property
    def total_D(self) -> int:
        return int(np.sum(self.D))

    @property
    def weights_offsets(self) -> np.ndarray:
        off = np.zeros(self.T, dtype=np.int64)
        cur = 0
        for t in range(self.T):
            off[t] = cur
            nbytes = int(self.rows[t]) * int(self.D[t]) * ELEM_BYTES[int(self.weights_dtype[t])]
            cur += (nbytes + TABLE_ALIGN - 1) // TABLE_ALIGN * TABLE_ALIGN
        return off

    @property
    def weights_bytes(self) -> int:
        t = self.T - 1
        nbytes = int(self.rows[t]) * int(self.D[t]) * ELEM_BYTES[int(self.weights_dtype[t])]
        return int(self.weights_offsets[t]) + (nbytes + TABLE_ALIGN - 1) // TABLE_ALIGN * TABLE_ALIGN

    @property
    def weighted(self) -> bool:
        return self.per_sample_weights is not None

    def bag_lengths(self) -> np.ndarray:
        return np.diff(self.offsets)

    def layout_arrays(self) -> dict:
        return dict(
            T=self.T,
            table_row_base=self.table_row_base,
            D_offsets=self.D_offsets,
            weights_offsets=self.weights_offsets,
            weights_dtype=self.weights_dtype.astype(np.int32),
            table_weighted=self.table_weighted.astype(np.uint8),
            out_dtype=self.out_dtype,
            pooling=self.pooling,
        )


# ---------------------------------------------------------------------------
# counter hash (lowbias32) on int64 torch tensors, exact on every device
# ---------------------------------------------------------------------------

def _mul32(x, m: int):
    lo, hi = m & 0xFFFF, m >> 16
    return ((x * lo) + (((x * hi) & 0xFFFF) << 16)) & _MASK32


def _lowbias32(x):
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def table_hash_u32(seed: int, t: int, rows, cols):
    """32-bit hash words for the elements (rows[:,None], cols[None,:]) of table t.

    ``rows`` and ``cols`` are int64 torch tensors (any device).  Returns an
    int64 tensor of shape [len(rows), len(cols)] with values in [0, 2**32).
    """
    import torch

    base = _lowbias32(torch.tensor((seed * 0x9E37 + 0x1234567) & _MASK32, dtype=torch.int64, device=rows.device))
    base = _lowbias32(base ^ ((t * 0x632B + 0x5BD1E995) & _MASK32))
    r = _lowbias32(base ^ (rows & _MASK32))
    x = (r[:, None] + cols[None, :]) & _MASK32
    return _lowbias32(x)


def _usym_values(h, a: float, dtype_code: int):
    """Map hash words to U(-a, a) and round once to the table dtype."""
    import torch

    k = ((h >> 8) - (1 << 23)).to(torch.float32) * (2.0 ** -23)  # exact, in [-1, 1)
    v = k * torch.tensor(a, dtype=torch.float32, device=h.device)  # one fp32 rounding
    if dtype_code == DT_F32:
        return v
    if dtype_code == DT_F16:
        return v.to(torch.float16)
    return v.to(torch.bfloat16)


_TORCH_DT = None


def _torch_dtype(code):
    import torch

    return {DT_F32: torch.float32, DT_F16: torch.float16, DT_BF16: torch.bfloat16}[code]


def table_rows(p: TBEProblem, t: int, row_ids, device="cpu"):
    """Regenerate rows ``row_ids`` of table ``t`` as a torch tensor in the table dtype."""
    import torch

    code = int(p.weights_dtype[t])
    if t in p.host_tables:
        full = p.host_tables[t]
        ids = torch.as_tensor(np.asarray(row_ids, dtype=np.int64))
        return full[ids].to(device)
    dist = p.weight_dist[t]
    assert dist[0] == "usym"
    rows = torch.as_tensor(np.asarray(row_ids, dtype=np.int64), device=device)
    cols = torch.arange(int(p.D[t]), dtype=torch.int64, device=device)
    h = table_hash_u32(p.weight_seed, t, rows, cols)
    return _usym_values(h, dist[1], code)


def materialize_weights(p: TBEProblem, device="cpu", chunk_elems: int = 1 << 25):
    """Build the packed weight buffer (uint8 tensor) on ``device``."""
    import torch

    buf = torch.zeros(p.weights_bytes, dtype=torch.uint8, device=device)
    woff = p.weights_offsets
    for t in range(p.T):
        code = int(p.weights_dtype[t])
        R, D = int(p.rows[t]), int(p.D[t])
        eb = ELEM_BYTES[code]
        view = buf[int(woff[t]): int(woff[t]) + R * D * eb].view(_torch_dtype(code)).view(R, D)
        if t in p.host_tables:
            view.copy_(p.host_tables[t].to(device))
            continue
        step = max(1, chunk_elems // D)
        for r0 in range(0, R, step):
            r1 = min(R, r0 + step)
            view[r0:r1] = table_rows(p, t, np.arange(r0, r1), device=device)
    return buf


# ---------------------------------------------------------------------------
# id / length samplers
# ---------------------------------------------------------------------------

def _zipf_ids(rng, rows: int, alpha: float, n: int, permute: bool = True) -> np.ndarray:
    """Bounded Zipf over ranks 1..rows, P(k) ~ k^-alpha, by inverse CDF on the
    exact cumulative table; rank -> id through a seeded random permutation
    (permute=False: id = rank - 1, so the hot rows sit next to each other)."""
    perm = rng.permutation(rows).astype(np.int64)
    if not permute:
        perm = np.arange(rows, dtype=np.int64)
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    k = np.arange(1, rows + 1, dtype=np.float64)
    cdf = np.cumsum(k ** (-alpha))
    cdf /= cdf[-1]
    u = rng.random(n)
    r = np.searchsorted(cdf, u, side="right")
    np.minimum(r, rows - 1, out=r)
    return perm[r]


def _band_ids(rng, rows: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n ids of one table whose row multiplicities (run lengths in the
    backward) are drawn uniformly from [lo, hi]; distinct rows are chosen
    at random and the lookups shuffled.  When the remainder is too short to
    start another run it joins a run that stays within hi, so at most one
    run per table falls outside the band."""
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    runs = []
    left = n
    while left > 0:
        k = int(rng.integers(lo, hi + 1))
        if k > left:
            k = left
        runs.append(k)
        left -= k
    if len(runs) > 1 and runs[-1] < lo:
        tail = runs.pop()
        for j in range(len(runs)):  # fold the short tail into a run with room for it
            if runs[j] + tail <= hi:
                runs[j] += tail
                tail = 0
                break
        if tail:
            runs.append(tail)
    if len(runs) > rows:
        raise ValueError("table too small for the requested run lengths")
    rows_used = rng.choice(rows, size=len(runs), replace=False).astype(np.int64)
    ids = np.repeat(rows_used, np.asarray(runs, np.int64))
    return ids[rng.permutation(n)]


# run-length bands of the band workloads (lookups per distinct row)
RUN_BANDS = {"band_short": (1, 3), "band_mid": (32, 255), "band_long": (1024, 4096)}


def _assemble(T, B, lengths_tb, ids_per_table):
    """lengths_tb: [T, B] bag lengths; ids_per_table[t]: ids for table t in bag order."""
    lens = lengths_tb.reshape(-1).astype(np.int64)
    offsets = np.zeros(T * B + 1, dtype=np.int64)
    np.cumsum(lens, out=offsets[1:])
    indices = np.concatenate(ids_per_table).astype(np.int64) if T else np.zeros(0, np.int64)
    assert indices.shape[0] == offsets[-1]
    return indices, offsets


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

# mid_uniform shares mid_skewed's seed: same tables, lengths and empty bags, uniform ids (the control)
CONFIG_SEEDS = {"tiny": 1001, "mid_skewed": 1002, "mixed": 1003, "small_table": 1004, "bwd_skew": 1005,
                "mid_uniform": 1002, "mid_identity": 1002, "band_short": 1007, "band_mid": 1007,
                "band_long": 1007}


def config_names():
    return list(CONFIG_SEEDS)


def make_config(name: str, B: int | None = None, rows_scale: float = 1.0, batch: int = 0,
                seed: int | None = None, with_grad: bool = True) -> TBEProblem:
    """Build one of the named workloads: the five of the method's
    measurements, a uniform-id control and an unpermuted-Zipf sensitivity
    case of the mid-size one, and three
    run-length bands (every distinct row read 1..3, 32..255 or 1024..4096
    times) for mapping where the short/long threshold pays.

    ``B`` and ``rows_scale`` shrink a workload for parity tests; ``batch``
    selects one of several index batches drawn for the same tables.
    """
    seed = CONFIG_SEEDS[name] if seed is None else seed
    lay = np.random.default_rng([seed, 0])
    irng = np.random.default_rng([seed, 1, batch])
    grng = np.random.default_rng([seed, 2, batch])

    def scaled(r):
        return max(1, int(round(r * rows_scale)))

    host_tables = {}
    if name == "tiny":
        T, Bv = 3, (4 if B is None else B)
        rows = np.array([scaled(100), scaled(50), scaled(20)], np.int64)
        D = np.array([8, 16, 4], np.int32)
        wdt = np.full(T, DT_F32, np.int32)
        out_dt = DT_F32
        wdist = [("usym", 0.05)] * T
        while True:
            lens = irng.integers(0, 6, size=(T, Bv))
            if (lens == 0).any():
                break
        ids = [irng.integers(0, rows[t], size=int(lens[t].sum())) for t in range(T)]
        weighted = np.zeros(T, np.uint8)
        recipe = "T=3 fp32 rows 100/50/20 D 8/16/4; L~U{0..5} resampled until one bag is empty; uniform ids"
    elif name in ("mid_skewed", "mid_uniform", "mid_identity"):
        T, Bv = 8, (2048 if B is None else B)
        rows = np.full(T, scaled(100_000), np.int64)
        D = np.full(T, 128, np.int32)
        wdt = np.full(T, DT_F16, np.int32)
        out_dt = DT_F16
        wdist = [("usym", 0.05)] * T
        lens = irng.poisson(20.0, size=(T, Bv))
        empty_b = irng.integers(0, Bv, size=T)
        lens[np.arange(T), empty_b] = 0
        if name == "mid_skewed":
            ids = [_zipf_ids(irng, int(rows[t]), 1.05, int(lens[t].sum())) for t in range(T)]
            how = "ids Zipf(1.05) through a per-table permutation"
        elif name == "mid_identity":
            ids = [_zipf_ids(irng, int(rows[t]), 1.05, int(lens[t].sum()), permute=False) for t in range(T)]
            how = "ids Zipf(1.05) with rank k at id k-1 (hot rows adjacent; sensitivity case)"
        else:
            ids = [irng.integers(0, rows[t], size=int(lens[t].sum())) for t in range(T)]
            how = "uniform ids (control for the skewed workload: same tables and lengths)"
        weighted = np.zeros(T, np.uint8)
        recipe = ("T=8 fp16 100k rows D=128 W~U(-0.05,0.05); B=2048; L~Poisson(20) with one "
                  f"seed-chosen empty bag per table; {how}; fp16 out")
    elif name == "mixed":
        T, Bv = 40, (8192 if B is None else B)
        rows = np.array([scaled(round(math.exp(x))) for x in lay.uniform(math.log(1e4), math.log(1e7), size=T)], np.int64)
        D = lay.choice(np.array([32, 64, 128, 256], np.int32), size=T).astype(np.int32)
        wdt = np.array([DT_F16 if t % 2 == 0 else DT_BF16 for t in range(T)], np.int32)
        out_dt = DT_F32
        wdist = [("usym", 0.05)] * T
        means = np.exp(lay.uniform(0.0, math.log(80.0), size=T))
        wsel = lay.permutation(T)[:20]
        weighted = np.zeros(T, np.uint8)
        weighted[wsel] = 1
        lens = np.stack([irng.poisson(means[t], size=Bv) for t in range(T)])
        ids = [_zipf_ids(irng, int(rows[t]), 1.1, int(lens[t].sum())) for t in range(T)]
        recipe = ("T=40 rows round(exp(U(ln1e4,ln1e7))), D from {32,64,128,256}, fp16 even t / bf16 odd t; "
                  "B=8192; per-table mean length exp(U(0,ln80)), Poisson; ids Zipf(1.1)+perm; "
                  "psw U(0,1) on a seeded set of 20 tables; fp32 out")
    elif name == "small_table":
        T, Bv = 1, (65536 if B is None else B)
        rows = np.array([64], np.int64)
        D = np.array([128], np.int32)
        wdt = np.array([DT_F16], np.int32)
        out_dt = DT_F32
        import torch

        w = (lay.standard_normal((64, 128)) * 0.02).astype(np.float32).astype(np.float16)
        host_tables[0] = torch.from_numpy(w.copy())
        wdist = [("normal", 0.02)]
        lens = irng.integers(64, 513, size=(T, Bv))
        ids = [irng.integers(0, 64, size=int(lens[0].sum()))]
        weighted = np.zeros(T, np.uint8)
        recipe = "T=1 fp16 64x128 W~N(0,0.02); B=65536; L~U{64..512}; uniform ids; fp32 out"
    elif name == "bwd_skew":
        T, Bv = 16, (16384 if B is None else B)
        rows = np.full(T, scaled(1_000_000), np.int64)
        D = np.full(T, 128, np.int32)
        wdt = np.full(T, DT_F32, np.int32)
        out_dt = DT_F32
        wdist = [("usym", 0.05)] * T
        lens = irng.poisson(50.0, size=(T, Bv))
        ids = [_zipf_ids(irng, int(rows[t]), 1.2, int(lens[t].sum())) for t in range(T)]
        weighted = np.zeros(T, np.uint8)
        recipe = "T=16 fp32 1M rows D=128 W~U(-0.05,0.05); B=16384; L~Poisson(50); ids Zipf(1.2)+perm; fp32 out"
    elif name in RUN_BANDS:
        lo, hi = RUN_BANDS[name]
        T, Bv = 8, (8192 if B is None else B)
        rows = np.full(T, scaled(1_000_000), np.int64)
        D = np.full(T, 128, np.int32)
        wdt = np.full(T, DT_F32, np.int32)
        out_dt = DT_F32
        wdist = [("usym", 0.05)] * T
        lens = irng.poisson(20.0, size=(T, Bv))
        ids = [_band_ids(irng, int(rows[t]), int(lens[t].sum()), lo, hi) for t in range(T)]
        weighted = np.zeros(T, np.uint8)
        recipe = (f"T=8 fp32 1M rows D=128 W~U(-0.05,0.05); B=8192; L~Poisson(20); every distinct row "
                  f"read U{{{lo}..{hi}}} times (shuffled over the bags); fp32 out")
    else:
        raise KeyError(name)

    indices, offsets = _assemble(T, Bv, lens, ids)
    psw = None
    if weighted.any():
        psw = irng.random(indices.shape[0]).astype(np.float32)
    grad = None
    if with_grad:
        grad = grng.standard_normal((Bv, int(D.sum()))).astype(np.float32)
    return TBEProblem(name=name, T=T, B=Bv, rows=rows, D=D, weights_dtype=wdt, out_dtype=out_dt,
                      table_weighted=weighted, indices=indices, offsets=offsets,
                      per_sample_weights=psw, grad_out=grad, weight_seed=seed,
                      weight_dist=wdist, host_tables=host_tables, recipe=recipe)


def make_problem(T, B, rows, D, weights_dtype, out_dtype, lengths, ids, psw=None, grad_out=None,
                 table_weighted=None, seed=7, host_tables=None, name="custom", pooling=0) -> TBEProblem:
    """Assemble a problem from explicit per-table lengths [T,B] and id lists."""
    rows = np.asarray(rows, np.int64)
    D = np.asarray(D, np.int32)
    wdt = np.asarray(weights_dtype, np.int32)
    lengths = np.asarray(lengths, np.int64).reshape(T, B)
    indices, offsets = _assemble(T, B, lengths, [np.asarray(x, np.int64) for x in ids])
    tw = np.zeros(T, np.uint8) if table_weighted is None else np.asarray(table_weighted, np.uint8)
    if psw is not None and table_weighted is None:
        tw = np.ones(T, np.uint8)
    return TBEProblem(name=name, T=T, B=B, rows=rows, D=D, weights_dtype=wdt, out_dtype=out_dtype,
                      table_weighted=tw, indices=indices, offsets=offsets,
                      per_sample_weights=None if psw is None else np.asarray(psw, np.float32),
                      grad_out=None if grad_out is None else np.asarray(grad_out, np.float32),
                      weight_seed=seed, weight_dist=[("usym", 0.05)] * T,
                      host_tables=dict(host_tables or {}), recipe="explicit", pooling=int(pooling))
