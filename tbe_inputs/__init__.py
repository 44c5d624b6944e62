"""Seeded synthetic inputs for table-batched embedding bags (TBE).

This module only *draws* inputs: packed table layouts, jagged indices/offsets,
per-sample weights, output gradients and table contents.  It contains none of
the operator's arithmetic (no gathers, no pooling, no sorting, no reductions),
so both the CUDA library's tests and the CPU oracle can consume what it makes
without sharing any computation.

Layout conventions (the packed-table format described on the page
"FBTriton table-batched embeddings: the backward win is a threshold moved from
32 to 256", section "A lookup table that is most of the model"):

* all tables live in one byte buffer; table ``t`` starts at byte
  ``weights_offsets[t]`` (256-byte aligned here) and is row-major
  ``[rows_t, D_t]`` in its own dtype;
* ``offsets`` is feature-major with ``T*B + 1`` entries: bag ``(t, b)`` is
  ``indices[offsets[t*B + b] : offsets[t*B + b + 1]]``;
* ids are table-local (``0 <= id < rows_t``);
* ``table_row_base`` is the running sum of table row counts (``[T+1]``) and
  ``D_offsets`` the running sum of table widths (``[T+1]``).

Dtype codes (a data-format convention, not arithmetic): 0 = fp32, 1 = fp16,
2 = bf16.
"""

from .gen import (  # noqa: F401
    DT_F32,
    DT_F16,
    DT_BF16,
    DTYPE_NAMES,
    ELEM_BYTES,
    RUN_BANDS,
    TBEProblem,
    make_problem,
    make_config,
    config_names,
    materialize_weights,
    table_rows,
    table_hash_u32,
)
