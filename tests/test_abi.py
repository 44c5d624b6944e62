"""The C-ABI library builds, loads and exports every declared symbol (CPU only)."""

import ctypes
import os
import re

import pytest

import table_embedding_bags_gb300 as tbe
from table_embedding_bags_gb300.build import INCLUDE, build

HEADER = os.path.join(INCLUDE, "tbe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(tbe_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build()
    return tbe.load_library()


def test_header_matches_binding_list():
    assert declared_functions() == sorted(tbe.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_host_only_calls(lib):
    assert lib.tbe_plan_device_bytes(1) == 256
    assert lib.tbe_plan_device_bytes(0) == 0
    assert lib.tbe_plan_device_bytes(tbe.TBE_MAX_TABLES + 1) == 0
    assert lib.tbe_status_string(tbe.TBE_ERR_WORKSPACE) == b"workspace too small"
    assert b"sm_103a" in lib.tbe_version()
    t = tbe.get_tuning()
    assert t["long_run_threshold"] >= 1 and t["fwd_unroll"] in (4, 8)
    with pytest.raises(tbe.TBEError):
        tbe.set_tuning(fwd_unroll=3)
    with pytest.raises(tbe.TBEError):
        tbe.set_tuning(long_chunk=33)
    assert tbe.get_tuning() == t


@pytest.mark.parametrize("field,bad", [("fwd_lanes_per_row", 3), ("fwd_lanes_per_row", 64), ("fwd_lanes_per_row", 0),
                                       ("red_unroll", 6), ("fwd_ring", 4), ("short_item_lookups", 31),
                                       ("fwd_blocks_per_sm", -1), ("long_run_threshold", 0)])
def test_tuning_rejects_out_of_range(lib, field, bad):
    t = tbe.get_tuning()
    with pytest.raises(tbe.TBEError):
        tbe.set_tuning(**{field: bad})
    assert tbe.get_tuning() == t  # a rejected call changes nothing


def test_tuning_round_trip(lib):
    t = tbe.get_tuning()
    assert t["long_chunk"] == 0 and t["fwd_ring"] == 3 and t["red_unroll"] in (4, 8)
    try:
        tbe.set_tuning(long_chunk=128, short_item_lookups=64, fwd_lanes_per_row=8, red_unroll=8, fwd_ring=0)
        u = tbe.get_tuning()
        assert (u["long_chunk"], u["short_item_lookups"], u["fwd_lanes_per_row"], u["red_unroll"], u["fwd_ring"]) == \
            (128, 64, 8, 8, 0)
    finally:
        tbe.set_tuning(**t)
    assert tbe.get_tuning() == t
    # null arguments are rejected on the host before any CUDA call
    assert lib.tbe_plan_create(None, None, 0, None, None) == tbe.TBE_ERR_INVALID_ARG
    assert lib.tbe_forward(None, None, None, 0, None, 0, None, None, None, None) == tbe.TBE_ERR_INVALID_ARG
    assert lib.tbe_backward_workspace_bytes(None, 1, 1) == 0
    # the bounded-wait self-test checks its arguments before any CUDA call
    assert lib.tbe_wait_selftest(2, 10, None, None) == tbe.TBE_ERR_INVALID_ARG
    assert lib.tbe_wait_selftest(0, 0, None, None) == tbe.TBE_ERR_INVALID_ARG


def test_exact_update_rejects_without_plan(lib):
    opt = tbe.Optimizer(tbe.TBE_OPT_EXACT_SGD, 0.1, 0.0)
    rc = lib.tbe_exact_update(None, ctypes.byref(opt), None, None, None, 0, None, 0, None, None, None)
    assert rc == tbe.TBE_ERR_INVALID_ARG
    rc = lib.tbe_exact_update(None, None, None, None, None, 0, None, 0, None, None, None)
    assert rc == tbe.TBE_ERR_INVALID_ARG


def _layout(T, trb, doff, woff, wdt, out_dtype=0, pooling=0):
    import numpy as np

    keep = [np.ascontiguousarray(trb, np.int64), np.ascontiguousarray(doff, np.int32),
            np.ascontiguousarray(woff, np.int64), np.ascontiguousarray(wdt, np.int32)]
    L = tbe._Layout(T, *(a.ctypes.data for a in keep), None, out_dtype, pooling)
    return L, keep


# layouts that tbe_plan_create must refuse before it touches the device
BAD_LAYOUTS = {
    "no_tables": (dict(T=0, trb=[0], doff=[0], woff=[], wdt=[]), tbe.TBE_ERR_INVALID_ARG),
    "too_many_tables": (dict(T=tbe.TBE_MAX_TABLES + 1, trb=[0, 1], doff=[0, 4], woff=[0], wdt=[0]),
                        tbe.TBE_ERR_INVALID_ARG),
    "row_base_not_zero": (dict(T=1, trb=[5, 10], doff=[0, 4], woff=[0], wdt=[0]), tbe.TBE_ERR_INVALID_ARG),
    "rows_decrease": (dict(T=2, trb=[0, 10, 4], doff=[0, 4, 8], woff=[0, 256], wdt=[0, 0]),
                      tbe.TBE_ERR_INVALID_ARG),
    "zero_width": (dict(T=2, trb=[0, 10, 20], doff=[0, 4, 4], woff=[0, 256], wdt=[0, 0]), tbe.TBE_ERR_INVALID_ARG),
    "unknown_dtype": (dict(T=1, trb=[0, 10], doff=[0, 4], woff=[0], wdt=[7]), tbe.TBE_ERR_INVALID_ARG),
    "unknown_out_dtype": (dict(T=1, trb=[0, 10], doff=[0, 4], woff=[0], wdt=[0], out_dtype=9),
                          tbe.TBE_ERR_INVALID_ARG),
    "unknown_pooling": (dict(T=1, trb=[0, 10], doff=[0, 4], woff=[0], wdt=[0], pooling=2), tbe.TBE_ERR_INVALID_ARG),
    "row_not_16_bytes": (dict(T=1, trb=[0, 10], doff=[0, 3], woff=[0], wdt=[0]), tbe.TBE_ERR_UNSUPPORTED),
    "half_row_not_16_bytes": (dict(T=1, trb=[0, 10], doff=[0, 4], woff=[0], wdt=[1]), tbe.TBE_ERR_UNSUPPORTED),
    "table_not_aligned": (dict(T=2, trb=[0, 10, 20], doff=[0, 4, 8], woff=[0, 8], wdt=[0, 0]),
                          tbe.TBE_ERR_UNSUPPORTED),
    "rows_beyond_int32": (dict(T=1, trb=[0, 1 << 31], doff=[0, 4], woff=[0], wdt=[0]), tbe.TBE_ERR_UNSUPPORTED),
}


@pytest.mark.parametrize("name", sorted(BAD_LAYOUTS))
def test_plan_create_refuses_bad_layouts(lib, name):
    kw, want = BAD_LAYOUTS[name]
    L, _keep = _layout(kw["T"], kw["trb"], kw["doff"], kw["woff"], kw["wdt"], kw.get("out_dtype", 0), kw.get("pooling", 0))
    meta = (ctypes.c_uint8 * (1 << 20))()
    base = (ctypes.addressof(meta) + 15) // 16 * 16
    h = ctypes.c_void_p()
    rc = lib.tbe_plan_create(ctypes.byref(L), ctypes.c_void_p(base), (1 << 20) - 16, None, ctypes.byref(h))
    assert rc == want and not h.value


def test_plan_create_checks_its_metadata_buffer(lib):
    L, _keep = _layout(1, [0, 10], [0, 4], [0], [0])
    meta = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(meta) + 15) // 16 * 16
    h = ctypes.c_void_p()
    need = lib.tbe_plan_device_bytes(1)
    assert lib.tbe_plan_create(ctypes.byref(L), None, need, None, ctypes.byref(h)) == tbe.TBE_ERR_INVALID_ARG
    assert lib.tbe_plan_create(ctypes.byref(L), ctypes.c_void_p(base), need - 1, None,
                               ctypes.byref(h)) == tbe.TBE_ERR_INVALID_ARG
    assert lib.tbe_plan_create(ctypes.byref(L), ctypes.c_void_p(base + 4), need, None,
                               ctypes.byref(h)) == tbe.TBE_ERR_INVALID_ARG


def test_argument_checks_before_the_abi():
    """The binding's tensor checks (no GPU needed: host tensors are refused
    first, then dtype and size)."""
    import torch

    import table_embedding_bags_gb300 as tbe

    with pytest.raises(tbe.TBEError, match="CUDA"):
        tbe._need(torch.zeros(4, dtype=torch.int64), (torch.int64,), 4, "indices")
    with pytest.raises(tbe.TBEError, match="required"):
        tbe._need(None, (torch.int64,), 4, "indices")
    tbe._need(None, (torch.float32,), 4, "per_sample_weights", optional=True)
