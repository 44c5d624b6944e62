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
                                       ("red_unroll", 6), ("fwd_ring", 2), ("short_item_lookups", 31),
                                       ("fwd_blocks_per_sm", -1), ("long_run_threshold", 0)])
def test_tuning_rejects_out_of_range(lib, field, bad):
    t = tbe.get_tuning()
    with pytest.raises(tbe.TBEError):
        tbe.set_tuning(**{field: bad})
    assert tbe.get_tuning() == t  # a rejected call changes nothing


def test_tuning_round_trip(lib):
    t = tbe.get_tuning()
    assert t["long_chunk"] == 0 and t["fwd_ring"] == 1 and t["red_unroll"] in (4, 8)
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


def test_exact_update_rejects_without_plan(lib):
    opt = tbe.Optimizer(tbe.TBE_OPT_EXACT_SGD, 0.1, 0.0)
    rc = lib.tbe_exact_update(None, ctypes.byref(opt), None, None, None, 0, None, 0, None, None, None)
    assert rc == tbe.TBE_ERR_INVALID_ARG
    rc = lib.tbe_exact_update(None, None, None, None, None, 0, None, 0, None, None, None)
    assert rc == tbe.TBE_ERR_INVALID_ARG
