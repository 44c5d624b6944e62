"""The backward for callers that cannot allocate device memory (GPU).

Some callers -- a plugin that an engine hands only a stream and its tensors --
cannot provide a workspace.  tbe_backward_static_workspace() serves them from
an array compiled into the library.  This file checks, through the C ABI,
that two calls in a row give the same rows, run boundaries, sorted positions
and row gradients as tbe_backward() with a caller workspace, that the second
call leaves the device's allocated and free memory unchanged, and that a
batch too large for the array is refused.  It is collected last so that a run that
stops at the first failure has already run every other test; it also passes
on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest

import parity
from tbe_inputs import make_config

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tbe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import table_embedding_bags_gb300 as m

    m.load_library()
    return m


def _outputs(bufs, N):
    U = int(bufs.unique_count[-1].item())
    return dict(U=U, unique_count=bufs.unique_count.cpu().numpy(),
                unique_rows=bufs.unique_rows[:U].cpu().numpy(),
                run_starts=bufs.run_starts[:U + 1].cpu().numpy(),
                sorted_positions=bufs.sorted_positions[:N].cpu().numpy(),
                row_grads=bufs.row_grads[:U * 128].cpu().numpy().astype(np.float64))


def test_static_workspace_matches_caller_workspace(tbe):
    p = make_config("mid_skewed")
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    assert tbe.tbe_backward_workspace_bytes(plan, p.B, p.N) <= tbe.TBE_STATIC_WORKSPACE_BYTES
    ref_bufs = tbe.BackwardBuffers(plan, p.B, p.N)
    tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, bufs=ref_bufs)
    torch.cuda.synchronize()
    ref = _outputs(ref_bufs, p.N)
    lib = tbe.load_library()
    outs = [tbe.BackwardBuffers(plan, p.B, p.N, with_workspace=False) for _ in range(2)]
    statuses = [torch.zeros(1, dtype=torch.int32, device="cuda") for _ in range(2)]
    for call in range(2):  # the array keeps the previous call's contents
        bufs, status = outs[call], statuses[call]
        assert bufs.workspace is None
        torch.cuda.synchronize()
        if call == 1:  # after the first call (which looks up the array's address): nothing is allocated
            used_before, free_before = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
        rc = lib.tbe_backward_static_workspace(
            plan.handle, ctypes.c_void_p(d["grad"].data_ptr()), ctypes.c_void_p(d["indices"].data_ptr()), p.N,
            ctypes.c_void_p(d["offsets"].data_ptr()), p.B, None, ctypes.c_void_p(bufs.unique_rows.data_ptr()),
            ctypes.c_void_p(bufs.run_starts.data_ptr()), ctypes.c_void_p(bufs.sorted_positions.data_ptr()),
            ctypes.c_void_p(bufs.row_grads.data_ptr()), bufs.row_grads_capacity,
            ctypes.c_void_p(bufs.unique_count.data_ptr()), ctypes.c_void_p(status.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == tbe.TBE_OK, f"call {call}: {tbe.load_library().tbe_status_string(rc)}"
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.memory_allocated() == used_before
            assert torch.cuda.mem_get_info()[0] == free_before
        assert int(status.item()) == 0
        got = _outputs(bufs, p.N)
        assert got["U"] == ref["U"]
        for k in ("unique_count", "unique_rows", "run_starts", "sorted_positions"):
            np.testing.assert_array_equal(got[k], ref[k], err_msg=f"call {call}: {k}")
        # same tolerance as the parity tests: |a - b| <= 1e-5 * |b| per element
        np.testing.assert_allclose(got["row_grads"], ref["row_grads"], rtol=1e-5, atol=0,
                                   err_msg=f"call {call}: row_grads")


def test_static_workspace_refuses_too_large(tbe):
    p = make_config("bwd_skew", B=4096, rows_scale=0.01, with_grad=False)
    plan = tbe.Plan.from_problem(p)
    assert tbe.tbe_backward_workspace_bytes(plan, p.B, p.N) > tbe.TBE_STATIC_WORKSPACE_BYTES
    lib = tbe.load_library()
    rc = lib.tbe_backward_static_workspace(plan.handle, None, None, p.N, None, p.B, None, None, None, None,
                                           None, 0, None, None, None)
    assert rc == tbe.TBE_ERR_WORKSPACE
