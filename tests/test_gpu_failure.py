"""Failure reporting on the GPU without a fault: the library's bounded waits
give up and report TBE_DEV_TIMEOUT instead of hanging, and the device keeps
working afterwards (GPU).

A wait is made to run out by pointing it at something nothing completes (a
look-back word no kernel publishes, an mbarrier nobody arrives on) with a
short poll limit; nothing traps and no copy is left in flight.
"""

import numpy as np
import pytest

import oracle
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


@pytest.mark.parametrize("kind", [0, 1], ids=["lookback_word", "mbarrier"])
def test_bounded_wait_times_out_and_device_stays_usable(tbe, kind):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tbe.wait_selftest(kind, 1000, st)
    torch.cuda.synchronize()
    assert int(st.item()) == tbe.TBE_DEV_TIMEOUT
    # the same context runs a forward and a backward correctly afterwards
    p = make_config("tiny")
    w_dev, w_host = parity.weights_pair(p)
    d = parity.upload(p)
    plan = tbe.Plan.from_problem(p)
    st.zero_()
    out = tbe.tbe_forward(plan, w_dev, d["indices"], d["offsets"], p.B, dev_status=st)
    bufs = tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ost, ref, ref_abs = oracle.problem_forward(p, w_host)
    assert ost == 0
    parity.compare_forward(p, parity.to_f64(out), ref, ref_abs)
    idx = oracle.backward_indexing(p.layout_arrays(), p.indices, p.offsets, p.B)
    U = int(bufs.unique_count[-1].item())
    assert U == idx["U"]
    assert np.array_equal(bufs.unique_rows[:U].cpu().numpy(), idx["unique_rows"])


def test_selftest_rejects_bad_arguments(tbe):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for kind, polls in [(2, 10), (-1, 10), (0, 0), (1, (1 << 20) + 1)]:
        with pytest.raises(tbe.TBEError):
            tbe.wait_selftest(kind, polls, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
