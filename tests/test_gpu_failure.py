"""The failure path on the GPU, without faulting or hanging it: a bounded wait on a barrier
phase that nothing completes gives up after its limit, reports EC_DEVERR_TIMEOUT through the
device error word, and the context stays usable (a decode afterwards matches the oracle).
The wait is the same bounded mbarrier wait every kernel of the library uses."""
import time

import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import entropy_gated_kv_gb300 as E

    E.lib()
    return E


def test_bounded_wait_times_out_and_the_context_survives(E):
    import torch

    from entropy_gated_kv_gb300 import _capi as C

    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    E.selftest_bounded_wait(dev_err, 20_000_000)  # 20 ms
    status, word = E.read_device_error(dev_err)
    elapsed = time.perf_counter() - t0
    assert status == C.EC_ERR_TIMEOUT, (status, word)
    assert word & C.EC_DEVERR_TIMEOUT
    assert 0.015 <= elapsed < 5.0, elapsed  # it waited about its limit, then returned

    # the context still works
    rng = np.random.default_rng(0)
    x = rng.standard_normal((4, 5000)).astype(np.float32)
    ids, ent, conf = (t.cpu().numpy() for t in E.entropy_decode(torch.from_numpy(x).cuda()))
    ids_o, ent_o, conf_o = O.entropy_decode(x.astype(np.float64))
    np.testing.assert_array_equal(ids, ids_o)
    assert np.max(np.abs(ent - ent_o)) <= 1e-3


def test_read_floor_reads_without_side_effects():
    # the measurement aid reads the buffer and leaves the sink alone (it keeps the loads only)
    import torch

    import entropy_gated_kv_gb300 as E

    buf = torch.arange(3 * 4096 + 8, dtype=torch.int32, device="cuda")  # ragged: not a whole number of CTAs
    sink = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    E.read_floor(buf, sink)
    torch.cuda.synchronize()
    assert int(sink.item()) == 7
