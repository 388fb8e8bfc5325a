"""GPU test of ec_entropy_decode_noalloc, the allocation-free variant of the entropy decode.

Callers such as a serving runtime's custom-op interface hold only their input and output
buffers and cannot allocate scratch; this entry point uses a library-owned static device
array instead. The test calls it through the C ABI twice in a row and compares each result
with the float64 oracle and with the workspace entry point (ids exact, entropy and
log-confidence within 1e-3, the tolerance of the entropy parity tests). One case takes the
split launch, the one that keeps per-chunk partials and per-row counters in the static
array, and calls it with two different row counts, so that the second call's counters lie
where the first call left partial results: only the call's own clearing of its counters
makes the second result right. It also checks that an oversized request is refused.

This file is collected last, so a run that stops at the first failure has already run every
other test; it passes alone in a fresh process too (the first call sets up the array's
address).
"""
import ctypes

import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

ENT_TOL = 1e-3


@pytest.fixture(scope="module")
def env():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import entropy_gated_kv_gb300 as E

    E.lib()
    return E, torch


def _call_noalloc(E, logits, V, code, n_rows):
    """ec_entropy_decode_noalloc through the C ABI; returns host arrays."""
    import torch

    ids = torch.empty(n_rows, dtype=torch.int32, device="cuda")
    ent = torch.empty(n_rows, dtype=torch.float32, device="cuda")
    conf = torch.empty(n_rows, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = E.lib().ec_entropy_decode_noalloc(ctypes.c_void_p(logits.data_ptr()), logits.stride(0), n_rows, V, code,
                                           ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(ent.data_ptr()),
                                           ctypes.c_void_p(conf.data_ptr()), ctypes.c_void_p(s))
    assert st == 0, E.lib().ec_status_string(st)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), ent.cpu().numpy(), conf.cpu().numpy()


def _compare(got, want):
    np.testing.assert_array_equal(got[0], want[0])
    assert np.max(np.abs(got[1].astype(np.float64) - want[1])) <= ENT_TOL
    assert np.max(np.abs(got[2].astype(np.float64) - want[2])) <= ENT_TOL


def _oracle(lg_bits, dtype):
    ids, ent, conf = O.entropy_decode(O.widen(lg_bits, dtype))
    return ids, ent, conf


def _device(torch, lg, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(lg).view(np.int16)).cuda().view(torch.bfloat16), 1
    return torch.from_numpy(np.ascontiguousarray(lg)).cuda(), 0


@pytest.mark.parametrize("cfg", [2, 1, 3])  # 2, 1: the cluster launch; 3: 78 MB, the streaming launch
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(env, cfg):
    E, torch = env
    w = W.workload(cfg)
    lg = W.step_logits(w).reshape(-1, w.V)
    t, code = _device(torch, lg, w.logits_dtype)
    want = _oracle(lg, w.logits_dtype)
    ids, ent, conf = E.entropy_decode(t)  # the existing entry point, with a workspace
    torch.cuda.synchronize()
    ws_result = (ids.cpu().numpy(), ent.cpu().numpy().astype(np.float64), conf.cpu().numpy().astype(np.float64))
    _compare(ws_result, want)
    first = _call_noalloc(E, t, w.V, code, t.shape[0])
    _compare(first, want)
    _compare(first, ws_result)
    second = _call_noalloc(E, t, w.V, code, t.shape[0])  # the shared array now holds the first call's data
    _compare(second, want)
    _compare(second, ws_result)


def test_noalloc_split_launch_with_changing_row_counts(env):
    # 100 and then 77 rows of a 126464-entry bf16 vocabulary: more rows than the cluster launch
    # takes, under the streaming threshold, so both calls run the split launch with 16 chunk
    # partials per row and one counter per row in the static array. The second call's counters
    # start 19712 bytes in, inside the first call's partials.
    E, torch = env
    w = W.workload(2).scaled(B=4, seed=71)
    lg = W.step_logits(w).reshape(-1, w.V)  # 128 rows, N(0, s^2) with s ~ U[0.5, 8]
    for r0, n in ((0, 100), (37, 77)):
        part = np.ascontiguousarray(lg[r0:r0 + n])
        t, code = _device(torch, part, "bf16")
        want = _oracle(part, "bf16")
        got = _call_noalloc(E, t, w.V, code, n)
        _compare(got, want)
        ids, ent, conf = E.entropy_decode(t)
        torch.cuda.synchronize()
        _compare(got, (ids.cpu().numpy(), ent.cpu().numpy().astype(np.float64), conf.cpu().numpy().astype(np.float64)))


def test_noalloc_refuses_requests_beyond_its_scratch(env):
    E, torch = env
    V = 126464
    # 16 vocabulary chunks per row of this vocabulary: 10000 rows need far more than 1 MiB
    need = E.entropy_decode_workspace_size(10000, V, "bf16")
    assert need > (1 << 20)
    t = torch.zeros(1, V, dtype=torch.bfloat16, device="cuda")  # never read: the call is refused first
    out = torch.empty(10000, dtype=torch.float32, device="cuda")
    st = E.lib().ec_entropy_decode_noalloc(ctypes.c_void_p(t.data_ptr()), V, 10000, V, 1,
                                           ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                           ctypes.c_void_p(out.data_ptr()), None)
    assert st == 2  # EC_ERR_UNSUPPORTED: larger than EC_NOALLOC_SCRATCH_BYTES
