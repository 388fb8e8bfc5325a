"""GPU parity of stage (a), the fused softmax / greedy decode / entropy kernel, against the
float64 oracle: decoded ids bit-exact (lowest index on ties), entropy and log-confidence
within 1e-3 absolute."""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import bf16_tensor, to_dev

pytestmark = pytest.mark.gpu

ENT_TOL = 1e-3


@pytest.fixture(scope="module")
def E():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import entropy_gated_kv_gb300 as E

    E.lib()
    return E


def run_gpu(E, stored: np.ndarray, dtype: str, V: int):
    import torch

    t = bf16_tensor(stored) if dtype == "bf16" else to_dev(stored.astype(np.float32))
    ids, ent, conf = E.entropy_decode(t, V=V)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), ent.cpu().numpy().astype(np.float64), conf.cpu().numpy().astype(np.float64)


def check(E, stored, dtype, V, reps=1):
    """Oracle on the given rows; the kernel on the rows repeated `reps` times (many rows take
    the kernel's one-CTA-per-chunk launch, few rows its one-cluster-per-row launch)."""
    x = O.widen(stored[:, :V], dtype)
    ids_o, ent_o, conf_o = O.entropy_decode(x)
    ids_o, ent_o, conf_o = np.tile(ids_o, reps), np.tile(ent_o, reps), np.tile(conf_o, reps)
    ids, ent, conf = run_gpu(E, np.concatenate([stored] * reps) if reps > 1 else stored, dtype, V)
    np.testing.assert_array_equal(ids, ids_o)
    assert np.max(np.abs(ent - ent_o)) <= ENT_TOL, np.max(np.abs(ent - ent_o))
    assert np.max(np.abs(conf - conf_o)) <= ENT_TOL, np.max(np.abs(conf - conf_o))
    return ent_o


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_workload_logits(E, cfg):
    w = W.workload(cfg)
    lg = W.step_logits(w).reshape(-1, w.V)
    check(E, lg, w.logits_dtype, w.V)


def test_trace_logits_high_and_low(E):
    w = W.workload(4)
    for step in (0, 1, 2, 3):
        lg = W.step_logits(w, step).reshape(-1, w.V)
        check(E, lg, "bf16", w.V)


def _bf16(a):
    return W.to_bf16_bits(np.asarray(a, dtype=np.float32))


@pytest.mark.parametrize("reps", [1, 128])
@pytest.mark.parametrize("V", [8192, 16384, 126464, 152064])
def test_ties_across_chunk_boundaries(E, V, reps):
    # maxima tied across the kernel's internal boundaries (8192-element chunks, slices of
    # ceil(V / 8 / 8) * 8 elements) and at the row's ends; the lowest index must win
    rng = np.random.default_rng(V)
    rows = []
    sl = -(-V // 64) * 8
    for pos in [(0, V - 1), (8191, 8192), (8192, 16383 if V > 16383 else V - 1), (V - 2, V - 1), (5, 8192 + 5),
                (sl - 1, sl), (sl, 2 * sl + 3), (7 * sl - 1, V - 1)]:
        x = rng.standard_normal(V).astype(np.float32)
        for p in pos:
            if p < V:
                x[p] = 40.0
        rows.append(x)
    x = rng.standard_normal(V).astype(np.float32)
    x[:] = 3.0  # V-way tie
    rows.append(x)
    x = rng.standard_normal(V).astype(np.float32)
    x[997::997] = 30.0  # ties every 997 elements
    rows.append(x)
    lg = _bf16(np.stack(rows))
    check(E, lg, "bf16", V, reps)


@pytest.mark.parametrize("reps", [1, 128])
@pytest.mark.parametrize("V,stride", [(50257, 50264), (1, 8), (7, 8), (8193, 8200), (32000, 32000)])
def test_ragged_vocab_with_padded_stride(E, V, stride, reps):
    rng = np.random.default_rng(V)
    x = np.full((6, stride), 1e30, dtype=np.float32)  # padding must be ignored
    x[:, :V] = rng.standard_normal((6, V)) * np.array([0.5, 1, 2, 4, 8, 16])[:, None]
    check(E, _bf16(x), "bf16", V, reps)
    xf = np.full((6, stride), 1e30, dtype=np.float32)
    xf[:, :V] = x[:, :V]
    check(E, xf, "f32", V, reps)


def test_neg_inf_one_hot_and_uniform_fp32(E):
    V = 32000
    rows = np.full((4, V), -np.inf, dtype=np.float32)
    rows[0, 123] = 2.0  # one-hot
    rows[1, :] = 0.5  # uniform
    rows[2, [7, 9000, 31999]] = 1.0  # 3-way tie, -inf elsewhere
    rows[3, :] = np.random.default_rng(0).standard_normal(V)
    rows[3, ::3] = -np.inf
    ent_o = check(E, rows, "f32", V)
    assert abs(ent_o[1] - math.log(V)) < 1e-12 and ent_o[0] == 0.0 and abs(ent_o[2] - math.log(3)) < 1e-12


def test_many_rows_and_repeat_with_same_workspace(E):
    import torch

    w = W.workload(2)
    lg = W.step_logits(w).reshape(-1, w.V)
    t = bf16_tensor(np.concatenate([lg] * 9))  # 288 rows
    ws = E.workspace(E.entropy_decode_workspace_size(t.shape[0], w.V, "bf16"))
    a = E.entropy_decode(t, ws=ws)
    b = E.entropy_decode(t, ws=ws)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    assert int(ws.view(torch.uint8).sum()) >= 0


def test_zero_rows_is_a_no_op(E):
    import torch

    t = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    ids, ent, conf = E.entropy_decode(t)
    torch.cuda.synchronize()
    assert ids.numel() == 0
