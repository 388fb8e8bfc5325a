"""GPU parity of the partial forward of one transformer layer (ec_layer_forward) against the
float64 oracle: the forward the step's flag selects (EntropyCache, gist.science zh summary
§2.2, partial forward: only the recompute set is recomputed, the rest is read from the K/V
cache), for the LLaMA-style layers of the evaluated models.

Checked: the refreshed cache rows (within the bf16 tolerance; every other row bit-exact and
untouched) and the layer output of the recompute rows, per row ||y - y_ref|| <= 2e-2 ||y_ref||
and per element |y - y_ref| <= 2e-2 (|y_ref| + rms(y_ref)) (the attention tolerance: the layer
rounds every intermediate to bf16). The RoPE table is checked against its closed form.
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import bf16_bits, bf16_tensor, to_dev

pytestmark = pytest.mark.gpu
RTOL = 2e-2


@pytest.fixture(scope="module")
def E():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import entropy_gated_kv_gb300 as E

    E.lib()
    return E


def rows_close(got, ref, rtol=RTOL):
    """Per row Frobenius and per element checks (got, ref: [R, n] float64)."""
    for r in range(ref.shape[0]):
        nr = np.linalg.norm(ref[r])
        rel = np.linalg.norm(got[r] - ref[r]) / max(nr, 1e-30)
        if not rel <= rtol:
            return False, f"row {r}: relative error {rel:.3e}"
        rms = math.sqrt(float(np.mean(ref[r] ** 2)))
        bad = np.abs(got[r] - ref[r]) > rtol * (np.abs(ref[r]) + rms)
        if bad.any():
            i = int(np.argwhere(bad)[0][0])
            return False, f"row {r} elem {i}: {got[r, i]} vs {ref[r, i]}"
    return True, "ok"


def test_rope_table_closed_form(E):
    import torch

    for L, D, theta in ((1024, 128, 500000.0), (300, 64, 10000.0), (5, 2, 1.0)):
        cs, sn = E.rope_table(L, D, theta)
        torch.cuda.synchronize()
        ang = np.arange(L)[:, None] * float(np.float32(theta)) ** (-2.0 * np.arange(D // 2) / D)[None, :]
        np.testing.assert_allclose(cs.cpu().numpy(), np.cos(ang), atol=2e-7)
        np.testing.assert_allclose(sn.cpu().numpy(), np.sin(ang), atol=2e-7)


def run_layer(E, *, B, L, Hq, Hkv, D, d_ff, theta, idx_list, sample=None, seed=0):
    import torch

    d = Hq * D
    p = E.Params(B=B, L=L, Hq=Hq, Hkv=Hkv, D=D, V=8, C_max=1, k=1)
    wts = W.layer_weights(d, Hq, Hkv, D, d_ff, seed=seed)
    x_src = W.layer_input(B, L, d, seed=seed)
    rng = np.random.default_rng(seed)
    kc = W.to_bf16_bits(rng.standard_normal((B, L, Hkv, D), dtype=np.float32))
    vc = W.to_bf16_bits(rng.standard_normal((B, L, Hkv, D), dtype=np.float32))
    cs, sn = E.rope_table(L, D, theta)
    w = E.LayerWeights(**{n: bf16_tensor(wts[n]) for n in wts}, rope_cos=cs, rope_sin=sn, eps=1e-5)
    idx = np.zeros((B, L), dtype=np.int32)
    R = np.zeros(B, dtype=np.int32)
    for b, ids in enumerate(idx_list):
        idx[b, : len(ids)] = ids
        R[b] = len(ids)
    k_dev, v_dev = bf16_tensor(kc), bf16_tensor(vc)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = E.layer_forward(p, w, to_dev(idx), to_dev(R), bf16_tensor(x_src), k_dev, v_dev, dev_err=dev_err)
    status, word = E.read_device_error(dev_err)
    assert status == 0, f"device error word {word:#x}"
    y_g = O.widen(bf16_bits(y), "bf16")
    kc_g, vc_g = bf16_bits(k_dev), bf16_bits(v_dev)
    W64 = {n: O.widen(wts[n], "bf16") for n in wts}
    for b, ids in enumerate(idx_list):
        ids = np.asarray(ids, dtype=np.int64)
        rows = None if sample is None or len(ids) <= sample else np.sort(rng.choice(len(ids), sample, replace=False))
        o = O.layer_forward(x_src=O.widen(x_src[b], "bf16"), idx=ids, k_cache=O.widen(kc[b], "bf16"),
                            v_cache=O.widen(vc[b], "bf16"), weights=W64, Hq=Hq, Hkv=Hkv,
                            theta=float(np.float32(theta)), eps=1e-5, rows=rows)
        # cache rows outside the recompute set are untouched; inside, the fresh k / v
        other = np.setdiff1d(np.arange(L), ids)
        np.testing.assert_array_equal(kc_g[b][other], kc[b][other])
        np.testing.assert_array_equal(vc_g[b][other], vc[b][other])
        for name, got, ref in (("k", kc_g[b][ids], o["k"]), ("v", vc_g[b][ids], o["v"])):
            ok, msg = rows_close(O.widen(got, "bf16").reshape(len(ids), -1), ref.reshape(len(ids), -1))
            assert ok, f"b={b} {name}: {msg}"
        ok, msg = rows_close(y_g[b][o["rows"]], o["y"])
        assert ok, f"b={b} y: {msg}"


def _llada_partial_idx():
    # the recompute set of the LLaDA-8B layer step (workload 2): 31 masked positions + the last 64
    w = W.workload(2)
    st = W.snapshot_state(w)
    x = O.widen(W.step_logits(w)[0], w.logits_dtype)
    o = O.step(logits=x, cand_pos=st["cand_pos"][0], cand_count=int(st["cand_count"][0]), tokens=st["tokens"][0],
               mask=st["mask"][0], ring=st["ring"][0], ring_head=int(st["ring_head"][0]),
               ring_count=int(st["ring_count"][0]), n_dec=w.n_dec, tau=w.tau)
    assert not o["flag"] and o["R"] == 95
    return o["idx"]


def test_llada_layer_partial_forward(E):
    run_layer(E, B=1, L=1024, Hq=32, Hkv=32, D=128, d_ff=12288, theta=500000.0, idx_list=[_llada_partial_idx()])


def test_llada_layer_full_forward(E):
    run_layer(E, B=1, L=1024, Hq=32, Hkv=32, D=128, d_ff=12288, theta=500000.0, idx_list=[np.arange(1024)],
              sample=32, seed=1)


def test_gqa_two_sequences_ragged(E):
    # Hq 8 / Hkv 2 x 64 (two heads per 128-feature tile), L 300 (two row blocks, the second
    # ragged), one sequence full and one partial with scattered rows
    rng = np.random.default_rng(5)
    part = np.sort(rng.choice(300, 77, replace=False))
    run_layer(E, B=2, L=300, Hq=8, Hkv=2, D=64, d_ff=1024, theta=10000.0, idx_list=[np.arange(300), part], seed=2)


def test_dream_shape_partial_forward(E):
    # Dream-7B's layer shape: d 3584 (28 x 128), 4 KV heads, d_ff 18944, two sequences
    rng = np.random.default_rng(6)
    ids = [np.sort(rng.choice(2048, 95, replace=False)), np.arange(1900, 2048)]
    run_layer(E, B=2, L=2048, Hq=28, Hkv=4, D=128, d_ff=18944, theta=1000000.0, idx_list=ids, seed=3)
