"""GPU parity of one whole EntropyCache step (ec_step) against the float64 oracle on the
seeded workloads: committed positions and tokens, mask, history, flags, recompute set and the
refreshed caches bit for bit; E within 1e-3; attention within the bf16 tolerance.

Exemptions (the fp32 kernel and the fp64 oracle may round a near-tie differently):
  - a sequence's flag, and the recompute set that depends on it, when |E_oracle - tau| <= 1e-4;
  - the committed set when the oracle's n_dec-th and next confidence differ by <= 1e-5: the
    device's choice must lie in the tied band, and the oracle then adopts it (teacher forcing)
    so that the mask, history, gate, recompute set, caches and attention are still checked.
Each exemption is reported; the seeded workloads hit none of them.
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import attention_close, bf16_bits, bf16_tensor, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import entropy_gated_kv_gb300 as E

    E.lib()
    return E


def params_of(E, w):
    return E.Params(B=w.B, L=w.L, Hq=w.Hq, Hkv=w.Hkv, D=w.D, V=w.V, C_max=w.C_max, k=w.k, n_dec=w.n_dec, tau=w.tau,
                    logits_dtype=w.logits_dtype)


def run_and_check(E, w, st_h, lg, lay, sample_rows=None, seed=0):
    import torch

    p = params_of(E, w)
    st = E.DecodeState.from_arrays(p, tokens=st_h["tokens"], mask=st_h["mask"], ring=st_h["ring"],
                                   ring_head=st_h["ring_head"], ring_count=st_h["ring_count"])
    logits = bf16_tensor(lg) if w.logits_dtype == "bf16" else to_dev(lg)
    dev = {n: bf16_tensor(lay[n]) for n in ("k_cache", "v_cache", "k_src", "v_src", "q_src")}
    dev["out"] = torch.zeros(w.B, w.L, w.Hq, w.D, dtype=torch.bfloat16, device="cuda")
    E.step(p, st, logits, to_dev(st_h["cand_pos"]), to_dev(st_h["cand_count"]), [dev])
    status, word = E.read_device_error(st.dev_err)
    assert status == 0, f"device error word {word:#x}"
    g = {f: getattr(st, f).cpu().numpy() for f in st.FIELDS}
    kc, vc, out = bf16_bits(dev["k_cache"]), bf16_bits(dev["v_cache"]), bf16_bits(dev["out"])
    rng = np.random.default_rng(seed)
    flags = []
    for b in range(w.B):
        x = O.widen(lg[b], w.logits_dtype)
        cnt = int(st_h["cand_count"][b])
        o = O.step(logits=x, cand_pos=st_h["cand_pos"][b], cand_count=cnt, tokens=st_h["tokens"][b],
                   mask=st_h["mask"][b], ring=st_h["ring"][b], ring_head=int(st_h["ring_head"][b]),
                   ring_count=int(st_h["ring_count"][b]), n_dec=w.n_dec, tau=w.tau)
        conf_sorted = sorted(o["log_conf"][:cnt], reverse=True)
        gpu_dec = [int(x) for x in g["dec_pos"][b] if x >= 0]
        if cnt > w.n_dec and conf_sorted[w.n_dec - 1] - conf_sorted[w.n_dec] <= 1e-5:
            # commit near-tie: the device ranks fp32 confidences, the oracle fp64. The device's
            # choice must be n_dec candidates from the top of the ranking (each within 1e-5 of
            # the n_dec-th confidence or above it); the oracle then adopts that choice and
            # everything that follows from it is checked as usual.
            band = conf_sorted[w.n_dec - 1] - 1e-5
            allowed = {int(st_h["cand_pos"][b][i]) for i in range(cnt) if o["log_conf"][i] >= band}
            assert len(gpu_dec) == w.n_dec and set(gpu_dec) <= allowed, (b, gpu_dec, sorted(allowed))
            rows = [i for i in range(cnt) if int(st_h["cand_pos"][b][i]) in gpu_dec]
            o = O.step(logits=x, cand_pos=st_h["cand_pos"][b], cand_count=cnt, tokens=st_h["tokens"][b],
                       mask=st_h["mask"][b], ring=st_h["ring"][b], ring_head=int(st_h["ring_head"][b]),
                       ring_count=int(st_h["ring_count"][b]), n_dec=w.n_dec, tau=w.tau, decoded_rows=rows)
            print(f"b={b}: commit near-tie exemption, device chose {gpu_dec}")
        assert gpu_dec == o["dec_pos"], (b, gpu_dec, o["dec_pos"])
        np.testing.assert_array_equal(g["tokens"][b], o["tokens"])
        np.testing.assert_array_equal(g["mask"][b], o["mask"])
        assert int(g["ring_head"][b]) == o["ring_head"] and int(g["ring_count"][b]) == o["ring_count"]
        np.testing.assert_array_equal(g["ring"][b], o["ring"])
        assert abs(float(g["E"][b]) - o["E"]) <= 1e-3, (g["E"][b], o["E"])
        exempt = abs(o["E"] - w.tau) <= 1e-4
        if exempt:
            print(f"b={b}: flag exemption, E_oracle={o['E']}")
        else:
            assert bool(g["flag"][b]) == o["flag"]
        full = bool(g["flag"][b])
        idx = O.recompute_set(o["mask"], O.history_last(o["ring"], o["ring_head"], o["ring_count"]), full)
        if not exempt:
            np.testing.assert_array_equal(idx, o["idx"])
        R = int(g["R"][b])
        assert R == len(idx)
        np.testing.assert_array_equal(g["idx"][b, :R], idx)
        flags.append(full)
        # caches: recompute rows refreshed from the fresh rows, all others untouched
        want_k = lay["k_cache"][b].copy()
        want_v = lay["v_cache"][b].copy()
        want_k[idx] = lay["k_src"][b][idx]
        want_v[idx] = lay["v_src"][b][idx]
        np.testing.assert_array_equal(kc[b], want_k)
        np.testing.assert_array_equal(vc[b], want_v)
        # attention of the recompute rows (a seeded sample of them on the large cases)
        rows = np.arange(R) if (sample_rows is None or R <= sample_rows) else np.sort(
            rng.choice(R, size=sample_rows, replace=False))
        ref = O.attention(O.widen(lay["q_src"][b][idx[rows]], "bf16"), O.widen(want_k, "bf16"),
                          O.widen(want_v, "bf16"), 1.0 / math.sqrt(w.D))
        ok, msg = attention_close(O.widen(out[b][rows], "bf16"), ref)
        assert ok, f"b={b}: {msg}"
    return flags


@pytest.mark.parametrize("cfg,sample", [(1, None), (2, None), (3, 48)])
def test_workload_step(E, cfg, sample):
    w = W.workload(cfg)
    flags = run_and_check(E, w, W.snapshot_state(w), W.step_logits(w), W.layer_tensors(w, 0), sample_rows=sample)
    if cfg in (1, 2):
        assert flags == [False]  # these seeds commit a low-entropy token: a partial step


def test_long_context_step(E):
    w = W.workload(5)
    run_and_check(E, w, W.snapshot_state(w), W.step_logits(w), W.layer_tensors(w, 0), sample_rows=32)


@pytest.mark.parametrize("cfg,scale", [(2, {}), (3, dict(B=2, L=512, prompt=256, gen=256, V=32000, seed=23))])
def test_always_full_step(E, cfg, scale):
    # tau < 0: every entropy (0 for an empty decode set) exceeds it, so every step is full and,
    # with no scope, ec_step runs the attention on the two-tile dense kernel (MHA and GQA)
    w = W.workload(cfg).scaled(tau=-1.0, **scale)
    flags = run_and_check(E, w, W.snapshot_state(w), W.step_logits(w), W.layer_tensors(w, 0), sample_rows=64)
    assert all(flags)


def test_mixed_flags_in_one_batch(E):
    # Dream-7B-shaped heads, four sequences: even ones commit a near-certain token (partial
    # step), odd ones a near-uniform one (full step).
    w = W.workload(3).scaled(B=4, L=512, prompt=256, gen=256, V=32000, seed=17)
    st_h = W.snapshot_state(w)
    rng = np.random.default_rng(17)
    lg = np.empty((w.B, w.C_max, w.V), np.float32)
    for b in range(w.B):
        if b % 2 == 0:
            lg[b] = rng.standard_normal((w.C_max, w.V))
            # peaks 8 .. 15.75 over the noise: the best rows have entropy ~0.1 (far below tau) and
            # confidences ~1e-2 apart, well clear of the 1e-5 commit near-tie exemption
            lg[b, np.arange(w.C_max), rng.integers(0, w.V, w.C_max)] += 8.0 + 0.25 * np.arange(w.C_max)
        else:
            lg[b] = rng.standard_normal((w.C_max, w.V)) * 0.5
    flags = run_and_check(E, w, st_h, W.to_bf16_bits(lg), W.layer_tensors(w, 0), sample_rows=64)
    assert flags == [False, True, False, True]


def test_mixed_flags_at_full_dream_shape(E):
    # The Dream-7B GQA workload at its own shape (B 8, 28 q / 4 kv heads x 128, L 2048,
    # V 152064 bf16) with per-sequence skip flags: even sequences get a confident candidate
    # (N(0, 1) noise plus a peak, a partial step), odd ones keep the Zipf-ranked logits of
    # the workload (every row has entropy > 3.5: a full step).
    w = W.workload(3)
    st_h = W.snapshot_state(w)
    lg = W.step_logits(w)
    rng = np.random.default_rng(31)
    for b in range(0, w.B, 2):
        x = rng.standard_normal((w.C_max, w.V), dtype=np.float32)
        x[np.arange(w.C_max), rng.integers(0, w.V, w.C_max)] += (8.0 + 0.25 * np.arange(w.C_max)).astype(np.float32)
        lg[b] = W.to_bf16_bits(x)
    flags = run_and_check(E, w, st_h, lg, W.layer_tensors(w, 0), sample_rows=32)
    assert flags == [False, True] * (w.B // 2)


def test_partial_step_with_short_history_and_ragged_candidates(E):
    # history count below k, fewer candidates than C_max, L not a multiple of 128
    w = W.workload(2).scaled(L=1000, prompt=936, gen=64, seed=23)
    st_h = W.snapshot_state(w)
    st_h["cand_count"][0] = 20
    lg = W.step_logits(w)
    flags = run_and_check(E, w, st_h, lg, W.layer_tensors(w, 0))
    assert int(st_h["ring_count"][0]) < w.k
    assert len(flags) == 1


def test_large_vocabulary_step_with_short_candidate_lists(E):
    # Dream-7B-shaped batch (78 MB of logits: the decode stage streams through persistent
    # CTAs) where sequences list fewer candidates than C_max, one none at all: the skipped
    # rows must be left out of the decode, the commit and the gate.
    w = W.workload(3)
    st_h = W.snapshot_state(w)
    st_h["cand_count"][:] = np.array([32, 5, 0, 17, 32, 1, 31, 32], dtype=st_h["cand_count"].dtype)
    run_and_check(E, w, st_h, W.step_logits(w), W.layer_tensors(w, 0), sample_rows=32)
