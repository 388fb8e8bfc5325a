"""GPU parity of the decoding schedules the entropy gate carries over to (pt summary §5
"Generalidade": sliding-window or block decoding; zh summary §5: a sub-block recompute
signal in block diffusion), run as device-resident decoding loops: every step builds its
candidates on the device (ec_candidates) from the mask the previous step left, then runs
ec_step. The float64 oracle follows the same trajectory and checks, at every step and for
every sequence, the candidates, the committed position and token, the mask, the history, E
(1e-3), the flag, the recompute set and the refreshed caches bit for bit, and the attention
of every recompute row within the bf16 tolerance.

Shapes: B 2, 8 x 64 MHA, L 512 (prompt 384 + generation 128), k 16, V 32000 bf16 logits,
one token per step, about 10% high-entropy steps (the "schedule" logits recipe).
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import attention_close, bf16_bits, bf16_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import entropy_gated_kv_gb300 as E

    E.lib()
    return E


def test_candidates_match_oracle(E):
    import torch

    rng = np.random.default_rng(61)
    for L, C_max in ((300, 32), (4096, 32), (77, 8), (2000, 1024)):
        p = E.Params(B=5, L=L, Hq=8, Hkv=8, D=64, V=100, C_max=C_max, k=4)
        mask = (rng.random((5, L)) < rng.random((5, 1))).astype(np.uint8)
        mask[3] = 0  # nothing masked
        st = E.DecodeState.from_arrays(p, mask=mask)
        for mode, fn in (("block", O.block_candidates), ("sliding", O.sliding_window_candidates)):
            for _ in range(6):
                start = int(rng.integers(0, L))
                width = int(rng.integers(1, C_max + 1))
                cp, cc = E.candidates(p, st, mode, start, width)
                torch.cuda.synchronize()
                cp, cc = cp.cpu().numpy(), cc.cpu().numpy()
                for b in range(5):
                    want = fn(mask[b], start, width)
                    assert cc[b] == len(want), (mode, L, b, start, width)
                    assert cp[b, : len(want)].tolist() == want
                    assert (cp[b, len(want):] == -1).all()


def _schedule_workload():
    return W.workload(4).scaled(B=2, L=512, prompt=384, gen=128, block=32, Hq=8, Hkv=8, D=64, V=32000, k=16,
                                logits_kind="schedule", n_layers=1, steps=128, seed=62)


def _run_schedule(E, mode: str, width: int):
    """mode 'sliding': windows of `width` positions opening at the first masked one;
    mode 'block': blocks of `width` positions decoded one after the other, each block the
    gate's scope."""
    import torch

    w = _schedule_workload().scaled(block=width)
    st_h = W.snapshot_state(w)  # the prompt decoded, the generation masked, an empty history
    lay = W.layer_tensors(w, 0)
    dev = {n: bf16_tensor(lay[n]) for n in ("k_cache", "v_cache", "k_src", "v_src", "q_src")}
    dev["out"] = torch.zeros(w.B, w.L, w.Hq, w.D, dtype=torch.bfloat16, device="cuda")
    base = E.Params(B=w.B, L=w.L, Hq=w.Hq, Hkv=w.Hkv, D=w.D, V=w.V, C_max=width, k=w.k, n_dec=1, tau=w.tau,
                    logits_dtype="bf16")
    st = E.DecodeState.from_arrays(base, tokens=st_h["tokens"], mask=st_h["mask"], ring=st_h["ring"],
                                   ring_head=st_h["ring_head"], ring_count=st_h["ring_count"])
    ws = E.workspace(E.step_workspace_size(base))
    cache = {n: lay[n].copy() for n in lay}
    tokens = st_h["tokens"].astype(np.int64)
    mask = st_h["mask"].copy()
    ring = st_h["ring"].astype(np.int64)
    head = st_h["ring_head"].astype(np.int64)
    count = st_h["ring_count"].astype(np.int64)
    n_full = 0
    n_exempt = [0]
    for t in range(w.steps):
        if mode == "block":
            lo = w.prompt + (t // width) * width
            scope = (lo, lo + width)
            p = E.Params(**{**base.__dict__, "scope_lo": lo, "scope_hi": lo + width})
            cp, cc = E.candidates(p, st, "block", lo, width)
        else:
            scope = None
            p = base
            cp, cc = E.candidates(p, st, "sliding", w.prompt, width)
        lg = W.step_logits(w.scaled(block=width), t)  # [B, width, V] bf16 bits
        E.step(p, st, bf16_tensor(lg), cp, cc, [dev], ws=ws)
        status, word = E.read_device_error(st.dev_err)
        assert status == 0, f"step {t}: device error word {word:#x}"
        g = {f: getattr(st, f).cpu().numpy() for f in ("dec_pos", "E", "flag", "R", "idx", "tokens", "mask", "ring",
                                                          "ring_head", "ring_count")}
        cpos, ccnt = cp.cpu().numpy(), cc.cpu().numpy()
        out = bf16_bits(dev["out"])
        for b in range(w.B):
            fn = O.block_candidates if mode == "block" else O.sliding_window_candidates
            cand = fn(mask[b], scope[0] if mode == "block" else w.prompt, width)
            assert ccnt[b] == len(cand) and cpos[b, : len(cand)].tolist() == cand, (t, b)
            args = dict(logits=O.widen(lg[b], "bf16"), cand_pos=np.array(cand + [-1] * (width - len(cand))),
                        cand_count=len(cand), tokens=tokens[b], mask=mask[b], ring=ring[b], ring_head=int(head[b]),
                        ring_count=int(count[b]), n_dec=1, tau=w.tau, scope=scope,
                        layers=[{n: O.widen(cache[n][b], "bf16") for n in ("k_cache", "v_cache", "k_src", "v_src",
                                                                           "q_src")}])
            o = O.step(**args)
            gpu_dec = [int(x) for x in g["dec_pos"][b] if x >= 0]
            conf = sorted(o["log_conf"][: len(cand)], reverse=True)
            if len(cand) > 1 and conf[0] - conf[1] <= 1e-5:  # commit near-tie: adopt the device's choice
                n_exempt[0] += 1
                allowed = [cand[i] for i in range(len(cand)) if o["log_conf"][i] >= conf[0] - 1e-5]
                assert len(gpu_dec) == 1 and gpu_dec[0] in allowed, (t, b, gpu_dec, allowed)
                o = O.step(**args, decoded_rows=[cand.index(gpu_dec[0])])
            assert gpu_dec == o["dec_pos"], (t, b)
            assert abs(float(g["E"][b]) - o["E"]) <= 1e-3, (t, b)
            assert abs(o["E"] - w.tau) > 1e-4  # the recipe keeps the gate clear of the margin
            assert bool(g["flag"][b]) == o["flag"], (t, b)
            n_full += int(o["flag"])
            R = int(g["R"][b])
            assert R == o["R"], (t, b)
            np.testing.assert_array_equal(g["idx"][b, :R], o["idx"])
            np.testing.assert_array_equal(g["tokens"][b], o["tokens"])
            np.testing.assert_array_equal(g["mask"][b], o["mask"])
            np.testing.assert_array_equal(g["ring"][b], o["ring"])
            tokens[b], mask[b], ring[b] = o["tokens"], o["mask"], o["ring"]
            head[b], count[b] = o["ring_head"], o["ring_count"]
            for n, src in (("k_cache", "k_src"), ("v_cache", "v_src")):
                cache[n][b][o["idx"]] = cache[src][b][o["idx"]]
            ok, msg = attention_close(O.widen(out[b, :R], "bf16"), o["layers"][0]["out"])
            assert ok, f"step {t} b {b}: {msg}"
    np.testing.assert_array_equal(bf16_bits(dev["k_cache"]), cache["k_cache"])
    np.testing.assert_array_equal(bf16_bits(dev["v_cache"]), cache["v_cache"])
    assert not mask[:, w.prompt:].any()  # one position per step: the generation is decoded
    assert n_exempt[0] == 0  # the recipe keeps the commit clear of near-ties
    return n_full


def test_sliding_window_decoding_trace(E):
    n_full = _run_schedule(E, "sliding", 16)
    assert 0 < n_full < 2 * 128 // 3  # the high-entropy steps (about 10%, step 0 included)


def test_block_scoped_decoding_trace(E):
    # block diffusion: four blocks of 32, each the gate's scope; attention is block-causal
    n_full = _run_schedule(E, "block", 32)
    assert 0 < n_full < 2 * 128 // 3
