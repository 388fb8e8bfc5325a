"""The hand-worked step of tests/golden/worked_step.txt: the float64 oracle (CPU) and the
C-ABI library (GPU) against closed-form expected values that neither of them produced.

The fixture's derivations follow "EntropyCache: Decoded Token Entropy Guided KV Caching for
Diffusion Language Models" ([zh] §2.2 / §2.3, [pt] §1 / §2 of the gist.science summaries).
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

import oracle as O

FIXTURE = os.path.join(os.path.dirname(__file__), "golden", "worked_step.txt")
TAUS = (1.1, 1.0)


def _value(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"ln": math.log, "e": math.e}))  # noqa: S307


def _items(text: str):
    out = []
    for tok in text.split():
        parts = [_value(x) for x in tok.split(",")]
        out.append(parts if len(parts) > 1 else parts[0])
    return np.array(out, dtype=np.float64)


def load() -> dict:
    """{section: {name: float64 array}} of the fixture."""
    sec, cur = {}, None
    with open(FIXTURE) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = sec.setdefault(line.strip("[]"), {})
                continue
            name, _, rhs = line.partition("=")
            cur[name.strip()] = _items(rhs)
    return sec


def inputs(fx: dict) -> dict:
    i = fx["inputs"]
    n = lambda key: int(i[key][0])  # noqa: E731
    L, V, C = n("L"), n("V"), n("cand_count")
    return {
        "L": L, "V": V, "D": n("D"), "n_dec": n("n_dec"), "k": n("k"), "scale": float(i["scale"][0]),
        "tokens": i["tokens"].astype(np.int64), "mask": i["mask"].astype(np.uint8),
        "cand_pos": i["cand_pos"].astype(np.int64), "cand_count": C,
        "ring": i["ring"].astype(np.int64), "ring_head": n("ring_head"), "ring_count": n("ring_count"),
        "logits": np.stack([i[f"logits.{r}"] for r in range(C)]),
        **{name: i[name][:, None, :] for name in ("k_cache", "v_cache", "k_src", "v_src", "q_src")},
    }


def test_fixture_is_self_consistent():
    # the printed probabilities behind the logits sum to one row by row, and the worked
    # entropies equal -sum p ln p of those probabilities (a check on the derivation itself)
    fx = load()
    x = inputs(fx)
    for r, row in enumerate(x["logits"]):
        w = np.exp(row)
        p = w / w.sum()
        assert math.isclose(-(p * np.log(p)).sum(), fx["decode"]["entropy"][r], rel_tol=1e-14)


def test_oracle_reproduces_the_worked_step():
    fx = load()
    x = inputs(fx)
    d = fx["decode"]
    for tau in TAUS:
        want = fx[f"expected tau={tau}"]
        lay = {n: x[n] for n in ("k_cache", "v_cache", "k_src", "v_src", "q_src")}
        o = O.step(logits=x["logits"], cand_pos=x["cand_pos"], cand_count=x["cand_count"], tokens=x["tokens"],
                   mask=x["mask"], ring=x["ring"], ring_head=x["ring_head"], ring_count=x["ring_count"],
                   n_dec=x["n_dec"], tau=tau, layers=[lay], scale=x["scale"])
        np.testing.assert_array_equal(o["ids"], d["ids"])
        np.testing.assert_allclose(o["entropy"], d["entropy"], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(o["log_conf"], d["log_conf"], rtol=1e-13, atol=1e-15)
        assert o["dec_pos"] == d["dec_pos"].astype(int).tolist()
        assert math.isclose(o["E"], float(d["E"][0]), rel_tol=1e-13)
        np.testing.assert_array_equal(o["tokens"], d["tokens"])
        np.testing.assert_array_equal(o["mask"], d["mask"])
        np.testing.assert_array_equal(o["ring"], d["ring"])
        assert (o["ring_head"], o["ring_count"]) == (int(d["ring_head"][0]), int(d["ring_count"][0]))
        assert o["flag"] == bool(want["flag"][0])
        np.testing.assert_array_equal(o["idx"], want["idx"])
        out = o["layers"][0]
        np.testing.assert_array_equal(out["k_cache"][:, 0], want["k_cache"])
        np.testing.assert_array_equal(out["v_cache"][:, 0], want["v_cache"])
        np.testing.assert_allclose(out["out"][:, 0], want["out"], rtol=1e-13)


# ---- the C-ABI library on the GPU ---------------------------------------------------------
# The 2-wide head is embedded in a 64-wide one (the library's smallest head size) with zero
# padding, which leaves every score and the first two output columns unchanged. Logits are
# fp32: ln of a small integer rounds to fp32 within 3e-8, so the decode results may move by
# 1e-5 at most; keys, values and queries are small integers, exact in bf16.
GPU_D = 64
DEC_TOL = 1e-5


def _pad(a: np.ndarray) -> np.ndarray:
    out = np.zeros(a.shape[:-1] + (GPU_D,), np.float32)
    out[..., : a.shape[-1]] = a
    return out


@pytest.mark.gpu
def test_library_reproduces_the_worked_step():
    import torch

    from tests._helpers import attention_close

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import entropy_gated_kv_gb300 as E

    fx = load()
    x = inputs(fx)
    d = fx["decode"]
    L, V, C = x["L"], x["V"], x["cand_count"]
    dev = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a)).to("cuda", dt)  # noqa: E731

    # (a) alone
    ids, ent, conf = (t.cpu().numpy() for t in E.entropy_decode(dev(x["logits"], torch.float32)))
    np.testing.assert_array_equal(ids, d["ids"])
    np.testing.assert_allclose(ent, d["entropy"], rtol=0, atol=DEC_TOL)
    np.testing.assert_allclose(conf, d["log_conf"], rtol=0, atol=DEC_TOL)

    # the whole step, at both thresholds
    for tau in TAUS:
        want = fx[f"expected tau={tau}"]
        p = E.Params(B=1, L=L, Hq=1, Hkv=1, D=GPU_D, V=V, C_max=C, k=x["k"], n_dec=x["n_dec"], tau=tau,
                     logits_dtype="f32")
        st = E.DecodeState.from_arrays(p, tokens=x["tokens"][None], mask=x["mask"][None], ring=x["ring"][None],
                                       ring_head=[x["ring_head"]], ring_count=[x["ring_count"]])
        lay = {n: dev(_pad(x[n])[None], torch.bfloat16) for n in ("k_cache", "v_cache", "k_src", "v_src", "q_src")}
        lay["out"] = torch.zeros(1, L, 1, GPU_D, dtype=torch.bfloat16, device="cuda")
        E.step(p, st, dev(x["logits"][None], torch.float32), dev(x["cand_pos"][None], torch.int32),
               dev([C], torch.int32), [lay], scale=x["scale"])
        status, word = E.read_device_error(st.dev_err)
        assert status == 0, f"device error word {word:#x}"
        g = {f: getattr(st, f).cpu().numpy()[0] for f in st.FIELDS if f != "dev_err"}
        np.testing.assert_array_equal(g["dec_pos"], d["dec_pos"])
        assert abs(float(g["E"]) - float(d["E"][0])) <= DEC_TOL
        np.testing.assert_array_equal(g["tokens"], d["tokens"])
        np.testing.assert_array_equal(g["mask"], d["mask"])
        np.testing.assert_array_equal(g["ring"], d["ring"])
        assert (int(g["ring_head"]), int(g["ring_count"])) == (int(d["ring_head"][0]), int(d["ring_count"][0]))
        assert int(g["flag"]) == int(want["flag"][0])
        R = int(g["R"])
        assert R == len(want["idx"])
        np.testing.assert_array_equal(g["idx"][:R], want["idx"])
        kc = lay["k_cache"].float().cpu().numpy()[0, :, 0]
        vc = lay["v_cache"].float().cpu().numpy()[0, :, 0]
        np.testing.assert_array_equal(kc, _pad(want["k_cache"]))
        np.testing.assert_array_equal(vc, _pad(want["v_cache"]))
        out = lay["out"].float().cpu().numpy()[0, :R, :, :].astype(np.float64)
        ok, msg = attention_close(out, _pad(want["out"])[:, None, :].astype(np.float64))
        assert ok, f"tau={tau}: {msg}"
