"""The bench's JSON line, built from a synthetic measurement on the CPU: every key of the
contract is present, and the derived numbers (whole-job steps/s, per-step time, the roofline's
achieved rate and fraction, the launch count) follow from the inputs by the stated formulas."""
import argparse
import json

import pytest

import bench


def _args(**kw):
    a = dict(steps=1000, warmup=5, workload=bench.WORKLOAD, tau=None, no_cpu_baseline=True, cpu_seconds=1.0)
    a.update(kw)
    return argparse.Namespace(**a)


def _res(ms=25.0, attn_us=9.0, ent_us=6.0):
    return {
        "ms": ms,
        "kernels": {"R": 95, "entropy_decode_us": ent_us, "partial_attention_us": attn_us, "kv_scatter_us": 2.0,
                    "read_floor_us": 2.7},
        "flag": False,
        "R": 95,
        "copy_mb": 58.0,
        "ncopy": 17,
        "touched_mb": 25.0,
        "e2e": {"value": 5000.0, "unit": "steps/s", "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 2},
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []},
    }


def _line(capsys, args, res, world=1):
    bench.emit_ours(args, res, 0, world)
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1, out  # exactly one JSON line
    return json.loads(out[0])


def test_every_contract_key_and_derived_value(capsys):
    line = _line(capsys, _args(), _res())
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["metric"] == bench.METRIC
    assert line["value"] == pytest.approx(1000 / 0.025)  # whole-job steps per second
    assert line["ms_per_step"] == pytest.approx(0.025)
    assert (line["unit"], line["n_gpus"], line["steps"], line["warmup"]) == ("steps/s", 1, 1000, 5)
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["data"] == "synthetic" and "workload" in line["config"]
    assert line["gpu_launches"] == 4 * 1000  # the step's four kernels per timed step
    assert line["e2e"]["value"] == 5000.0 and line["clocks"]["sm_mhz"] == 2070.0


def test_roofline_is_the_slowest_stage_against_its_bound(capsys):
    line = _line(capsys, _args(), _res(attn_us=9.0, ent_us=6.0))
    roof = line["roofline"]
    assert roof["kernel"] == "partial_attention"  # the larger per-step time
    assert roof["bound"] == "hbm"  # 87 flops per byte at R = 95, below the ridge
    alg = bench.algorithmic(bench.bench_workload(_args()), 95)
    assert roof["achieved"] == pytest.approx(alg["partial_attention_bytes"] / 9e-6 / 1e9)
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in roof
    # when the decode stage is the slower one it becomes the reported kernel
    line = _line(capsys, _args(), _res(attn_us=5.0, ent_us=6.0))
    assert line["roofline"]["kernel"] == "entropy_decode" and line["roofline"]["unit"] == "GB/s"


def test_whole_job_value_scales_with_ranks(capsys):
    line = _line(capsys, _args(), _res(), world=2)
    assert line["n_gpus"] == 2
    assert line["value"] == pytest.approx(2 * 1000 / 0.025)  # every rank's steps over the slowest rank's time


def test_flat_state_layout():
    # the e2e loop restores the decode state with one copy and reads E, flag and R back as one
    # slice: every field must be a view of the flat buffer, naturally aligned, the mask 16-byte
    # aligned (the library reads it with 16-byte loads), and E, flag, R adjacent in that order
    import numpy as np
    import torch

    import entropy_gated_kv_gb300 as E

    p = E.Params(B=3, L=40, Hq=1, Hkv=1, D=64, V=100, C_max=4, k=5, n_dec=2)
    tokens = np.arange(120).reshape(3, 40)
    st, flat, (r0, r1) = bench.flat_state(E, p, "cpu", tokens=tokens, mask=np.ones((3, 40)))
    base = flat.data_ptr()
    for f in E.DecodeState.FIELDS:
        t = getattr(st, f)
        off = t.data_ptr() - base
        assert 0 <= off and off + t.numel() * t.element_size() <= flat.numel(), f
        assert off % (16 if f == "mask" else t.element_size()) == 0, f
    assert st.flag.dtype == torch.uint8 and tuple(st.flag.shape) == (3,)
    assert st.E.data_ptr() - base == r0 and st.R.data_ptr() - base + 3 * 4 == r1
    np.testing.assert_array_equal(st.tokens.numpy(), tokens)
    st.E.fill_(0.5)
    st.flag.fill_(1)
    st.R.fill_(7)
    blob = flat[r0:r1].clone()
    assert blob[:12].view(torch.float32).tolist() == [0.5] * 3
    assert blob[12:15].tolist() == [1, 1, 1]
    assert blob[-12:].view(torch.int32).tolist() == [7] * 3


def test_reference_arm_line():
    # the oracle arm runs on the host cores: one JSON line with the same metric, unit and
    # direction as ours, marked impl = reference, its e2e equal to its own value with no copies
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "steps/s" and d["higher_is_better"] is True and d["warmup"] >= 3
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]


def test_config_entry_against_its_binding_roofline():
    # A `configs` entry from a synthetic measurement: the decode against HBM, the attention
    # against the roofline its arithmetic intensity selects (tensor above the ridge, else HBM).
    import workloads as W

    pk = bench.peaks()
    kern = {"entropy_decode_us": 8.0, "partial_attention_us": 20.0, "kv_scatter_us": 3.0, "read_floor_us": 4.0}
    w = W.workload(2)
    e = bench.summarise_config(w, 20000.0, 1, 1024, kern, 50e6, "host")  # a full step, R = L
    alg = bench.algorithmic(w, 1024)
    assert e["us_per_step"] == pytest.approx(50.0)
    assert e["entropy_decode"]["of_read_floor"] == pytest.approx(0.5)  # the floor's time over the decode's
    assert e["entropy_decode"]["GB/s"] == pytest.approx(alg["entropy_decode_bytes"] / 8e-6 / 1e9)
    att = e["partial_attention"]
    assert att["bound"] == "tensor"  # 512 flops per byte
    assert att["TFLOP/s"] == pytest.approx(alg["partial_attention_flops"] / 20e-6 / 1e12)
    assert att["frac_bound"] == pytest.approx(att["TFLOP/s"] / pk["bf16_tflops"])
    e = bench.summarise_config(w, 40000.0, 0, 95, kern, 50e6, "host")  # partial: 87 flops per byte
    assert e["partial_attention"]["bound"] == "hbm"
    assert e["partial_attention"]["frac_bound"] == pytest.approx(e["partial_attention"]["frac_hbm"])


@pytest.mark.parametrize("n,rate", [(40, 0.0), (40, 0.1), (40, 0.25), (40, 0.5), (40, 1.0), (7, 0.3), (1, 1.0)])
def test_full_step_pattern(n, rate):
    """The flag-rate runs of the layer forward: round(rate * n) full steps, spread so that every
    window of n / m consecutive steps holds one of them."""
    p = bench.full_step_pattern(n, rate)
    m = round(rate * n)
    assert len(p) == n and sum(p) == m
    if 0 < m < n:
        where = [i for i, f in enumerate(p) if f]
        gaps = {b - a for a, b in zip(where, where[1:])}
        assert max(gaps) - min(gaps) <= 1
