#!/usr/bin/env python3
"""EntropyCache denoising-step benchmark on GB300.

Workload: the LLaDA-8B-shaped layer step (B 1, 32 x 128 MHA, L 1024 = 768 + 256, 32 masked
candidates, k 64, V 126464 bf16 logits ~ N(0, s^2), s ~ U[0.5, 8], tau 1), seeded synthetic
data. One step = ec_step: (a) entropy decode of the 32 candidate rows, (b)+(c) gate,
history and recompute set, K/V refresh of the set and query gather, (d) attention of the set
against the 1024-row cache. With this seed the committed token has entropy 0.74 < tau, so
the step is a partial one with R = 95 recompute rows.

Our arm (default): K steps replayed from CUDA graphs of up to 500 steps. Every step owns a
fresh copy of the decode state (restored inside the graph, counted in the time), and steps
rotate over enough copies of the per-step inputs that the bytes they touch in one rotation
(logits and K/V cache, at least 400 MB) cannot stay in the 129 MB L2. Per-kernel times for the
roofline come from CUDA-event timing of each kernel's own entry point, each rotating over
400 MB of its own inputs. The e2e figure runs ec_step from pinned host buffers with the
host<->device copies inside the timed region.

Reference arm (--impl reference): the float64 CPU oracle of the same step, timed on the host
cores: every one of its K steps is a whole oracle step (all candidate rows, every recompute row
over all heads), unless K whole steps would not fit in a few minutes.

Multi-GPU: the step does not shard across GPUs (one sequence batch per step); N > 1 runs N
independent replicas, one per rank, with no collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "EntropyCache steps/s at LLaDA-8B layer shape; % of HBM / tensor-core roofline"
WORKLOAD = 2
ROTATION_BYTES = 400 << 20  # bytes touched per rotation of the timed inputs (L2 is 129 MB)
CHUNK = 500
STEADY_CHUNK = 500
STEADY_REPEATS = 5


# ---- multi-rank helpers (replicas: one independent step loop per rank, no data exchange) ----


def init_ranks(world: int, backend: str | None = None) -> None:
    """One process group for the timing barrier and reduction: NCCL when each rank has a GPU,
    gloo otherwise, or the given backend (the CPU tests of this logic pass gloo)."""
    if world <= 1:
        return
    import torch
    import torch.distributed as dist

    if backend is not None:
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    else:
        dist.init_process_group("gloo")


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Barrier, then the largest of the ranks' timed-region lengths: the job's time at this N."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    dist.barrier()
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_throughput(world: int, steps: int, ms: float) -> float:
    """Whole-job steps/s: each of the `world` ranks ran `steps` steps of its own replica in at
    most `ms` milliseconds."""
    return world * steps / (ms / 1e3)


def kernel_source_hash(name: str) -> str:
    """Hash of a kernel's source file (ncu counters are only valid for the source they came from)."""
    import hashlib

    path = os.path.join(ROOT, "entropy_gated_kv_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel: str, source: str) -> float | None:
    """DRAM bytes per launch from profiles/traffic.json, if captured on the current source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)[kernel]
        return float(d["dram_bytes_per_launch"]) if d["source_sha"] == kernel_source_hash(source) else None
    except Exception:
        return None


def run_profile(steps: int, workload: int = WORKLOAD, tau: float | None = None) -> None:
    """A few eager steps of the workload (no graphs, no timing), then as many calls of the
    standalone decode entry on the step's logits and of the output projection fused with the
    decode (on a full step, of the dense attention first): a short program for ncu."""
    import torch

    import entropy_gated_kv_gb300 as E
    from entropy_gated_kv_gb300 import build as B

    B.build()
    w = W.workload(workload)
    p = E.Params(B=w.B, L=w.L, Hq=w.Hq, Hkv=w.Hkv, D=w.D, V=w.V, C_max=w.C_max, k=w.k, n_dec=w.n_dec,
                 tau=w.tau if tau is None else tau, logits_dtype=w.logits_dtype)
    st_h = W.snapshot_state(w)
    lay = W.layer_tensors(w, 0)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    layer = {n: bf(lay[n]) for n in ("k_cache", "v_cache", "k_src", "v_src", "q_src")}
    layer["out"] = torch.zeros(w.B, w.L, w.Hq, w.D, dtype=torch.bfloat16, device="cuda")
    lg_h = W.step_logits(w)
    logits = bf(lg_h) if w.logits_dtype == "bf16" else torch.from_numpy(np.ascontiguousarray(lg_h)).cuda()
    cp = torch.from_numpy(st_h["cand_pos"]).cuda()
    cc = torch.from_numpy(st_h["cand_count"]).cuda()
    ws = E.workspace(E.step_workspace_size(p))
    for _ in range(steps):
        st = E.DecodeState.from_arrays(p, tokens=st_h["tokens"], mask=st_h["mask"], ring=st_h["ring"],
                                       ring_head=st_h["ring_head"], ring_count=st_h["ring_count"])
        E.step(p, st, logits, cp, cc, [layer], ws=ws)
    if int(st.flag.max().item()) and w.D == 128:  # a full step: also the dense attention
        for _ in range(steps):
            E.dense_attention(p, layer["q_src"], layer["k_cache"], layer["v_cache"], layer["out"])
    rows = logits.view(-1, w.V)
    ews = E.workspace(E.entropy_decode_workspace_size(rows.shape[0], w.V, rows.dtype))
    for _ in range(steps):
        E.entropy_decode(rows, ws=ews)
    if w.d_model > 0:  # and the output projection fused with the decode, on a random weight
        g = torch.Generator(device="cuda").manual_seed(w.seed)
        hid = torch.randn(rows.shape[0], w.d_model, device="cuda", generator=g).to(torch.bfloat16)
        wt = (torch.randn(w.V, w.d_model, device="cuda", generator=g) / w.d_model ** 0.5).to(torch.bfloat16)
        for _ in range(steps):
            E.lm_head_entropy(hid, wt)
        del hid, wt
    if workload == 2:  # and the partial, then the full, forward of one layer of that shape
        torch.cuda.synchronize()
        dev = torch.device("cuda", torch.cuda.current_device())
        lp, lw, x_src, kc, vc, idx_p, R_p, dff, _ = layer_setup(E, dev)
        lws = E.workspace(E.layer_forward_workspace_size(lp, dff), dev)
        full_idx = torch.arange(w.L, dtype=torch.int32, device=dev).view(1, w.L)
        full_R = torch.tensor([w.L], dtype=torch.int32, device=dev)
        for idx, R in ((idx_p, R_p), (full_idx, full_R)):
            for _ in range(steps):
                E.layer_forward(lp, lw, idx, R, x_src, kc, vc, ws=lws)
    torch.cuda.synchronize()
    status, word = E.read_device_error(st.dev_err)
    print(json.dumps({"profile_steps": steps, "R": int(st.R[0]), "flag": int(st.flag[0]), "status": status}))


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def workload_desc(w) -> str:
    return (f"{w.name}: B{w.B}, {w.Hq}x{w.D} {'MHA' if w.Hq == w.Hkv else 'GQA'}, L={w.L} ({w.prompt}+{w.gen}, "
            f"block {w.block}), {w.C_max} masked candidates, k={w.k}, V={w.V} {w.logits_dtype} logits, "
            f"tau={w.tau}, one attention layer")


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------------------
# our arm


def bench_workload(args):
    """The workload timed: workload 2 by default; --workload / --tau override it."""
    w = W.workload(args.workload)
    if args.tau is not None:
        w = w.scaled(tau=float(args.tau))
    return w


def params_of(E, w):
    return E.Params(B=w.B, L=w.L, Hq=w.Hq, Hkv=w.Hkv, D=w.D, V=w.V, C_max=w.C_max, k=w.k, n_dec=w.n_dec, tau=w.tau,
                    logits_dtype=w.logits_dtype)


def host_inputs(w, dev):
    """The workload's own seeded inputs (the arrays the parity tests check), on the device."""
    import torch

    lg_h = W.step_logits(w)
    lay_h = W.layer_tensors(w, 0)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    base = {n: bf(lay_h[n]) for n in ("k_cache", "v_cache", "k_src", "v_src", "q_src")}
    base["logits"] = bf(lg_h) if w.logits_dtype == "bf16" else torch.from_numpy(lg_h).to(dev)
    return base, lg_h, lay_h


def device_inputs(w, dev, seed, logits=None):
    """Inputs of the workload's shapes and distributions drawn on the device (the step's time
    depends only on shapes and on the gate, which the host-drawn logits and state decide):
    K/V cache and queries ~ N(0, 1), fresh rows = cache + N(0, 0.05^2), all bf16."""
    import torch

    g = torch.Generator(device=dev).manual_seed(int(seed))
    bf = torch.bfloat16
    kv = (w.B, w.L, w.Hkv, w.D)
    d = {}
    for n in ("k", "v"):
        c = torch.randn(kv, generator=g, device=dev)
        d[f"{n}_cache"] = c.to(bf)
        d[f"{n}_src"] = (d[f"{n}_cache"].float() + 0.05 * torch.randn(kv, generator=g, device=dev)).to(bf)
        del c
    d["q_src"] = torch.randn(w.B, w.L, w.Hq, w.D, generator=g, device=dev).to(bf)
    if logits is not None:
        d["logits"] = logits
    return d


def touched_bytes(base) -> int:
    """Bytes a step reads in bulk from one copy of its inputs: the logits and the whole K/V
    cache (the fresh rows and queries of the recompute set are a small part)."""
    return sum(base[n].numel() * base[n].element_size() for n in ("logits", "k_cache", "v_cache") if n in base)


def rotation_copies(base, min_bytes=ROTATION_BYTES, max_copies=64) -> int:
    """Copies of the per-step inputs to rotate over: enough that the bytes the steps touch in
    one rotation (at least min_bytes, about three times the 129 MB L2) cannot stay in L2."""
    return max(1, min(max_copies, -(-min_bytes // touched_bytes(base))))


def make_copies(base, w, dev, min_bytes=None, max_copies=64):
    """Copies of the per-step inputs to rotate over (rotation_copies), so no step finds its
    inputs in L2."""
    import torch

    per = sum(t.numel() * t.element_size() for t in base.values())
    n = rotation_copies(base, min_bytes or ROTATION_BYTES, max_copies)
    copies = []
    for c in range(n):
        d = {k: (t if c == 0 else t.clone()) for k, t in base.items()}
        d["out"] = torch.zeros(w.B, w.L, w.Hq, w.D, dtype=torch.bfloat16, device=dev)
        copies.append(d)
    return copies, per


class StepLoop:
    """K steps of ec_step over rotating input copies, replayed from CUDA graphs of up to CHUNK
    steps. Every step owns a fresh copy of the decode state, restored inside the graph."""

    def __init__(self, E, p, w, copies, st_h, dev, nstate):
        import torch

        self.E, self.p, self.w, self.copies, self.dev = E, p, w, copies, dev
        self.cand_pos = torch.from_numpy(st_h["cand_pos"]).to(dev)
        self.cand_count = torch.from_numpy(st_h["cand_count"]).to(dev)
        self.ws = E.workspace(E.step_workspace_size(p), dev)
        self.pristine = E.DecodeState.from_arrays(p, device=dev, tokens=st_h["tokens"], mask=st_h["mask"],
                                                  ring=st_h["ring"], ring_head=st_h["ring_head"],
                                                  ring_count=st_h["ring_count"])
        self.nstate = nstate
        self.states = {f: getattr(self.pristine, f).unsqueeze(0).repeat(nstate, *([1] * getattr(self.pristine, f).dim()))
                       .contiguous() for f in E.DecodeState.FIELDS}

    def state(self, i):
        s = object.__new__(self.E.DecodeState)
        for f in self.E.DecodeState.FIELDS:
            setattr(s, f, self.states[f][i])
        return s

    def restore(self, n):
        for f in self.E.DecodeState.FIELDS:
            src = getattr(self.pristine, f)
            self.states[f][:n].copy_(src.unsqueeze(0).expand(n, *src.shape))

    def one(self, i, slot):
        c = self.copies[i % len(self.copies)]
        self.E.step(self.p, self.state(slot), c["logits"], self.cand_pos, self.cand_count,
                    [dict(k_cache=c["k_cache"], v_cache=c["v_cache"], k_src=c["k_src"], v_src=c["v_src"],
                          q_src=c["q_src"], out=c["out"])], ws=self.ws)

    def capture(self, n):
        import torch

        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.restore(n)
                for i in range(n):
                    self.one(i, i)
        torch.cuda.current_stream().wait_stream(s)
        return g

    def warm_eager(self, n):
        """n eager steps; returns (flag of sequence max, R summed over the batch)."""
        import torch

        self.restore(self.nstate)
        for i in range(n):
            self.one(i, i % self.nstate)
        torch.cuda.synchronize()
        st0 = self.state(0)
        status, word = self.E.read_device_error(st0.dev_err)
        if status != 0:
            raise RuntimeError(f"device error word {word:#x} during warm-up")
        return int(st0.flag.max().item()), int(st0.R.sum().item()), st0

    def check(self):
        status, word = self.E.read_device_error(self.state(0).dev_err)
        if status != 0:
            raise RuntimeError(f"device error word {word:#x} during the timed steps")


def replay_ms(graphs, dev):
    """CUDA-event time of one pass over `graphs` (each replayed once, in order)."""
    import torch

    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for g in graphs:
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def warm_replay(g, min_ms=100.0):
    """Untimed replays of g for at least min_ms of wall time: clocks and caches settle before
    a timed region, whatever its length."""
    import torch

    t0 = time.perf_counter()
    while (time.perf_counter() - t0) * 1e3 < min_ms:
        g.replay()
        torch.cuda.synchronize()


def run_ours(args, rank: int, world: int) -> dict | None:
    import torch

    import entropy_gated_kv_gb300 as E
    from entropy_gated_kv_gb300 import build as B

    B.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = bench_workload(args)
    p = params_of(E, w)
    K, Wm = args.steps, args.warmup
    st_h = W.snapshot_state(w)
    base, lg_h, lay_h = host_inputs(w, dev)
    ncopy = rotation_copies(base)
    copies = []
    for c in range(ncopy):
        d = {n: t.clone() for n, t in base.items()}
        d["out"] = torch.zeros(w.B, w.L, w.Hq, w.D, dtype=torch.bfloat16, device=dev)
        copies.append(d)
    del base

    G = max(1, min(CHUNK, K))
    loop = StepLoop(E, p, w, copies, st_h, dev, max(G, Wm, STEADY_CHUNK, 1))
    flag, R, st0 = loop.warm_eager(Wm)
    g_main = loop.capture(G)
    rem = K % G
    g_rem = loop.capture(rem) if rem else None
    warm_replay(g_main)  # untimed: the timed region starts on a settled GPU

    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t0.record()
        for _ in range(K // G):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        t1.record()
        torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    loop.check()

    copy_mb = sum(t.numel() * t.element_size() for t in copies[0].values()) / 1e6
    res = {"ms": ms, "flag": flag, "R": R, "clocks": clk.summary(), "copy_mb": copy_mb, "ncopy": ncopy,
           "touched_mb": touched_bytes(copies[0]) / 1e6}
    # steady-state rate: the median over repeats of 4 x STEADY_CHUNK graph-replayed steps
    g_st = loop.capture(STEADY_CHUNK)
    warm_replay(g_st, 50.0)
    reps = [4 * STEADY_CHUNK / (replay_ms([g_st] * 4, dev) / 1e3) for _ in range(STEADY_REPEATS)]
    loop.check()
    res["steady"] = {"steps_per_s": statistics.median(reps), "repeats": STEADY_REPEATS,
                     "steps_each": 4 * STEADY_CHUNK, "spread": [min(reps), max(reps)]}
    del g_main, g_rem, g_st
    if rank == 0:
        res["kernels"] = time_kernels(E, p, w, copies, st0, dev, min(K, 2000) if K >= 200 else 2000)
        per_step = sum(lay_h[n].nbytes for n in ("k_src", "v_src", "q_src")) + lg_h.nbytes
        n_e2e = max(10, min(K, 2000, int(20e9 // per_step)))  # at most ~20 GB of host->device traffic
        res["e2e"] = run_e2e(E, p, w, lay_h, lg_h, st_h, dev, n_e2e)
        del copies, loop
        torch.cuda.empty_cache()
        if not args.no_configs:
            res["configs"] = run_configs(E, dev, args)
    return res


def config_entry(E, w, dev, n_steps, inputs: str, seed: int) -> dict:
    """steps/s and per-kernel times of one workload's single step (see run_configs)."""
    import torch

    p = params_of(E, w)
    st_h = W.snapshot_state(w)
    if inputs == "host":
        base, _, _ = host_inputs(w, dev)
    else:
        lg_h = W.step_logits(w)
        lg = (torch.from_numpy(lg_h.view(np.int16)).to(dev).view(torch.bfloat16) if w.logits_dtype == "bf16"
              else torch.from_numpy(lg_h).to(dev))
        base = device_inputs(w, dev, seed, logits=lg)
    copies, per = make_copies(base, w, dev)
    del base
    G = max(1, min(CHUNK, n_steps))
    loop = StepLoop(E, p, w, copies, st_h, dev, G)
    flag, R, st0 = loop.warm_eager(3)
    g = loop.capture(G)
    warm_replay(g, 50.0)
    reps = max(1, n_steps // G)
    ms = replay_ms([g] * reps, dev)
    loop.check()
    kern = time_kernels(E, p, w, copies, st0, dev, min(2000, max(50, n_steps)), lm_head=False)
    del g, loop, copies
    torch.cuda.empty_cache()
    return summarise_config(w, reps * G / (ms / 1e3), flag, R, kern, per, inputs)


def summarise_config(w, steps_per_s, flag, R, kern, per_copy_bytes, inputs) -> dict:
    """One `configs` entry: the step rate and each kernel against its binding roofline."""
    pk = peaks()
    alg = algorithmic(w, R)
    ent_gbs = alg["entropy_decode_bytes"] / (kern["entropy_decode_us"] * 1e3)
    att_gbs = alg["partial_attention_bytes"] / (kern["partial_attention_us"] * 1e3)
    att_tfs = alg["partial_attention_flops"] / (kern["partial_attention_us"] * 1e6)
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    intensity = alg["partial_attention_flops"] / alg["partial_attention_bytes"]
    att_bound = "tensor" if intensity > ridge else "hbm"
    extra = {}
    if "dense_attention_us" in kern:  # the two-tile dense kernel on the same full step
        d_tfs = alg["partial_attention_flops"] / (kern["dense_attention_us"] * 1e6)
        extra["dense_attention"] = {"us": kern["dense_attention_us"], "TFLOP/s": d_tfs,
                                    "frac_bf16": d_tfs / pk["bf16_tflops"],
                                    "kernel": "ec_dense_attention (two query tiles per CTA, a softmax warpgroup each)"}
    return {
        "workload": workload_desc(w),
        "step": f"{'full' if flag else 'partial'} (R={R} over the batch)",
        "steps_per_s": steps_per_s,
        "us_per_step": 1e6 / steps_per_s,
        "inputs": inputs,
        "l2": (f"inputs rotate over copies of {per_copy_bytes / 1e6:.1f} MB, at least {ROTATION_BYTES >> 20} MB "
               f"touched per rotation (logits + K/V cache); the per-kernel times rotate over their own inputs"),
        "entropy_decode": {"us": kern["entropy_decode_us"], "GB/s": ent_gbs, "frac_hbm": ent_gbs / pk["hbm_gbs"],
                           "read_floor_us": kern["read_floor_us"],
                           "read_floor_frac_hbm": alg["entropy_decode_bytes"] / (kern["read_floor_us"] * 1e3) / pk["hbm_gbs"],
                           "of_read_floor": kern["read_floor_us"] / kern["entropy_decode_us"]},
        "partial_attention": {"us": kern["partial_attention_us"], "GB/s": att_gbs, "TFLOP/s": att_tfs,
                              "flop_per_byte": intensity, "bound": att_bound,
                              "frac_hbm": att_gbs / pk["hbm_gbs"], "frac_bf16": att_tfs / pk["bf16_tflops"],
                              "frac_bound": (att_tfs / pk["bf16_tflops"]) if att_bound == "tensor"
                              else att_gbs / pk["hbm_gbs"]},
        "kv_scatter": {"us": kern["kv_scatter_us"]},
        "decision_us": kern["entropy_decode_us"],
        **extra,
    }


def trace_logits_device(w, step, gen, dev):
    """Candidate logits of one step of the decode trace, drawn on the device with the trace
    recipe of the workloads module (high-entropy steps N(0, 0.5^2); low ones N(0, 1) with one
    peak per row of height 17.25 - 0.25 (c - 1 - i)), bf16."""
    import torch

    B, C, V = w.B, w.C_max, w.V
    out = torch.empty(B, C, V, dtype=torch.float32, device=dev)
    c = w.block - step % w.block
    height = (17.25 - 0.25 * (c - 1 - torch.arange(C, device=dev))).float()
    for b in range(B):
        if W.trace_is_high(w, step, b):
            out[b] = torch.randn(C, V, generator=gen, device=dev) * 0.5
        else:
            out[b] = torch.randn(C, V, generator=gen, device=dev)
            peak = torch.randint(0, V, (C,), generator=gen, device=dev)
            out[b, torch.arange(C, device=dev), peak] = height
    return out.to(torch.bfloat16)


def run_trace(E, dev, n_steps) -> dict:
    """A timed stretch of the 256-step decode trace over the 32-layer LLaDA-shaped attention
    stack (B 4, 32 x 128, L 4096): the first n_steps steps of the trajectory, each one ec_step
    over all 32 layers, replayed from one CUDA graph (state restored inside). The same stretch
    with no layers (stages (a)-(c) alone) gives the decision share of the step time."""
    import torch

    w = W.workload(4)
    p = params_of(E, w)
    st_h = W.snapshot_state(w)
    gen = torch.Generator(device=dev).manual_seed(w.seed)
    layers = []
    for l in range(w.n_layers):
        d = device_inputs(w, dev, 1000 + l)
        d["out"] = torch.zeros(w.B, w.L, w.Hq, w.D, dtype=torch.bfloat16, device=dev)
        layers.append(d)
    logits = [trace_logits_device(w, t, gen, dev) for t in range(n_steps)]
    ws = E.workspace(E.step_workspace_size(p), dev)
    init = dict(tokens=st_h["tokens"], mask=st_h["mask"], ring=st_h["ring"], ring_head=st_h["ring_head"],
                ring_count=st_h["ring_count"])
    pristine = E.DecodeState.from_arrays(p, device=dev, **init)
    st = pristine.clone()
    # discovery pass: each step's candidates are the still-masked positions of its block
    cands, n_full = [], 0
    mask = st_h["mask"].copy()
    for t in range(n_steps):
        cp, cc = W.trace_candidates(w, mask, t)
        cands.append((torch.from_numpy(cp).to(dev), torch.from_numpy(cc).to(dev)))
        E.step(p, st, logits[t].view(w.B * w.C_max, w.V), cands[t][0], cands[t][1], layers, ws=ws)
        mask = st.mask.cpu().numpy()
        n_full += int(st.flag.sum().item())
    status, word = E.read_device_error(st.dev_err)
    if status != 0:
        raise RuntimeError(f"device error word {word:#x} in the trace")

    def capture(with_layers):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for f in E.DecodeState.FIELDS:
                    getattr(st, f).copy_(getattr(pristine, f))
                for t in range(n_steps):
                    E.step(p, st, logits[t].view(w.B * w.C_max, w.V), cands[t][0], cands[t][1],
                           layers if with_layers else [], ws=ws)
        torch.cuda.current_stream().wait_stream(s)
        return g

    g_all, g_dec = capture(True), capture(False)
    g_all.replay()
    g_dec.replay()
    torch.cuda.synchronize()
    t_all = statistics.median(replay_ms([g_all], dev) for _ in range(3))
    t_dec = statistics.median(replay_ms([g_dec] * 10, dev) / 10 for _ in range(3))
    status, word = E.read_device_error(st.dev_err)
    if status != 0:
        raise RuntimeError(f"device error word {word:#x} in the timed trace")
    del g_all, g_dec, layers, logits
    torch.cuda.empty_cache()
    return {
        "workload": (f"{w.name}: B{w.B}, {w.Hq}x{w.D} MHA, {w.n_layers} layers, L={w.L} ({w.prompt}+{w.gen}, block "
                     f"{w.block}), k={w.k}, V={w.V} bf16 logits, tau={w.tau}; steps 0..{n_steps - 1} of {w.steps}"),
        "steps": n_steps,
        "full_fraction": n_full / (n_steps * w.B),
        "steps_per_s": n_steps / (t_all / 1e3),
        "ms_per_step": t_all / n_steps,
        "decision_us_per_step": t_dec * 1e3 / n_steps,
        "decision_share": t_dec / t_all,
        "decision": "stages (a)-(c1): the decode kernel and the select kernel, timed as the same steps with no layers",
        "inputs": "K/V/Q drawn on the device per layer; logits drawn on the device with the trace recipe",
    }


def layer_setup(E, dev):
    """One LLaDA-8B-shaped layer (d 4096, 32 x 128 MHA, d_ff 12288, L 1024; weights drawn on the
    device at the usual initialisation scale) and the headline step's recompute set, chosen by
    the library's own select stage: (params, weights, x_src, k, v, idx, R, d_ff, workload)."""
    import torch

    w = W.workload(2)
    d, dff, L = w.Hq * w.D, 12288, w.L
    p = params_of(E, w)
    g = torch.Generator(device=dev).manual_seed(7)
    bf = torch.bfloat16

    def mat(r, c):
        return (torch.randn(r, c, generator=g, device=dev) / c ** 0.5).to(bf)

    cs, sn = E.rope_table(L, w.D, 500000.0, device=dev)
    lw = E.LayerWeights(wq=mat(d, d), wk=mat(w.Hkv * w.D, d), wv=mat(w.Hkv * w.D, d), wo=mat(d, d),
                        wg=mat(dff, d), wu=mat(dff, d), wd=mat(d, dff),
                        gamma1=(1 + 0.1 * torch.randn(d, generator=g, device=dev)).to(bf),
                        gamma2=(1 + 0.1 * torch.randn(d, generator=g, device=dev)).to(bf), rope_cos=cs, rope_sin=sn)
    x_src = torch.randn(1, L, d, generator=g, device=dev).to(bf)
    kc = torch.randn(1, L, w.Hkv, w.D, generator=g, device=dev).to(bf)
    vc = torch.randn(1, L, w.Hkv, w.D, generator=g, device=dev).to(bf)
    # the headline step's recompute set, from the library's own select stage
    st_h = W.snapshot_state(w)
    base, _, _ = host_inputs(w, dev)
    st = E.DecodeState.from_arrays(p, device=dev, tokens=st_h["tokens"], mask=st_h["mask"], ring=st_h["ring"],
                                   ring_head=st_h["ring_head"], ring_count=st_h["ring_count"])
    E.step(p, st, base["logits"], torch.from_numpy(st_h["cand_pos"]).to(dev),
           torch.from_numpy(st_h["cand_count"]).to(dev), [], ws=E.workspace(E.step_workspace_size(p), dev))
    torch.cuda.synchronize()
    del base
    return p, lw, x_src, kc, vc, st.idx, st.R, dff, w


def full_step_pattern(n, rate):
    """Which of n steps are full when a fraction `rate` of them is: round(rate * n) full steps
    spread evenly over the n (step i is full when floor((i + 1) * m / n) > floor(i * m / n))."""
    m = round(rate * n)
    return [(i + 1) * m // n > i * m // n for i in range(n)]


def run_layer_forward(E, dev, n_steps) -> dict:
    """The partial forward of one LLaDA-8B-shaped layer for the headline step's recompute set
    (R = 95), against the full forward (R = L): the time per layer of the forward each flag
    selects, and its roofline (weight bytes for the partial forward, tensor-core flops for the
    full one). Then the time per layer over a run of steps in which a given fraction are full
    (the flag rate), against a run of full steps only. Graph-replayed."""
    import torch

    p, lw, x_src, kc, vc, idx_p, R_p, dff, w = layer_setup(E, dev)
    d, L, bf = w.Hq * w.D, w.L, torch.bfloat16
    ws = E.workspace(E.layer_forward_workspace_size(p, dff), dev)
    y = torch.empty(1, L, d, dtype=bf, device=dev)
    out = {}
    full_idx = torch.arange(L, dtype=torch.int32, device=dev).view(1, L)
    R_full = torch.tensor([L], dtype=torch.int32, device=dev)

    def time_run(pattern):
        """Mean time per layer forward over one graph of the pattern's steps (True = full)."""
        for full in sorted(set(pattern)):
            E.layer_forward(p, lw, full_idx if full else idx_p, R_full if full else R_p, x_src, kc, vc, y=y, ws=ws)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(gr, stream=s):
                for full in pattern:
                    E.layer_forward(p, lw, full_idx if full else idx_p, R_full if full else R_p, x_src, kc, vc,
                                    y=y, ws=ws)
        torch.cuda.current_stream().wait_stream(s)
        warm_replay(gr, 50.0)
        us = statistics.median(replay_ms([gr], dev) for _ in range(3)) * 1e3 / len(pattern)
        del gr
        return us

    for name, idx, R in (("partial", idx_p, R_p), ("full", full_idx, R_full)):
        n = n_steps if name == "partial" else max(10, n_steps // 8)
        us = time_run([name == "full"] * n)
        rows = int(R.sum().item())
        params = d * (d + 2 * w.Hkv * w.D) + d * d + 3 * d * dff
        wbytes = 2 * params
        flops = 2 * rows * params + 4 * w.Hq * rows * L * w.D
        pk = peaks()
        out[name] = {"R": rows, "us": us, "weight_GB/s": wbytes / (us * 1e3), "TFLOP/s": flops / (us * 1e6),
                     "frac_hbm": wbytes / (us * 1e3) / pk["hbm_gbs"], "frac_bf16": flops / (us * 1e6) / pk["bf16_tflops"]}
    out["full_over_partial"] = out["full"]["us"] / out["partial"]["us"]
    n_mix = 40
    by_rate = {}
    for rate in (0.0, 0.1, 0.25, 0.5, 1.0):
        us = time_run(full_step_pattern(n_mix, rate))
        by_rate[f"{rate:g}"] = {"us_per_layer": us, "speedup_vs_all_full": None}
    for v in by_rate.values():
        v["speedup_vs_all_full"] = by_rate["1"]["us_per_layer"] / v["us_per_layer"]
    out["by_flag_rate"] = by_rate
    out["by_flag_rate_run"] = (f"{n_mix} layer forwards per graph, the given fraction of them full (R = L) and spread "
                               f"evenly, the rest partial (R = {int(R_p.sum().item())})")
    out["workload"] = (f"one LLaDA-8B-shaped layer: d {d}, {w.Hq} x {w.D} MHA, d_ff {dff}, L {L}; RMSNorm, QKV + RoPE, "
                       f"K/V refresh, attention, O-proj + residual, RMSNorm, SwiGLU, down + residual")
    out["weights_MB"] = 2 * (d * (d + 2 * w.Hkv * w.D) + d * d + 3 * d * dff) / 1e6
    del lw, ws
    torch.cuda.empty_cache()
    return out


def run_configs(E, dev, args) -> dict:
    """Every synthetic workload besides the headline: workload 1 (tiny, fp32 logits), the
    headline layer with tau below every entropy (a full step, R = L), workload 3 (the Dream-7B
    GQA batch), workload 5 (the 32K-row cache) and a stretch of the workload-4 trace."""
    out = {}
    out["tiny"] = config_entry(E, W.workload(1), dev, 2000, "host", 1)
    out["llada_layer_full"] = config_entry(E, W.workload(2).scaled(tau=-1.0), dev, 500, "host", 2)
    out["dream_gqa"] = config_entry(E, W.workload(3), dev, 50, "device", 3)
    out["long_context"] = config_entry(E, W.workload(5), dev, 500, "device", 5)
    out["llada_trace"] = run_trace(E, dev, args.trace_steps)
    out["llada_layer_forward"] = run_layer_forward(E, dev, 200)
    return out


def time_kernels(E, p, w, copies, st0, dev, n, lm_head=True) -> dict:
    """Average duration of each stage's kernel, timed alone through its own entry point over
    the rotating input copies (CUDA events on the launching stream, graph-replayed)."""
    import torch

    rows = w.B * w.C_max
    R = st0.R.clone()
    idx = st0.idx.clone()
    out = {}
    ent_ws = E.workspace(E.entropy_decode_workspace_size(rows, w.V, w.logits_dtype), dev)
    att_ws = E.workspace(E.partial_attention_workspace_size(p), dev)
    ids = torch.empty(rows, dtype=torch.int32, device=dev)
    ent = torch.empty(rows, dtype=torch.float32, device=dev)
    conf = torch.empty(rows, dtype=torch.float32, device=dev)
    # recompute-row queries in idx order, as the step's gather leaves them
    c0 = copies[0]
    qfull = torch.zeros(w.B, w.L, w.Hq, w.D, dtype=torch.bfloat16, device=dev)
    for b in range(w.B):
        r = int(R[b].item())
        qfull[b, :r] = c0["q_src"][b, idx[b, :r].long()]
    # each stage rotates over its own inputs, enough copies that they cannot stay in L2
    lg_bytes = c0["logits"].numel() * c0["logits"].element_size()
    n_lg = max(1, min(64, -(-ROTATION_BYTES // lg_bytes)))
    logits_rot = [copies[i]["logits"] if i < len(copies) else c0["logits"].clone() for i in range(n_lg)]
    kv_bytes = 2 * c0["k_cache"].numel() * c0["k_cache"].element_size()
    n_kv = max(1, min(64, -(-ROTATION_BYTES // kv_bytes)))
    kv_rot = [(copies[i]["k_cache"], copies[i]["v_cache"]) if i < len(copies) else
              (c0["k_cache"].clone(), c0["v_cache"].clone()) for i in range(n_kv)]
    att_out = torch.zeros(w.B, w.L, w.Hq, w.D, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()

    nc = len(copies)

    def stage_entropy(i):
        E.entropy_decode(logits_rot[i % n_lg].view(rows, w.V), ws=ent_ws, out=(ids, ent, conf))

    def stage_attention(i):
        kc, vc = kv_rot[i % n_kv]
        E.partial_attention(p, qfull, kc, vc, R, att_out, ws=att_ws)

    def stage_scatter(i):
        c = copies[i % nc]
        E.kv_scatter(p, c["k_cache"], c["v_cache"], c["k_src"], c["v_src"], idx, R, src_by_position=True)

    sink = torch.zeros(4, dtype=torch.int32, device=dev)

    def stage_floor(i):  # a plain read of the same logits in the decode's launch shape
        E.read_floor(logits_rot[i % n_lg], sink)

    def timed(fn, n):
        G = min(n, CHUNK)
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(G):
                    fn(i)
        torch.cuda.current_stream().wait_stream(s)
        g.replay()
        torch.cuda.synchronize()
        reps = max(1, n // G)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * G)  # us per launch

    # stage (a) from the hidden states: the output projection fused with the decode, on a
    # random bf16 weight of the model's shape (V x d_model, about 1 GB: no L2 reuse)
    if lm_head and w.d_model > 0:
        g = torch.Generator(device=dev).manual_seed(w.seed)
        hid = torch.randn(rows, w.d_model, device=dev, generator=g).to(torch.bfloat16)
        wt = (torch.randn(w.V, w.d_model, device=dev, generator=g) / w.d_model ** 0.5).to(torch.bfloat16)
        lm_ws = E.workspace(E.lm_head_entropy_workspace_size(rows), dev)

        def stage_lm_head(i):
            E.lm_head_entropy(hid, wt, ws=lm_ws, out=(ids, ent, conf))

        out["lm_head_entropy_us"] = timed(stage_lm_head, min(n, 200))
        out["lm_head_bytes"] = (w.V + rows) * w.d_model * 2
        del wt
    out["entropy_decode_us"] = timed(stage_entropy, n)
    out["read_floor_us"] = timed(stage_floor, n)
    out["partial_attention_us"] = timed(stage_attention, n)
    if int(R.sum().item()) == w.B * w.L and w.D == 128:  # a full step: the dense kernel too
        def stage_dense(i):
            kc, vc = kv_rot[i % n_kv]
            E.dense_attention(p, qfull, kc, vc, att_out)

        out["dense_attention_us"] = timed(stage_dense, n)
    out["kv_scatter_us"] = timed(stage_scatter, n)
    out["R"] = int(R.sum().item())  # recompute rows over the batch
    out["rotations"] = {"steps": nc, "logits": n_lg, "kv_cache": n_kv}
    del logits_rot, kv_rot, qfull, att_out
    return out


def flat_state(E, p, dev, **arrays):
    """A DecodeState whose fields are views of one flat device buffer (256-byte aligned), so
    that it is restored with one copy; E, flag and R are adjacent at the end, so that they read
    back as one slice. Returns (state, flat buffer, (start, end) byte range of E..R)."""
    import torch

    B, L, k = p.B, p.L, p.k
    spec = [("tokens", torch.int32, (B, L)), ("mask", torch.uint8, (B, L)), ("ring", torch.int32, (B, k)),
            ("ring_head", torch.int32, (B,)), ("ring_count", torch.int32, (B,)), ("dec_pos", torch.int32, (B, p.n_dec)),
            ("idx", torch.int32, (B, L)), ("dev_err", torch.int32, (1,)), ("E", torch.float32, (B,)),
            ("flag", torch.int32, (B,)), ("R", torch.int32, (B,))]
    offs, off = {}, 0
    for name, dt, shape in spec:
        nb = int(np.prod(shape)) * torch.tensor([], dtype=dt).element_size()
        offs[name] = (off, nb)
        off += (nb + 255) // 256 * 256 if name not in ("E", "flag") else nb
    flat = torch.zeros(off, dtype=torch.uint8, device=dev)
    st = object.__new__(E.DecodeState)
    for name, dt, shape in spec:
        o, nb = offs[name]
        t = flat[o:o + nb].view(dt).view(shape)
        setattr(st, name, t)
    # flag is one byte per sequence in the ABI: keep a uint8 view over the first bytes of its slot
    o, _ = offs["flag"]
    st.flag = flat[o:o + B]
    for name, a in arrays.items():
        getattr(st, name).copy_(torch.as_tensor(a).to(getattr(st, name).dtype))
    return st, flat, (offs["E"][0], offs["R"][0] + offs["R"][1])


def run_e2e(E, p, w, lay_h, lg_h, st_h, dev, n) -> dict:
    """ec_step end to end from pinned host buffers, pipelined as a serving loop would run it:
    every step copies its inputs host->device (one copy of one pinned blob) and reads its
    results back (the output rows and R / flag / E), with step i+1's upload and step i-1's
    readback on two copy streams overlapping step i's kernels. Device inputs and outputs are
    double-buffered; events order each buffer's reuse."""
    import torch

    bf = torch.bfloat16
    parts = [("logits", lg_h)] + [
        (k_, lay_h[k_]) for k_ in ("k_src", "v_src", "q_src")]
    offs, off = {}, 0
    for k_, a in parts:
        nb = np.ascontiguousarray(a).nbytes
        offs[k_] = (off, nb, a.shape)
        off += (nb + 255) // 256 * 256
    blob_h = torch.empty(off, dtype=torch.uint8).pin_memory()
    for k_, a in parts:
        o, nb, _ = offs[k_]
        blob_h[o:o + nb].copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)))
    blob_d = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]

    def view(blob, k_, dt):
        o, nb, shape = offs[k_]
        return blob[o:o + nb].view(dt).view(shape)

    kc = torch.from_numpy(lay_h["k_cache"].view(np.int16)).to(dev)
    vc = torch.from_numpy(lay_h["v_cache"].view(np.int16)).to(dev)
    out = [torch.empty(w.B, w.L, w.Hq, w.D, dtype=bf, device=dev) for _ in range(2)]
    out_h = [torch.empty(w.B, w.L, w.Hq, w.D, dtype=bf).pin_memory() for _ in range(2)]
    cand_pos = torch.from_numpy(st_h["cand_pos"]).to(dev)
    cand_count = torch.from_numpy(st_h["cand_count"]).to(dev)
    ws = E.workspace(E.step_workspace_size(p), dev)
    init = dict(tokens=st_h["tokens"], mask=st_h["mask"], ring=st_h["ring"], ring_head=st_h["ring_head"],
                ring_count=st_h["ring_count"])
    _, pristine_flat, _ = flat_state(E, p, dev, **init)
    st, st_flat, (r0, r1) = flat_state(E, p, dev, **init)
    small = [torch.empty(r1 - r0, dtype=torch.uint8, device=dev) for _ in range(2)]
    small_h = [torch.empty(r1 - r0, dtype=torch.uint8).pin_memory() for _ in range(2)]
    h2d = off
    d2h = out[0].numel() * 2 + (r1 - r0)
    s_in, s_cp, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, done, out_read = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    started = [False, False]

    def step(i):
        sl = i & 1
        with torch.cuda.stream(s_in):
            if started[sl]:
                s_in.wait_event(done[sl])  # the step two back has consumed this input buffer
            blob_d[sl].copy_(blob_h, non_blocking=True)
            in_ready[sl].record(s_in)
        with torch.cuda.stream(s_cp):
            s_cp.wait_event(in_ready[sl])
            if started[sl]:
                s_cp.wait_event(out_read[sl])  # its outputs have been read back
            st_flat.copy_(pristine_flat, non_blocking=True)  # the same starting state every step
            lg = view(blob_d[sl], "logits", bf if w.logits_dtype == "bf16" else torch.float32)
            E.step(p, st, lg, cand_pos, cand_count,
                   [dict(k_cache=kc.view(bf), v_cache=vc.view(bf), k_src=view(blob_d[sl], "k_src", bf),
                         v_src=view(blob_d[sl], "v_src", bf), q_src=view(blob_d[sl], "q_src", bf), out=out[sl])],
                   ws=ws, stream=s_cp)
            small[sl].copy_(st_flat[r0:r1], non_blocking=True)  # E, flag, R
            done[sl].record(s_cp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[sl])
            out_h[sl].copy_(out[sl], non_blocking=True)
            small_h[sl].copy_(small[sl], non_blocking=True)
            out_read[sl].record(s_out)
        started[sl] = True

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream(dev)
    a.record(cur)
    for s_ in (s_in, s_cp, s_out):
        s_.wait_stream(cur)
    for i in range(n):
        step(i)
    for s_ in (s_in, s_cp, s_out):
        cur.wait_stream(s_)
    b.record(cur)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    return {"value": n / (ms / 1e3), "unit": "steps/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": n, "pipelined": "upload of step i+1 and readback of step i-1 overlap step i"}


def algorithmic(w, R) -> dict:
    """Algorithmic bytes / flops per launch of each stage; R = recompute rows over the batch."""
    esz = 2 if w.logits_dtype == "bf16" else 4
    kv_row = w.Hkv * w.D * 2
    q_row = w.Hq * w.D * 2
    return {
        "entropy_decode_bytes": w.B * w.C_max * w.V * esz + w.B * w.C_max * 12,
        "partial_attention_bytes": w.B * 2 * w.L * kv_row + 2 * R * q_row,
        "partial_attention_flops": 4 * w.Hq * R * w.L * w.D,
        "kv_scatter_bytes": R * (4 * kv_row + 2 * q_row),
    }


def emit_ours(args, res, rank, world):
    w = bench_workload(args)
    pk = peaks()
    K = args.steps
    ms_per_step = res["ms"] / K
    value = job_throughput(world, K, res["ms"])
    kern = res["kernels"]
    alg = algorithmic(w, kern["R"])
    ent_gbs = alg["entropy_decode_bytes"] / (kern["entropy_decode_us"] * 1e-6) / 1e9
    att_gbs = alg["partial_attention_bytes"] / (kern["partial_attention_us"] * 1e-6) / 1e9
    att_tfs = alg["partial_attention_flops"] / (kern["partial_attention_us"] * 1e-6) / 1e12
    sc_gbs = alg["kv_scatter_bytes"] / (kern["kv_scatter_us"] * 1e-6) / 1e9
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    att_tensor = alg["partial_attention_flops"] / alg["partial_attention_bytes"] > ridge
    att_roof = ({"bound": "tensor", "achieved": att_tfs, "peak": pk["bf16_tflops"], "unit": "TFLOP/s"} if att_tensor
                else {"bound": "hbm", "achieved": att_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s"})
    cands = {
        "entropy_decode": (kern["entropy_decode_us"], {"bound": "hbm", "achieved": ent_gbs, "peak": pk["hbm_gbs"],
                                                       "unit": "GB/s"}),
        "partial_attention": (kern["partial_attention_us"], att_roof),
    }
    dom = max(cands, key=lambda k_: cands[k_][0])
    roof = dict(cands[dom][1])
    roof["kernel"] = dom
    roof["frac"] = roof["achieved"] / roof["peak"]
    src = {"entropy_decode": "entropy_decode.cu", "partial_attention": "attention.cu"}[dom]
    roof["traffic"] = profiled_traffic(dom, src) if args.workload == WORKLOAD and args.tau is None else None
    roof["peak_source"] = pk["source"] + " (burst; kernel timed alone)"
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "steps/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_desc(w), "step": f"{'full' if res['flag'] else 'partial'} (R={res['R']} over the batch)",
                   "l2": (f"inputs rotate over {res['ncopy']} copies of {res['copy_mb']:.0f} MB, {res['touched_mb']:.0f} MB "
                          f"touched per step (logits + K/V cache): {res['ncopy'] * res['touched_mb']:.0f} MB per rotation, "
                          f"L2 is 129 MB; the per-kernel times rotate over {ROTATION_BYTES >> 20} MB of their own inputs"),
                   "timing": (f"CUDA graphs of {min(CHUNK, K)} steps, state restore inside, after at least 100 ms "
                              f"of untimed replays")},
        "roofline": roof,
        "kernels": {
            "entropy_decode": {"us": kern["entropy_decode_us"], "GB/s": ent_gbs, "frac_hbm": ent_gbs / pk["hbm_gbs"],
                               "read_floor_us": kern["read_floor_us"],
                               "read_floor_frac_hbm": alg["entropy_decode_bytes"] / (kern["read_floor_us"] * 1e3) / pk["hbm_gbs"],
                               "of_read_floor": kern["read_floor_us"] / kern["entropy_decode_us"]},
            "partial_attention": {"us": kern["partial_attention_us"], "GB/s": att_gbs, "TFLOP/s": att_tfs,
                                  "frac_hbm": att_gbs / pk["hbm_gbs"], "frac_bf16": att_tfs / pk["bf16_tflops"]},
            "kv_scatter": {"us": kern["kv_scatter_us"], "GB/s": sc_gbs},
        },
        "e2e": res["e2e"],
        "gpu_launches": 4 * K,
        "clocks": res["clocks"],
    }
    if "steady" in res:
        line["steady"] = res["steady"]
    targets = {"entropy_decode_hbm": {"kernel": "entropy_decode", "workload": w.name, "frac": ent_gbs / pk["hbm_gbs"],
                                      "goal": 0.70, "of": "measured HBM copy bandwidth",
                                      "read_floor_frac": alg["entropy_decode_bytes"] / (kern["read_floor_us"] * 1e3)
                                      / pk["hbm_gbs"]}}
    cfg = res.get("configs") or {}
    if "llada_layer_full" in cfg:
        fa = cfg["llada_layer_full"]["partial_attention"]
        targets["attention_bf16"] = {"kernel": "partial_attention", "workload": "llada_layer, full step (R = L)",
                                     "frac": fa["frac_bf16"], "goal": 0.50, "of": "measured bf16 dense (cuBLAS burst)"}
        da = cfg["llada_layer_full"].get("dense_attention")
        if da:  # the kernel for steps known to be full, on the same step
            targets["attention_bf16"]["dense_attention_frac"] = da["frac_bf16"]
    if "dream_gqa" in cfg:
        targets["entropy_decode_hbm_dream"] = {"kernel": "entropy_decode", "workload": "dream_gqa (78 MB)",
                                               "frac": cfg["dream_gqa"]["entropy_decode"]["frac_hbm"],
                                               "goal": 0.70, "of": "measured HBM copy bandwidth",
                                               "read_floor_frac": cfg["dream_gqa"]["entropy_decode"]["read_floor_frac_hbm"]}
    line["targets"] = targets
    if cfg:
        line["configs"] = cfg
    if "lm_head_entropy_us" in kern:  # not part of the timed step, which starts from logits
        lm_gbs = kern["lm_head_bytes"] / (kern["lm_head_entropy_us"] * 1e3)
        line["kernels"]["lm_head_entropy"] = {"us": kern["lm_head_entropy_us"], "GB/s": lm_gbs,
                                              "frac_hbm": lm_gbs / pk["hbm_gbs"], "d_model": w.d_model}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    print(json.dumps(line))


# --------------------------------------------------------------------------------------
# oracle timing (reference arm and cpu_baseline)


class OracleStep:
    """The float64 oracle's whole step on the headline workload: decode and entropy of every
    candidate row, commit, gate, history, recompute set, K/V refresh and attention of every
    recompute row over all heads (oracle.step). Nothing is sampled."""

    def __init__(self):
        import oracle as O

        self.O = O
        w = W.workload(WORKLOAD)
        self.w = w
        self.st = W.snapshot_state(w)
        self.x = O.widen(W.step_logits(w)[0], w.logits_dtype)
        lay = W.layer_tensors(w, 0)
        self.layer = {n: O.widen(lay[n][0], "bf16") for n in ("k_cache", "v_cache", "k_src", "v_src", "q_src")}

    def run(self) -> dict:
        st = self.st
        return self.O.step(logits=self.x, cand_pos=st["cand_pos"][0], cand_count=int(st["cand_count"][0]),
                           tokens=st["tokens"][0], mask=st["mask"][0], ring=st["ring"][0],
                           ring_head=int(st["ring_head"][0]), ring_count=int(st["ring_count"][0]),
                           n_dec=self.w.n_dec, tau=self.w.tau, layers=[self.layer])


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def time_oracle(os_: OracleStep, n: int | None = None, budget_s: float | None = None) -> dict:
    """Runs whole oracle steps (n of them, or as many as fit in budget_s) and returns the rate,
    the wall time and the threads actually used (process CPU time over wall time: NumPy's BLAS
    may run the attention products on several threads)."""
    c0, t0 = time.process_time(), time.perf_counter()
    k = 0
    while (n is not None and k < n) or (budget_s is not None and (k < 1 or time.perf_counter() - t0 < budget_s)):
        os_.run()
        k += 1
    wall = time.perf_counter() - t0
    cpu = time.process_time() - c0
    return {"steps": k, "wall_s": wall, "rate": k / wall, "threads": max(1, round(cpu / wall))}


def cpu_baseline(budget_s: float = 15.0) -> dict:
    os_ = OracleStep()
    os_.run()  # warm
    r = time_oracle(os_, budget_s=budget_s)
    return {"value": r["rate"], "unit": "steps/s", "cores": r["threads"], "cores_available": cpu_cores(),
            "kind": "oracle",
            "sample": (f"full step: {r['steps']} whole float64 oracle steps of the headline workload (all "
                       f"{int(os_.st['cand_count'][0])} candidate rows, every recompute row over all heads), "
                       f"no sampling; cores = process CPU time / wall time"), "wall_s": r["wall_s"]}


def run_reference(args) -> None:
    os_ = OracleStep()
    K, Wm = args.steps, args.warmup
    t0 = time.perf_counter()
    os_.run()
    t_step = time.perf_counter() - t0
    budget = 150.0  # the whole --steps K --warmup W run stays within a few minutes
    if (K + Wm) * t_step <= budget:
        for _ in range(Wm):
            os_.run()
        r = time_oracle(os_, n=K)
        sample = f"full step: each of {K} steps is a whole float64 oracle step, no sampling"
    else:  # K too large to run in full: time as many whole steps as the budget allows
        for _ in range(min(Wm, 3)):
            os_.run()
        r = time_oracle(os_, budget_s=budget)
        sample = (f"full steps: {r['steps']} whole float64 oracle steps timed within a {budget:.0f} s budget (the "
                  f"{K} requested steps would take {K * t_step:.0f} s); value = their rate")
    value = r["rate"]
    w = W.workload(WORKLOAD)
    cb = {"value": value, "unit": "steps/s", "cores": r["threads"], "cores_available": cpu_cores(), "kind": "oracle",
          "sample": sample + "; cores = process CPU time / wall time", "wall_s": r["wall_s"]}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": 1, "steps": K,
            "warmup": Wm, "ms_per_step": 1e3 / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(w), "step": "partial (R=95 over the batch)",
                       "l2": "host memory (CPU oracle)", "timing": "wall clock over whole oracle steps"},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--workload", type=int, default=WORKLOAD, choices=[1, 2, 3, 5],
                    help="workload to time (default 2, the LLaDA-8B layer step)")
    ap.add_argument("--tau", type=float, default=None, help="override tau (e.g. -1 forces a full step)")
    ap.add_argument("--no-configs", action="store_true", help="time only the headline workload")
    ap.add_argument("--trace-steps", type=int, default=64, help="steps of the decode trace timed under configs")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="run this many eager steps and exit (a short program for ncu)")
    args = ap.parse_args()
    if args.profile_steps > 0:
        run_profile(args.profile_steps, args.workload, args.tau)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    init_ranks(world)
    res = run_ours(args, rank, world)
    if rank == 0:
        emit_ours(args, res, rank, world)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
