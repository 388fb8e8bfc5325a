"""Seeded synthetic inputs for the EntropyCache step, shared by the tests and the benchmark.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic. Both the oracle and the CUDA library receive exactly the arrays made here:
bf16 tensors as uint16 bit patterns (rounded to nearest even from float32 draws), fp32 as
float32, integers as int32/uint8.

The five workloads follow the shapes of the models the EntropyCache summaries evaluate
(LLaDA-8B-Instruct, Dream-7B-Instruct; gist.science summaries §4) and the decode-history
example k = 64 (pt summary, lay section "Não esqueça o que acabou de acontecer"). The
benchmark suites the pages evaluate on (GSM8K, MATH500, MBPP, HumanEval, CoT sets) are not
available here; these synthetic distributions stand in for them:

  1 tiny         B1, 8 x 64 MHA, L 256 (128 + 128), V 32000 fp32, k 16
  2 llada_layer  B1, 32 x 128 MHA, L 1024 (768 + 256), V 126464 bf16, k 64
  3 dream_gqa    B8, 28 q / 4 kv x 128, L 2048 (1792 + 256), V 152064 bf16, k 64
  4 llada_trace  B4, 32 x 128 MHA, 32 layers, L 4096 (3840 + 256), V 126464 bf16, k 64,
                 256 steps, ~10% high-entropy steps
  5 long_context B1, 32 x 128 MHA, L 32768 (32512 + 256), V 126464 bf16, k 64

Logit distributions:
  gauss_scale  row i ~ N(0, s_i^2), s_i ~ U[0.5, 8]
  zipf         per row a random permutation gives every token a rank rho in 1..V and
               logit = -1.1 ln rho + N(0, 1)
  schedule     as trace, with the peak heights 17.75 - 0.125 pi(i) for a seeded permutation
               pi of the rows (block-wise and sliding-window decoding tests)
  trace        per (step, sequence) a Bernoulli(0.1) draw (step 0 always high) picks
               high: every row N(0, 0.5^2)  (entropy about ln V)
               low:  every row N(0, 1) except one seeded token set to a peak; with c
                     candidate rows this step (c = 32 - step mod 32), row i's peak is exactly
                     17.25 - 0.25 (c - 1 - i) (exact in bf16), so the most confident row has
                     entropy about 0.05 and the best rows' confidences differ by ~25%
K/V cache, queries ~ N(0, 1); fresh K/V rows = cache + N(0, 0.05^2); all bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "workload",
    "to_bf16_bits",
    "rng_for",
    "snapshot_state",
    "step_logits",
    "layer_pool",
    "layer_tensors",
    "trace_candidates",
    "layer_weights",
    "layer_input",
]


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    B: int
    L: int
    prompt: int
    gen: int
    block: int
    Hq: int
    Hkv: int
    D: int
    V: int
    k: int
    n_dec: int
    tau: float
    logits_dtype: str  # "f32" | "bf16"
    logits_kind: str  # "gauss_scale" | "zipf" | "trace"
    n_layers: int = 1
    steps: int = 1
    seed: int = 0
    d_model: int = 0  # hidden size of the model's output projection (Hq * D for these models)

    @property
    def C_max(self) -> int:
        return self.block

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS: dict[int, Workload] = {
    1: Workload(1, "tiny", B=1, L=256, prompt=128, gen=128, block=32, Hq=8, Hkv=8, D=64,
                V=32000, k=16, n_dec=1, tau=1.0, logits_dtype="f32",
                logits_kind="gauss_scale", seed=1, d_model=512),
    2: Workload(2, "llada_layer", B=1, L=1024, prompt=768, gen=256, block=32, Hq=32, Hkv=32,
                D=128, V=126464, k=64, n_dec=1, tau=1.0, logits_dtype="bf16",
                logits_kind="gauss_scale", seed=2, d_model=4096),
    3: Workload(3, "dream_gqa", B=8, L=2048, prompt=1792, gen=256, block=32, Hq=28, Hkv=4,
                D=128, V=152064, k=64, n_dec=1, tau=1.0, logits_dtype="bf16",
                logits_kind="zipf", seed=3, d_model=3584),
    4: Workload(4, "llada_trace", B=4, L=4096, prompt=3840, gen=256, block=32, Hq=32,
                Hkv=32, D=128, V=126464, k=64, n_dec=1, tau=1.0, logits_dtype="bf16",
                logits_kind="trace", n_layers=32, steps=256, seed=4, d_model=4096),
    5: Workload(5, "long_context", B=1, L=32768, prompt=32512, gen=256, block=32, Hq=32,
                Hkv=32, D=128, V=126464, k=64, n_dec=1, tau=1.0, logits_dtype="bf16",
                logits_kind="gauss_scale", seed=5, d_model=4096),
}


def workload(i: int) -> Workload:
    return WORKLOADS[i]


def rng_for(seed: int, *stream: int) -> np.random.Generator:
    """Independent, order-free random stream for (seed, stream...)."""
    return np.random.default_rng([int(seed), *[int(s) for s in stream]])


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------------------
# decode state


def snapshot_state(w: Workload) -> dict:
    """State at the start of the last generation block (single-step workloads), or at the
    start of generation (the trace).

    Prompt positions and every earlier generation block are decoded; within each decoded
    block the decode order is a seeded permutation. The ring holds the decode order so that
    entry t sits in slot t mod k. Candidates are the masked positions of the current block.
    """
    B, L, k = w.B, w.L, w.k
    tokens = np.full((B, L), -1, dtype=np.int32)
    mask = np.zeros((B, L), dtype=np.uint8)
    ring = np.zeros((B, k), dtype=np.int32)
    head = np.zeros(B, dtype=np.int32)
    count = np.zeros(B, dtype=np.int32)
    cand_pos = np.zeros((B, w.C_max), dtype=np.int32)
    cand_count = np.zeros(B, dtype=np.int32)
    n_blocks = w.gen // w.block
    decoded_blocks = n_blocks - 1 if w.steps == 1 else 0
    for b in range(B):
        r = rng_for(w.seed, 10, b)
        tokens[b, : w.prompt] = r.integers(0, w.V, size=w.prompt, dtype=np.int32)
        mask[b, w.prompt:] = 1
        order: list[int] = []
        for blk in range(decoded_blocks):
            start = w.prompt + blk * w.block
            perm = r.permutation(w.block) + start
            order.extend(int(p) for p in perm)
        for p in order:
            tokens[b, p] = r.integers(0, w.V)
            mask[b, p] = 0
        for t, p in enumerate(order):
            ring[b, t % k] = p
        head[b] = len(order) % k
        count[b] = min(len(order), k)
        cur = w.prompt + decoded_blocks * w.block
        masked_in_block = [p for p in range(cur, cur + w.block) if mask[b, p]]
        cand_pos[b, : len(masked_in_block)] = masked_in_block
        cand_count[b] = len(masked_in_block)
    return {
        "tokens": tokens,
        "mask": mask,
        "ring": ring,
        "ring_head": head,
        "ring_count": count,
        "cand_pos": cand_pos,
        "cand_count": cand_count,
    }


def trace_candidates(w: Workload, mask: np.ndarray, step: int) -> tuple[np.ndarray, np.ndarray]:
    """Candidates of a trace step: the still-masked positions of the current block."""
    blk = step // w.block
    start = w.prompt + blk * w.block
    cand_pos = np.zeros((w.B, w.C_max), dtype=np.int32)
    cand_count = np.zeros(w.B, dtype=np.int32)
    for b in range(w.B):
        ps = [p for p in range(start, start + w.block) if mask[b, p]]
        cand_pos[b, : len(ps)] = ps
        cand_count[b] = len(ps)
    return cand_pos, cand_count


# --------------------------------------------------------------------------------------
# logits


def _finish_logits(w: Workload, x: np.ndarray) -> np.ndarray:
    if w.logits_dtype == "bf16":
        return to_bf16_bits(x)
    return np.ascontiguousarray(x, dtype=np.float32)


def trace_is_high(w: Workload, step: int, b: int) -> bool:
    if step == 0:
        return True
    return bool(rng_for(w.seed, 30, step, b).random() < 0.1)


def step_logits(w: Workload, step: int = 0) -> np.ndarray:
    """Candidate logits [B, C_max, V] for one step, in stored form."""
    B, C, V = w.B, w.C_max, w.V
    out = np.empty((B, C, V), dtype=np.float32)
    for b in range(B):
        r = rng_for(w.seed, 20, step, b)
        if w.logits_kind == "gauss_scale":
            s = r.uniform(0.5, 8.0, size=C).astype(np.float32)
            out[b] = r.standard_normal((C, V), dtype=np.float32) * s[:, None]
        elif w.logits_kind == "zipf":
            for i in range(C):
                rank = r.permutation(V).astype(np.float32) + np.float32(1.0)
                out[b, i] = np.float32(-1.1) * np.log(rank) + r.standard_normal(V, dtype=np.float32)
        elif w.logits_kind == "schedule":
            # as "trace", but the peak heights 17.75 - 0.125 pi(i) (exact in bf16) follow a
            # seeded permutation pi of the rows, so that the most confident candidate is
            # anywhere in the window, not always the last row. At V = 32000 the best row has
            # entropy below 0.7 and its confidence leads the next one by more than 1e-4 in log
            if trace_is_high(w, step, b):
                out[b] = r.standard_normal((C, V), dtype=np.float32) * np.float32(0.5)
            else:
                out[b] = r.standard_normal((C, V), dtype=np.float32)
                peak = r.integers(0, V, size=C)
                height = 17.75 - 0.125 * r.permutation(C)
                out[b, np.arange(C), peak] = height.astype(np.float32)
        elif w.logits_kind == "trace":
            if trace_is_high(w, step, b):
                out[b] = r.standard_normal((C, V), dtype=np.float32) * np.float32(0.5)
            else:
                out[b] = r.standard_normal((C, V), dtype=np.float32)
                peak = r.integers(0, V, size=C)
                c = w.block - step % w.block
                height = 17.25 - 0.25 * (c - 1 - np.arange(C))
                out[b, np.arange(C), peak] = height.astype(np.float32)
        else:
            raise ValueError(w.logits_kind)
    return _finish_logits(w, out)


# --------------------------------------------------------------------------------------
# per-layer attention tensors


def _normal_bf16(r: np.random.Generator, shape: tuple[int, ...]) -> np.ndarray:
    return to_bf16_bits(r.standard_normal(shape, dtype=np.float32))


def layer_pool(w: Workload) -> dict:
    """One draw of every per-layer tensor (bf16 bit patterns): k_cache, v_cache, k_src, v_src
    [B, L, Hkv, D] and q_src [B, L, Hq, D]; fresh rows k_src/v_src = cache + N(0, 0.05^2)."""
    B, L, Hq, Hkv, D = w.B, w.L, w.Hq, w.Hkv, w.D
    kv_shape = (B, L, Hkv, D)
    q_shape = (B, L, Hq, D)
    out = {}
    for j, name in enumerate(("k_cache", "v_cache")):
        cache = _normal_bf16(rng_for(w.seed, 40, 0, j), kv_shape)
        noise = rng_for(w.seed, 41, 0, j).standard_normal(kv_shape, dtype=np.float32)
        noise *= np.float32(0.05)
        noise += bf16_bits_to_f32(cache)
        out[name] = cache
        out[name.replace("cache", "src")] = to_bf16_bits(noise)
        del noise
    out["q_src"] = _normal_bf16(rng_for(w.seed, 42, 0), q_shape)
    return out


def layer_tensors(w: Workload, layer: int = 0, pool: dict | None = None) -> dict:
    """bf16 bit patterns for one layer (see layer_pool). Layer 0 is the pool itself; layer l > 0
    of a multi-layer workload is a seeded circular shift of the pool, so 32 layers cost one
    draw. Pass `pool` to reuse a draw across calls."""
    base = pool if pool is not None else layer_pool(w)
    if w.n_layers == 1 or layer == 0:
        return dict(base)
    shift = int(rng_for(w.seed, 43, layer).integers(1, 1 << 30))
    out = {}
    for name, a in base.items():
        flat = a.reshape(-1)
        out[name] = np.roll(flat, shift % flat.size).reshape(a.shape)
    return out


def lm_head_inputs(n_rows: int, d_model: int, V: int, seed: int = 0, peaked: int = 0,
                   chunk_rows: int = 8192) -> tuple[np.ndarray, np.ndarray]:
    """Hidden states and an output-projection matrix, as bf16 bit patterns.

    weight [V, d_model] ~ N(0, 1 / d_model) (the usual initialisation scale, so logits are about
    N(0, 1)); hidden [n_rows, d_model] ~ N(0, 1). The first `peaked` rows get a large component
    along a seeded weight row, a confident prediction. Generated in float32 chunks of
    `chunk_rows` vocabulary rows so that a full-size matrix never exists in float64.
    """
    r = rng_for(seed, 41)
    weight = np.empty((V, d_model), dtype=np.uint16)
    for v0 in range(0, V, chunk_rows):
        v1 = min(V, v0 + chunk_rows)
        weight[v0:v1] = to_bf16_bits(r.standard_normal((v1 - v0, d_model), dtype=np.float32) / np.sqrt(d_model))
    hidden = r.standard_normal((n_rows, d_model))
    for i in range(min(peaked, n_rows)):
        v = int(r.integers(0, V))
        wv = bf16_bits_to_f32(weight[v]).astype(np.float64)
        hidden[i] += (12.0 + i) * wv / max(float(wv @ wv), 1e-30)
    return to_bf16_bits(hidden), weight


def layer_weights(d: int, Hq: int, Hkv: int, D: int, d_ff: int, seed: int = 0) -> dict:
    """One LLaMA-style layer's weights as bf16 bit patterns, at the usual initialisation scale
    (activations stay about unit size): wq [Hq D, d], wk, wv [Hkv D, d], wo [d, Hq D] and wg, wu
    [d_ff, d] ~ N(0, 1 / fan_in); wd [d, d_ff] ~ N(0, 1 / d_ff); gamma1, gamma2 [d] ~ 1 + N(0,
    0.1^2). Drawn in float32 chunks of rows."""
    r = rng_for(seed, 60)

    def mat(rows: int, cols: int) -> np.ndarray:
        out = np.empty((rows, cols), dtype=np.uint16)
        for a in range(0, rows, 2048):
            b = min(rows, a + 2048)
            out[a:b] = to_bf16_bits(r.standard_normal((b - a, cols), dtype=np.float32) / np.float32(np.sqrt(cols)))
        return out

    return {
        "wq": mat(Hq * D, d), "wk": mat(Hkv * D, d), "wv": mat(Hkv * D, d), "wo": mat(d, Hq * D),
        "wg": mat(d_ff, d), "wu": mat(d_ff, d), "wd": mat(d, d_ff),
        "gamma1": to_bf16_bits(1.0 + 0.1 * r.standard_normal(d, dtype=np.float32)),
        "gamma2": to_bf16_bits(1.0 + 0.1 * r.standard_normal(d, dtype=np.float32)),
    }


def layer_input(B: int, L: int, d: int, seed: int = 0) -> np.ndarray:
    """The layer input at every position, bf16 bits [B, L, d] ~ N(0, 1)."""
    return _normal_bf16(rng_for(seed, 61), (B, L, d))
