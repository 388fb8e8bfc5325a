"""Float64 CPU oracle for one EntropyCache denoising step.

TEST INFRASTRUCTURE ONLY. This module is the slow, plain reference that the CUDA library
is checked against. Only the test suite, the smoke check and the CPU-baseline leg of the
benchmark may import it; the product path (the C-ABI library and its Python binding) never
does, and there is no fallback from the product path to this code.

It shares no code with the CUDA path: no kernels, headers, helpers or tables. Inputs arrive
as NumPy arrays in their stored form (bf16 as uint16 bit patterns, fp32, int32) and are
widened exactly to float64 here.

Source of the method: "EntropyCache: Decoded Token Entropy Guided KV Caching for Diffusion
Language Models" (Cheong, Son, Lim, Yoo), in the two gist.science summaries of it:
  [zh] gist.science/zh/paper/2603.18489, §2.2 "EntropyCache Workflow" (the three stages of
       a denoising step and the max-entropy equation), §2.3 (O(V) compute, O(k) memory);
  [pt] gist.science/pt/paper/2603.18489, §1 "O Problema" (bidirectional attention), §2
       "Metodologia" / "Fluxo de Funcionamento" (decode, skip-or-recompute, history).

Readings where the pages are silent (each also listed in the design notes):
  - entropy uses the natural logarithm; softmax temperature is 1;
  - "decode" is greedy argmax, ties to the lowest vocabulary index;
  - the tokens decoded in a step (the set D) are the n_dec candidates with the highest
    confidence p(argmax), ties to the lower position; a NaN confidence ranks lowest;
    optionally (a confidence-threshold commit, one of the decoding strategies the gate carries
    over to: [pt] §5, [zh] §5) only those with p >= conf_threshold, at least one;
  - an empty D gives E = 0 (partial); a NaN E gives a full step; E == tau is partial;
  - the history pushes D in ascending position order and survives full steps;
  - attention is unmasked (bidirectional) with scale 1/sqrt(D) by default, query head h
    reading key/value head h // (Hq // Hkv).

Every function here is pinned by tests that do not re-derive it (closed forms, invariants,
brute force over tiny inputs, and a library attention routine); see tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "widen",
    "entropy_decode_row",
    "entropy_decode",
    "lm_head_entropy",
    "select_decoded",
    "max_entropy",
    "recompute_flag",
    "history_push",
    "history_last",
    "recompute_set",
    "block_candidates",
    "sliding_window_candidates",
    "kv_scatter",
    "attention",
    "rms_norm",
    "rope",
    "swiglu",
    "layer_forward",
    "step",
]


# --------------------------------------------------------------------------------------
# stored dtypes -> float64


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of stored elements: dtype 'bf16' (uint16 bit patterns) or 'f32'."""
    if dtype == "bf16":
        bits = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------------------
# (a) decode + entropy  —  [zh] §2.2, decode new tokens and E = max_i (-sum_j p_ij log p_ij)


def entropy_decode_row(x: np.ndarray) -> tuple[int, float, float]:
    """Greedy decode, Shannon entropy and log-confidence of one row of logits.

    Follows the definition directly ([zh] §2.2, the bracketed term of the max-entropy
    equation): p = softmax(x), H = -sum_j p_j ln p_j with 0 ln 0 = 0, the decoded token is
    the lowest index attaining max x, and log_conf = ln p of that token.
    """
    x = np.asarray(x, dtype=np.float64)
    m = x.max()
    ident = int(np.flatnonzero(x == m)[0])  # lowest index attaining the maximum
    e = np.exp(x - m)  # exp(-inf) = 0
    p = e / e.sum()
    nz = p > 0.0
    h = float(-np.sum(p[nz] * np.log(p[nz])))
    log_conf = float(np.log(p[ident]))
    return ident, h, log_conf


def entropy_decode(logits: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Row-wise entropy_decode_row over a [n_rows, V] float64 array."""
    logits = np.asarray(logits, dtype=np.float64)
    n = logits.shape[0]
    ids = np.zeros(n, dtype=np.int64)
    ent = np.zeros(n, dtype=np.float64)
    conf = np.zeros(n, dtype=np.float64)
    for i in range(n):
        ids[i], ent[i], conf[i] = entropy_decode_row(logits[i])
    return ids, ent, conf


def lm_head_entropy(hidden: np.ndarray, weight: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Stage (a) on logits produced from the candidates' hidden states.

    logits = hidden @ weight.T (hidden [n_rows, d_model], weight [V, d_model], float64), then
    entropy_decode of those logits ([zh] §2.2). The pages leave the product to the model (its
    output projection); the library computes it fused with the decode, and this is the plain
    composition it must match.
    """
    logits = np.asarray(hidden, dtype=np.float64) @ np.asarray(weight, dtype=np.float64).T
    return entropy_decode(logits)


# --------------------------------------------------------------------------------------
# (b) the decoded set and the max-entropy gate  —  [zh] §2.2, [pt] §2 "Decisão de Pulo"


def select_decoded(cand_pos: np.ndarray, count: int, log_conf: np.ndarray, n_dec: int,
                   conf_threshold: float = 0.0) -> list[int]:
    """Candidate rows committed this step: the n_dec most confident among the first `count`.

    Ranking key: higher log_conf first (NaN ranks lowest), then the smaller position.
    With conf_threshold > 0 (a confidence-threshold commit, a decoding variant) only those of
    them whose confidence p = exp(log_conf) is at least the threshold are committed, and the
    single most confident one when none is. Returns candidate row numbers sorted by ascending
    position.
    """

    def eff(i: int) -> float:
        c = float(log_conf[i])
        return -math.inf if math.isnan(c) else c

    order = sorted(range(int(count)), key=lambda i: (-eff(i), int(cand_pos[i])))
    chosen = order[: int(n_dec)]
    if conf_threshold > 0.0 and chosen:
        lt = math.log(conf_threshold)
        above = [i for i in chosen if eff(i) >= lt]
        chosen = above if above else chosen[:1]
    return sorted(chosen, key=lambda i: int(cand_pos[i]))


def max_entropy(entropy: np.ndarray, decoded_rows: list[int]) -> float:
    """E_{t+1} = max over the newly decoded tokens of their entropy ([zh] §2.2).

    0 for an empty set; NaN if any entropy in the set is NaN.
    """
    if not decoded_rows:
        return 0.0
    vals = [float(entropy[i]) for i in decoded_rows]
    if any(math.isnan(v) for v in vals):
        return math.nan
    return max(vals)


def recompute_flag(E: float, tau: float) -> bool:
    """Full recompute iff E > tau ([zh] §2.2; [pt] §2): E == tau reuses the cache; NaN is full."""
    E = float(E)
    if math.isnan(E):
        return True
    return bool(E > float(tau))


# --------------------------------------------------------------------------------------
# (c) decode history and recompute set  —  [zh] §2.2 / §2.3, [pt] §2 "Histórico"


def history_push(ring: np.ndarray, head: int, count: int, positions: list[int]) -> tuple[np.ndarray, int, int]:
    """Append positions (in the given order) to a FIFO of capacity k = len(ring).

    Slot `head` receives the next entry; the count saturates at k ([zh] §2.3: O(k) memory).
    """
    ring = np.array(ring, dtype=np.int64, copy=True)
    k = ring.shape[0]
    for p in positions:
        ring[head] = p
        head = (head + 1) % k
        count = min(count + 1, k)
    return ring, head, count


def history_last(ring: np.ndarray, head: int, count: int) -> list[int]:
    """The last min(k, count) pushed positions, most recent first."""
    k = len(ring)
    n = min(int(count), k)
    return [int(ring[(head - 1 - t) % k]) for t in range(n)]


def recompute_set(mask: np.ndarray, recent: list[int], full: bool,
                  scope: tuple[int, int] | None = None) -> np.ndarray:
    """Recompute set of one sequence, ascending ([zh] §2.2 partial forward; [pt] §2).

    Full step: every position. Partial step: still-masked positions union the k most recently
    decoded positions.

    With a scope (lo, hi) — block-by-block decoding, where the gate is a recompute signal for
    the block being decoded ([zh] §5, sub-block recompute in block diffusion) — every position
    considered is restricted to [lo, hi): a full step recomputes the block, a partial one the
    block's masked positions and the recent positions that lie in the block.
    """
    L = mask.shape[0]
    lo, hi = (0, L) if scope is None else (int(scope[0]), int(scope[1]))
    if full:
        return np.arange(lo, hi, dtype=np.int64)
    chosen = set(int(p) for p in np.flatnonzero(mask) if lo <= p < hi)
    chosen.update(int(p) for p in recent if lo <= p < hi)
    return np.array(sorted(chosen), dtype=np.int64)


# --------------------------------------------------------------------------------------
# decoding schedules the gate carries over to  —  [pt] §5 "Generalidade", [zh] §5


def block_candidates(mask: np.ndarray, start: int, width: int) -> list[int]:
    """Candidates of a block-decoding step: the masked positions of the block
    [start, start + width), ascending (clipped to the sequence)."""
    L = mask.shape[0]
    return [p for p in range(int(start), min(L, int(start) + int(width))) if mask[p]]


def sliding_window_candidates(mask: np.ndarray, start: int, width: int) -> list[int]:
    """Candidates of a sliding-window decoding step: the window begins at the first masked
    position at or after `start` and spans `width` positions; its masked positions,
    ascending. The window slides forward as its earliest position gets decoded."""
    L = mask.shape[0]
    f = next((p for p in range(int(start), L) if mask[p]), L)
    return [p for p in range(f, min(L, f + int(width))) if mask[p]]


def kv_scatter(cache: np.ndarray, idx: np.ndarray, fresh_rows: np.ndarray) -> np.ndarray:
    """Cache after refreshing the recompute rows: cache[idx[r]] = fresh_rows[r]."""
    out = np.array(cache, copy=True)
    for r, pos in enumerate(idx):
        out[int(pos)] = fresh_rows[r]
    return out


# --------------------------------------------------------------------------------------
# (d) bidirectional attention  —  [pt] §1 "Atenção Bidirecional"; [zh] §1


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Unmasked softmax attention of query rows against every key row, in float64.

    q [R, Hq, D], k and v [L, Hkv, D]; query head h reads key/value head h // (Hq // Hkv).
    out[r, h] = sum_j softmax_j(scale * q[r, h] . k[j, h//g]) v[j, h//g], two-pass softmax
    (row max subtracted, exponentials, normalisation).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    R, Hq, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    out = np.zeros((R, Hq, D), dtype=np.float64)
    for h in range(Hq):
        kv = h // g
        s = (q[:, h, :] @ k[:, kv, :].T) * scale  # [R, L]
        s = s - s.max(axis=1, keepdims=True)
        w = np.exp(s)
        w = w / w.sum(axis=1, keepdims=True)
        out[:, h, :] = w @ v[:, kv, :]
    return out


# --------------------------------------------------------------------------------------
# the partial forward of one transformer layer  —  [zh] §2.2 "前向传播 / 部分传播": only the
# recompute set is recomputed, every other position is read from the K/V cache. The layer is
# the LLaMA-style block of the evaluated models (RMSNorm, rotary position embedding,
# grouped-query attention, SwiGLU feed-forward); the pages name the models, not their layers,
# so this is the plainest reading of "a forward pass" of them.


def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """Root-mean-square normalisation over the last axis, then a per-feature gain:
    x / sqrt(mean(x^2) + eps) * gamma."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(gamma, dtype=np.float64)


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary position embedding of x [R, H, D] at positions pos [R], rotate-half pairing:
    feature i and i + D/2 form a pair rotated by the angle pos * theta^(-2i/D), i < D/2."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    inv = np.asarray(theta, dtype=np.float64) ** (-2.0 * np.arange(h, dtype=np.float64) / D)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]  # [R, D/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """SiLU(g) * u with SiLU(g) = g / (1 + exp(-g))."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g)) * np.asarray(u, dtype=np.float64)


def layer_forward(*, x_src: np.ndarray, idx: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                  weights: dict, Hq: int, Hkv: int, theta: float, eps: float,
                  rows: np.ndarray | None = None) -> dict:
    """Partial forward of one layer for the recompute rows idx of one sequence, in float64.

    x_src [L, d]: the layer input at every position; k_cache, v_cache [L, Hkv, D]; weights:
    wq [Hq D, d], wk, wv [Hkv D, d], wo [d, Hq D], wg, wu [d_ff, d], wd [d, d_ff], gamma1,
    gamma2 [d]. For every recompute row r (position idx[r]):
      x = x_src[idx], h = rms_norm(x, gamma1)
      q, k, v = h wq^T, h wk^T, h wv^T; q, k rotated at their positions (rope)
      the cache rows at idx take k and v (the K/V refresh of the recompute set)
      o = attention of q against the whole refreshed cache (unmasked, scale 1/sqrt(D))
      x2 = x + o wo^T;  y = x2 + swiglu(h2 wg^T, h2 wu^T) wd^T with h2 = rms_norm(x2, gamma2)
    rows: compute o, x2 and y for these recompute rows only (a sample); q, k, v and the caches
    are always complete.
    """
    W = {n: np.asarray(a, dtype=np.float64) for n, a in weights.items()}
    idx = np.asarray(idx, dtype=np.int64)
    R = idx.shape[0]
    D = k_cache.shape[-1]
    x = np.asarray(x_src, dtype=np.float64)[idx]
    h = rms_norm(x, W["gamma1"], eps)
    q = rope((h @ W["wq"].T).reshape(R, Hq, D), idx, theta)
    k = rope((h @ W["wk"].T).reshape(R, Hkv, D), idx, theta)
    v = (h @ W["wv"].T).reshape(R, Hkv, D)
    kc = kv_scatter(np.asarray(k_cache, dtype=np.float64), idx, k)
    vc = kv_scatter(np.asarray(v_cache, dtype=np.float64), idx, v)
    sel = np.arange(R) if rows is None else np.asarray(rows, dtype=np.int64)
    o = attention(q[sel], kc, vc, 1.0 / math.sqrt(D))
    x2 = x[sel] + o.reshape(len(sel), Hq * D) @ W["wo"].T
    h2 = rms_norm(x2, W["gamma2"], eps)
    y = x2 + swiglu(h2 @ W["wg"].T, h2 @ W["wu"].T) @ W["wd"].T
    return {"q": q, "k": k, "v": v, "k_cache": kc, "v_cache": vc, "o": o, "x2": x2, "y": y, "rows": sel}


# --------------------------------------------------------------------------------------
# one whole step  —  [zh] §2.2, the three stages in order


def step(
    *,
    logits: np.ndarray,
    cand_pos: np.ndarray,
    cand_count: int,
    tokens: np.ndarray,
    mask: np.ndarray,
    ring: np.ndarray,
    ring_head: int,
    ring_count: int,
    n_dec: int,
    tau: float,
    conf_threshold: float = 0.0,
    layers: list[dict] | None = None,
    scale: float | None = None,
    attention_rows: np.ndarray | None = None,
    decoded_rows: list[int] | None = None,
    scope: tuple[int, int] | None = None,
) -> dict:
    """One denoising step of one sequence.

    logits [C_max, V] float64 (candidate rows); tokens [L]; mask [L] (1 = masked);
    ring [k] with head/count. Each element of `layers` is a dict of float64 arrays
    k_cache, v_cache [L, Hkv, D], k_src, v_src [L, Hkv, D] (fresh rows by position) and
    q_src [L, Hq, D] (queries by position). attention_rows optionally restricts which
    recompute rows get an attention output (a sample); None computes all of them.
    decoded_rows optionally fixes the committed candidate rows instead of ranking them: a
    checker that finds two candidates' confidences tied within rounding adopts the device's
    choice among them this way, then checks everything that follows from it.
    scope (lo, hi), for block-by-block decoding: the recompute set is restricted to the block
    (recompute_set) and the recomputed rows attend to the keys [0, hi) only: the block and the
    blocks before it, none after it (block-causal attention).
    Returns decode results, the gate, the new state, idx and per-layer outputs.
    """
    C = int(cand_count)
    ids, ent, conf = entropy_decode(logits[:C]) if C > 0 else (
        np.zeros(0, np.int64), np.zeros(0), np.zeros(0))
    if decoded_rows is None:
        rows = select_decoded(cand_pos, C, conf, n_dec, conf_threshold)
    else:
        rows = sorted((int(i) for i in decoded_rows), key=lambda i: int(cand_pos[i]))
    tokens = np.array(tokens, dtype=np.int64, copy=True)
    mask = np.array(mask, dtype=np.uint8, copy=True)
    for i in rows:
        tokens[int(cand_pos[i])] = ids[i]
        mask[int(cand_pos[i])] = 0
    E = max_entropy(ent, rows)
    full = recompute_flag(E, tau)
    dec_positions = [int(cand_pos[i]) for i in rows]
    ring2, head2, count2 = history_push(ring, ring_head, ring_count, dec_positions)
    idx = recompute_set(mask, history_last(ring2, head2, count2), full, scope)
    hi = mask.shape[0] if scope is None else int(scope[1])
    out_layers = []
    for lay in layers or []:
        kc = kv_scatter(lay["k_cache"], idx, lay["k_src"][idx])
        vc = kv_scatter(lay["v_cache"], idx, lay["v_src"][idx])
        D = kc.shape[-1]
        sc = (1.0 / math.sqrt(D)) if scale is None else scale
        sel = idx if attention_rows is None else idx[attention_rows]
        o = attention(lay["q_src"][sel], kc[:hi], vc[:hi], sc)
        out_layers.append({"k_cache": kc, "v_cache": vc, "out": o})
    return {
        "ids": ids,
        "entropy": ent,
        "log_conf": conf,
        "decoded_rows": rows,
        "dec_pos": dec_positions,
        "E": E,
        "flag": bool(full),
        "tokens": tokens,
        "mask": mask,
        "ring": ring2,
        "ring_head": head2,
        "ring_count": count2,
        "idx": idx,
        "R": int(idx.shape[0]),
        "layers": out_layers,
    }
