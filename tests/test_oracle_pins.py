"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each test checks the oracle against a closed form, an invariant, a library routine computing
the same quantity, or brute force over tiny inputs, chosen so that a plausible slip (a wrong
log base, a dropped minus sign, a missing normalisation, a wrong tie rule, a transposed
operand, an off-by-one in the history) fails at least one of them.

Facts used (EntropyCache, gist.science zh summary §2.2 and pt summary §2):
  - E_{t+1} = max over the newly decoded tokens of -sum_j p_ij log p_ij;
  - E > tau triggers a full recompute, E <= tau reuses the cache except masked + last k;
  - with every position recomputed the attention is plain dense bidirectional attention.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --------------------------------------------------------------------------------------
# entropy / decode


@pytest.mark.parametrize("V", [1, 2, 7, 32000, 126464, 152064])
@pytest.mark.parametrize("c", [0.0, -3.5, 17.25])
def test_uniform_logits_give_ln_V(V, c):
    ident, h, lc = O.entropy_decode_row(np.full(V, c))
    assert abs(h - math.log(V)) <= 1e-12 * max(1.0, math.log(V)) + 1e-12
    assert abs(lc + math.log(V)) <= 1e-12 * max(1.0, math.log(V)) + 1e-12
    assert ident == 0  # a V-way tie decodes to the lowest index


@pytest.mark.parametrize("hot", [0, 5, 99])
def test_one_hot_gives_zero(hot):
    x = np.full(100, -np.inf)
    x[hot] = 3.0
    ident, h, lc = O.entropy_decode_row(x)
    assert ident == hot and h == 0.0 and lc == 0.0
    y = np.zeros(100)
    y[hot] = 1e4  # the others underflow to zero probability
    ident, h, lc = O.entropy_decode_row(y)
    assert ident == hot and abs(h) < 1e-300 and abs(lc) < 1e-300


@pytest.mark.parametrize("kk", [2, 3, 8, 64])
def test_k_way_tie_gives_ln_k_and_lowest_index(kk):
    rng = np.random.default_rng(kk)
    x = np.full(500, -np.inf)
    pos = np.sort(rng.choice(500, size=kk, replace=False))
    x[pos] = 1.5
    ident, h, lc = O.entropy_decode_row(x)
    assert ident == pos[0]
    assert abs(h - math.log(kk)) < 1e-13
    assert abs(lc + math.log(kk)) < 1e-13


@pytest.mark.parametrize("a,b", [(0.0, 0.0), (1.0, 0.0), (0.0, 2.5), (-3.0, 4.0), (10.0, -10.0)])
def test_two_logits_give_binary_entropy(a, b):
    # softmax of two logits is the logistic sigma(a - b); its entropy is the binary entropy
    p = 1.0 / (1.0 + math.exp(-(a - b)))
    hb = -sum(t * math.log(t) for t in (p, 1 - p) if t > 0)
    ident, h, lc = O.entropy_decode_row(np.array([a, b]))
    assert abs(h - hb) < 1e-12
    assert ident == (0 if a >= b else 1)
    assert abs(lc - math.log(max(p, 1 - p))) < 1e-12


def test_matches_scipy_entropy_of_softmax():
    rng = np.random.default_rng(7)
    for s in (0.1, 1.0, 4.0, 12.0):
        x = rng.standard_normal(3001) * s
        ident, h, lc = O.entropy_decode_row(x)
        p = scipy.special.softmax(x)
        assert abs(h - scipy.stats.entropy(p)) < 1e-10
        assert ident == int(np.argmax(x))
        assert abs(lc - math.log(p.max())) < 1e-10


def test_shift_and_permutation_invariance():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(777) * 3
    ident, h, lc = O.entropy_decode_row(x)
    i2, h2, lc2 = O.entropy_decode_row(x + 123.456)
    assert i2 == ident and abs(h2 - h) < 1e-11 and abs(lc2 - lc) < 1e-11
    perm = rng.permutation(777)
    i3, h3, lc3 = O.entropy_decode_row(x[perm])
    assert perm[i3] == ident and abs(h3 - h) < 1e-11 and abs(lc3 - lc) < 1e-11


def test_entropy_bounds_and_neg_inf_entries():
    rng = np.random.default_rng(3)
    for V in (2, 10, 1000):
        x = rng.standard_normal(V) * 5
        _, h, lc = O.entropy_decode_row(x)
        assert -1e-12 <= h <= math.log(V) + 1e-12
        assert lc <= 0
        # -inf entries carry zero probability and do not change the entropy of the rest
        y = np.concatenate([x, np.full(13, -np.inf)])
        _, h2, lc2 = O.entropy_decode_row(y)
        assert abs(h2 - h) < 1e-12 and abs(lc2 - lc) < 1e-12


def test_widen_is_exact():
    vals = np.array([0.0, 1.0, -2.5, 3.140625, 1e-20, -65280.0], dtype=np.float32)
    bits = W.to_bf16_bits(vals)
    back = O.widen(bits, "bf16")
    assert back.dtype == np.float64
    np.testing.assert_array_equal(back, np.array([0.0, 1.0, -2.5, 3.140625, back[4], -65280.0]))
    assert abs(back[4] - 1e-20) / 1e-20 < 2 ** -8
    np.testing.assert_array_equal(O.widen(vals, "f32"), vals.astype(np.float64))


# --------------------------------------------------------------------------------------
# decoded set, max-entropy gate


def _brute_decoded(cand_pos, count, conf, n_dec):
    """The unique subset S of size min(n_dec, count) whose members all outrank every
    non-member (higher confidence; equal confidence: smaller position; NaN lowest)."""
    def better(i, j):
        ci = -math.inf if math.isnan(conf[i]) else conf[i]
        cj = -math.inf if math.isnan(conf[j]) else conf[j]
        return ci > cj or (ci == cj and cand_pos[i] < cand_pos[j])

    n = min(n_dec, count)
    found = []
    for S in itertools.combinations(range(count), n):
        rest = [j for j in range(count) if j not in S]
        if all(better(i, j) for i in S for j in rest):
            found.append(sorted(S, key=lambda i: cand_pos[i]))
    assert len(found) == 1
    return found[0]


def test_select_decoded_brute_force():
    rng = np.random.default_rng(5)
    for trial in range(400):
        C = int(rng.integers(1, 8))
        count = int(rng.integers(0, C + 1))
        n_dec = int(rng.integers(1, C + 1))
        cand_pos = rng.choice(40, size=C, replace=False)
        conf = -rng.integers(0, 3, size=C).astype(np.float64)  # many exact ties
        if trial % 7 == 0 and C > 1:
            conf[rng.integers(0, C)] = np.nan
        got = O.select_decoded(cand_pos, count, conf, n_dec)
        assert got == _brute_decoded(cand_pos, count, conf, n_dec)


def test_max_entropy_and_flag_boundaries():
    ent = np.array([0.3, 1.0, 2.5, np.nan])
    assert O.max_entropy(ent, []) == 0.0
    assert O.max_entropy(ent, [0, 1]) == 1.0
    assert O.max_entropy(ent, [0, 2, 1]) == 2.5
    assert math.isnan(O.max_entropy(ent, [0, 3]))
    tau = 1.0
    assert O.recompute_flag(1.0, tau) is False  # E == tau reuses the cache
    assert O.recompute_flag(np.nextafter(1.0, 2.0), tau) is True
    assert O.recompute_flag(np.nextafter(1.0, 0.0), tau) is False
    assert O.recompute_flag(math.nan, tau) is True
    assert O.recompute_flag(0.0, tau) is False


# --------------------------------------------------------------------------------------
# history and recompute set


def test_history_matches_unbounded_list():
    rng = np.random.default_rng(9)
    for k in (1, 2, 5, 16):
        ring = np.zeros(k, dtype=np.int64)
        head = count = 0
        full: list[int] = []
        for _ in range(60):
            push = [int(v) for v in rng.integers(0, 1000, size=int(rng.integers(0, 4)))]
            ring, head, count = O.history_push(ring, head, count, push)
            full.extend(push)
            assert count == min(len(full), k)
            assert O.history_last(ring, head, count) == list(reversed(full))[:k]


def test_recompute_set_exhaustive_small():
    rng = np.random.default_rng(13)
    for L in range(1, 11):
        for bits in range(1 << L):
            mask = np.array([(bits >> p) & 1 for p in range(L)], dtype=np.uint8)
            recent = [int(v) for v in rng.choice(L, size=int(rng.integers(0, L + 1)), replace=False)]
            got = O.recompute_set(mask, recent, full=False)
            want = [p for p in range(L) if mask[p] == 1 or p in recent]
            assert got.tolist() == want
            assert O.recompute_set(mask, recent, full=True).tolist() == list(range(L))


# --------------------------------------------------------------------------------------
# attention


def _sdpa(q, k, v, scale):
    """torch's scaled_dot_product_attention in float64, GQA by repeating kv heads."""
    R, Hq, D = q.shape
    g = Hq // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("R,L,Hq,Hkv,D", [(5, 17, 2, 2, 8), (16, 16, 4, 1, 16), (3, 40, 6, 2, 64), (1, 1, 1, 1, 4)])
def test_attention_matches_library_sdpa(R, L, Hq, Hkv, D):
    rng = np.random.default_rng(R * 1000 + L)
    q = rng.standard_normal((R, Hq, D))
    k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    scale = 1.0 / math.sqrt(D)
    np.testing.assert_allclose(O.attention(q, k, v, scale), _sdpa(q, k, v, scale), rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(21)
    L, D = 9, 5
    v = rng.standard_normal((L, 1, D))
    q = rng.standard_normal((3, 1, D))
    # all keys equal: uniform weights, output is the mean of the value rows
    k = np.tile(rng.standard_normal((1, 1, D)), (L, 1, 1))
    np.testing.assert_allclose(O.attention(q, k, v, 0.7), np.broadcast_to(v.mean(axis=0), (3, 1, D)), atol=1e-13)
    # one key with a +50 score gap: output is that key's value row
    k = np.zeros((L, 1, D))
    k[4, 0, 0] = 50.0
    qq = np.zeros((1, 1, D))
    qq[0, 0, 0] = 1.0
    np.testing.assert_allclose(O.attention(qq, k, v, 1.0)[0, 0], v[4, 0], atol=1e-18 + 1e-20)
    # D = 1, L = 2 by hand
    q1 = np.array([[[2.0]]])
    k1 = np.array([[[1.0]], [[-0.5]]])
    v1 = np.array([[[3.0]], [[7.0]]])
    s0, s1 = 2.0 * 1.0 * 0.5, 2.0 * -0.5 * 0.5
    want = (math.exp(s0) * 3.0 + math.exp(s1) * 7.0) / (math.exp(s0) + math.exp(s1))
    assert abs(O.attention(q1, k1, v1, 0.5)[0, 0, 0] - want) < 1e-14


def test_attention_key_permutation_invariance():
    rng = np.random.default_rng(22)
    q = rng.standard_normal((4, 2, 8))
    k = rng.standard_normal((30, 1, 8))
    v = rng.standard_normal((30, 1, 8))
    perm = rng.permutation(30)
    np.testing.assert_allclose(O.attention(q, k, v, 0.35), O.attention(q, k[perm], v[perm], 0.35), atol=1e-13)


# --------------------------------------------------------------------------------------
# whole step, brute force on L <= 16


def _brute_step(logits, cand_pos, count, tokens, mask, decoded_history, n_dec, tau, k):
    """List-based restatement of one step: decode all candidates, commit the n_dec most
    confident, gate on their maximum entropy, recompute masked + last k decoded."""
    info = []
    for i in range(count):
        x = [float(t) for t in logits[i]]
        m = max(x)
        ident = x.index(m)
        z = sum(math.exp(t - m) for t in x)
        ps = [math.exp(t - m) / z for t in x]
        h = -sum(p * math.log(p) for p in ps if p > 0)
        info.append((math.log(ps[ident]), int(cand_pos[i]), ident, h))
    ranked = sorted(info, key=lambda t: (-t[0], t[1]))[:n_dec]
    tokens = list(tokens)
    mask = list(mask)
    for _, pos, ident, _ in ranked:
        tokens[pos] = ident
        mask[pos] = 0
    E = max((t[3] for t in ranked), default=0.0)
    full = E > tau
    hist = list(decoded_history) + sorted(t[1] for t in ranked)
    recent = set(hist[-k:]) if k > 0 else set()
    L = len(mask)
    idx = list(range(L)) if full else [p for p in range(L) if mask[p] or p in recent]
    return tokens, mask, E, full, idx, hist


def test_step_brute_force_tiny():
    rng = np.random.default_rng(31)
    for trial in range(300):
        L = int(rng.integers(2, 17))
        k = int(rng.integers(1, L + 1))
        Vv = int(rng.integers(2, 9))
        mask = (rng.random(L) < 0.5).astype(np.uint8)
        masked = np.flatnonzero(mask)
        if masked.size == 0:
            mask[0] = 1
            masked = np.array([0])
        C = int(masked.size)
        cand_pos = masked.astype(np.int64)
        count = int(rng.integers(0, C + 1))
        n_dec = int(rng.integers(1, C + 1))
        scale = rng.choice([0.05, 1.0, 6.0])
        logits = rng.standard_normal((C, Vv)) * scale
        if trial % 5 == 0:
            logits = np.round(logits)  # exact ties in the argmax and in the confidence
        tokens = rng.integers(0, Vv, size=L)
        decoded = [p for p in range(L) if not mask[p]]
        rng.shuffle(decoded)
        ring = np.zeros(k, dtype=np.int64)
        ring, head, cnt = O.history_push(ring, 0, 0, decoded)
        tau = float(rng.choice([0.0, 0.3, 1.0, 5.0]))
        got = O.step(logits=logits, cand_pos=cand_pos, cand_count=count, tokens=tokens, mask=mask,
                     ring=ring, ring_head=head, ring_count=cnt, n_dec=n_dec, tau=tau)
        t2, m2, E2, f2, idx2, hist2 = _brute_step(logits, cand_pos, count, tokens, mask, decoded, n_dec, tau, k)
        assert got["tokens"].tolist() == t2
        assert got["mask"].tolist() == m2
        assert abs(got["E"] - E2) < 1e-12
        assert got["flag"] == f2
        assert got["idx"].tolist() == idx2
        assert got["R"] == len(idx2)
        assert O.history_last(got["ring"], got["ring_head"], got["ring_count"]) == list(reversed(hist2))[:k]


def test_step_full_flag_attention_is_dense_attention():
    rng = np.random.default_rng(41)
    L, Hq, Hkv, D, Vv = 12, 4, 2, 8, 50
    mask = np.zeros(L, dtype=np.uint8)
    mask[8:] = 1
    logits = rng.standard_normal((4, Vv)) * 0.1  # near-uniform: high entropy, full step
    lay = {
        "k_cache": rng.standard_normal((L, Hkv, D)),
        "v_cache": rng.standard_normal((L, Hkv, D)),
        "k_src": rng.standard_normal((L, Hkv, D)),
        "v_src": rng.standard_normal((L, Hkv, D)),
        "q_src": rng.standard_normal((L, Hq, D)),
    }
    got = O.step(logits=logits, cand_pos=np.arange(8, 12), cand_count=4, tokens=np.zeros(L, np.int64),
                 mask=mask, ring=np.zeros(4, np.int64), ring_head=0, ring_count=0, n_dec=1, tau=1.0,
                 layers=[lay])
    assert got["flag"] and got["R"] == L
    out = got["layers"][0]["out"]
    dense = _sdpa(lay["q_src"], lay["k_src"], lay["v_src"], 1.0 / math.sqrt(D))
    np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-12)


# ---- (a) from hidden states: logits = hidden @ weight.T, then the decode -----------------


def test_lm_head_entropy_closed_forms_and_orientation():
    # hidden = identity rows, so logits row r is column r of weight: the rows below are logs
    # of small integers with closed-form entropies (softmax = the integers over their sum).
    # weight is not symmetric, so a transposed product would give other entropies.
    rows = [[1, 1, 1, 1], [1, 1, 2, 4], [12, 2, 1, 1], [1, 1, 1, 5]]
    logits = np.log(np.array(rows, dtype=np.float64))
    weight = logits.T.copy()  # [V = 4, d_model = 4]
    hidden = np.eye(4)
    ids, ent, conf = O.lm_head_entropy(hidden, weight)
    ln2, ln3, ln5 = math.log(2), math.log(3), math.log(5)
    np.testing.assert_array_equal(ids, [0, 3, 0, 3])
    np.testing.assert_allclose(ent, [2 * ln2, 1.75 * ln2, 19 / 8 * ln2 - 0.75 * ln3, 3 * ln2 - 5 / 8 * ln5],
                               rtol=1e-13)
    np.testing.assert_allclose(conf, [-2 * ln2, -ln2, ln3 - 2 * ln2, ln5 - 3 * ln2], rtol=1e-13)


def test_lm_head_entropy_brute_force_dot_products():
    rng = np.random.default_rng(7)
    for n, d, V in [(1, 1, 1), (3, 5, 7), (4, 16, 33)]:
        h = rng.standard_normal((n, d))
        w = rng.standard_normal((V, d))
        logits = [[sum(h[r, k] * w[v, k] for k in range(d)) for v in range(V)] for r in range(n)]
        want = O.entropy_decode(np.array(logits))
        got = O.lm_head_entropy(h, w)
        np.testing.assert_array_equal(got[0], want[0])
        np.testing.assert_allclose(got[1], want[1], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(got[2], want[2], rtol=1e-12, atol=1e-14)


def test_confidence_threshold_commit_by_hand():
    # confidences .9, .6, .3, .8 at positions 10..13, n_dec = 3: the three most confident are
    # rows 0 (.9), 3 (.8), 1 (.6)
    pos = np.array([10, 11, 12, 13])
    lc = np.log(np.array([0.9, 0.6, 0.3, 0.8]))
    assert O.select_decoded(pos, 4, lc, 3) == [0, 1, 3]
    assert O.select_decoded(pos, 4, lc, 3, conf_threshold=0.7) == [0, 3]  # .9 and .8 pass
    assert O.select_decoded(pos, 4, lc, 3, conf_threshold=0.6) == [0, 1, 3]  # >= includes .6
    assert O.select_decoded(pos, 4, lc, 3, conf_threshold=0.95) == [0]  # none: the best one
    assert O.select_decoded(pos, 4, lc, 1, conf_threshold=0.5) == [0]  # n_dec still caps
    assert O.select_decoded(pos, 0, lc, 3, conf_threshold=0.5) == []  # nothing to commit
    # NaN confidence never passes and ranks last
    lc2 = np.array([math.nan, math.log(0.8), math.log(0.2)])
    assert O.select_decoded(pos[:3], 3, lc2, 3, conf_threshold=0.5) == [1]


# --------------------------------------------------------------------------------------
# decoding schedules and the block-scoped gate ([pt] §5 "Generalidade", [zh] §5)


def test_scoped_recompute_set_exhaustive_small():
    # membership scan over every mask of L <= 8 and every scope [lo, hi)
    rng = np.random.default_rng(14)
    for L in range(1, 9):
        for bits in range(1 << L):
            mask = np.array([(bits >> p) & 1 for p in range(L)], dtype=np.uint8)
            recent = [int(v) for v in rng.choice(L, size=int(rng.integers(0, L + 1)), replace=False)]
            for lo in range(L):
                for hi in range(lo + 1, L + 1):
                    got = O.recompute_set(mask, recent, full=False, scope=(lo, hi)).tolist()
                    want = []
                    for p in range(L):
                        inside = lo <= p and p < hi
                        if inside and (mask[p] == 1 or p in recent):
                            want.append(p)
                    assert got == want, (L, bits, lo, hi)
                    assert O.recompute_set(mask, recent, full=True, scope=(lo, hi)).tolist() == list(range(lo, hi))
            # the whole sequence as the scope is the unscoped set
            assert (O.recompute_set(mask, recent, False, (0, L)).tolist()
                    == O.recompute_set(mask, recent, False).tolist())


def test_schedule_candidates_by_hand():
    mask = np.array([0, 0, 1, 0, 1, 1, 0, 1, 1, 0, 0, 1], dtype=np.uint8)  # masked: 2 4 5 7 8 11
    assert O.block_candidates(mask, 0, 4) == [2]
    assert O.block_candidates(mask, 4, 4) == [4, 5, 7]
    assert O.block_candidates(mask, 8, 4) == [8, 11]
    assert O.block_candidates(mask, 10, 8) == [11]  # clipped at L = 12
    assert O.block_candidates(mask, 0, 2) == []
    # sliding: the window opens at the first masked position at or after start
    assert O.sliding_window_candidates(mask, 0, 4) == [2, 4, 5]  # window 2..5
    assert O.sliding_window_candidates(mask, 3, 4) == [4, 5, 7]  # window 4..7
    assert O.sliding_window_candidates(mask, 6, 2) == [7, 8]  # window 7..8
    assert O.sliding_window_candidates(mask, 9, 5) == [11]  # window 11..15, clipped
    assert O.sliding_window_candidates(np.zeros(5, np.uint8), 0, 3) == []  # nothing masked


def test_schedule_candidates_invariants():
    rng = np.random.default_rng(15)
    for _ in range(400):
        L = int(rng.integers(1, 40))
        mask = (rng.random(L) < rng.random()).astype(np.uint8)
        W = int(rng.integers(1, 12))
        start = int(rng.integers(0, L))
        # blocks of width W tile the sequence: their candidates partition the masked positions
        tiles = [p for b0 in range(0, L, W) for p in O.block_candidates(mask, b0, W)]
        assert tiles == [int(p) for p in np.flatnonzero(mask)]
        got = O.sliding_window_candidates(mask, start, W)
        later = [int(p) for p in np.flatnonzero(mask) if p >= start]
        if not later:
            assert got == []
            continue
        assert got[0] == later[0]  # the window opens at the first masked position at or after start
        assert got == [p for p in later if p < later[0] + W]  # and takes every masked one in W


def _brute_scoped(logits, cand_pos, count, mask, decoded_history, tau, k, lo, hi):
    """List-based restatement of one block-scoped step with n_dec = 1: commit the most
    confident candidate, gate on its entropy; full: the block; partial: the block's masked
    positions and the recent positions inside the block."""
    best = None
    for i in range(count):
        x = [float(t) for t in logits[i]]
        m = max(x)
        z = sum(math.exp(t - m) for t in x)
        ps = [math.exp(t - m) / z for t in x]
        key = (-math.log(ps[x.index(m)]), int(cand_pos[i]))
        h = -sum(p * math.log(p) for p in ps if p > 0)
        if best is None or key < best[0]:
            best = (key, h)
    mask = list(mask)
    hist = list(decoded_history)
    E = 0.0
    if best is not None:
        mask[best[0][1]] = 0
        hist.append(best[0][1])
        E = best[1]
    recent = set(hist[-k:])
    if E > tau:
        return list(range(lo, hi)), E
    return [p for p in range(lo, hi) if mask[p] or p in recent], E


def test_scoped_step_brute_force_and_block_causal_attention():
    rng = np.random.default_rng(32)
    for trial in range(200):
        L = int(rng.integers(4, 17))
        lo = int(rng.integers(0, L - 1))
        hi = int(rng.integers(lo + 1, L + 1))
        k = int(rng.integers(1, L + 1))
        mask = np.zeros(L, np.uint8)
        mask[lo:] = (rng.random(L - lo) < 0.6)  # earlier blocks decoded
        cand = [p for p in range(lo, hi) if mask[p]]
        if not cand:
            mask[lo] = 1
            cand = [lo]
        logits = rng.standard_normal((len(cand), 6)) * rng.choice([0.1, 3.0])
        decoded = [p for p in range(L) if not mask[p]]
        rng.shuffle(decoded)
        ring, head, cnt = O.history_push(np.zeros(k, np.int64), 0, 0, decoded)
        tau = float(rng.choice([0.2, 1.0, 3.0]))
        got = O.step(logits=logits, cand_pos=np.array(cand), cand_count=len(cand), tokens=np.zeros(L, np.int64),
                     mask=mask, ring=ring, ring_head=head, ring_count=cnt, n_dec=1, tau=tau, scope=(lo, hi))
        idx, E = _brute_scoped(logits, cand, len(cand), mask, decoded, tau, k, lo, hi)
        assert got["idx"].tolist() == idx and abs(got["E"] - E) < 1e-12
    # attention of a block-scoped full step is dense attention over the keys [0, hi)
    L, lo, hi, Hq, Hkv, D = 16, 8, 12, 4, 2, 8
    mask = np.zeros(L, np.uint8)
    mask[lo:] = 1
    lay = {n: rng.standard_normal((L, Hkv if n != "q_src" else Hq, D))
           for n in ("k_cache", "v_cache", "k_src", "v_src", "q_src")}
    got = O.step(logits=rng.standard_normal((4, 50)) * 0.1, cand_pos=np.arange(lo, hi), cand_count=4,
                 tokens=np.zeros(L, np.int64), mask=mask, ring=np.zeros(4, np.int64), ring_head=0, ring_count=0,
                 n_dec=1, tau=1.0, layers=[lay], scope=(lo, hi))
    assert got["flag"] and got["idx"].tolist() == list(range(lo, hi))
    kc = lay["k_cache"].copy()
    vc = lay["v_cache"].copy()
    kc[lo:hi] = lay["k_src"][lo:hi]
    vc[lo:hi] = lay["v_src"][lo:hi]
    want = _sdpa(lay["q_src"][lo:hi], kc[:hi], vc[:hi], 1.0 / math.sqrt(D))
    np.testing.assert_allclose(got["layers"][0]["out"], want, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------------------
# the partial forward of one layer ([zh] §2.2 partial forward): RMSNorm, RoPE, SwiGLU, the block


def test_rms_norm_closed_forms():
    np.testing.assert_allclose(O.rms_norm(np.array([3.0, 4.0]), np.ones(2), 0.0),
                               [3.0 / math.sqrt(12.5), 4.0 / math.sqrt(12.5)], rtol=1e-15)
    c = np.full(7, -2.5)
    gamma = np.arange(1.0, 8.0)
    np.testing.assert_allclose(O.rms_norm(c, gamma, 0.0), -gamma, rtol=1e-15)  # a constant row: its sign times gamma
    rng = np.random.default_rng(51)
    x = rng.standard_normal((5, 64))
    y = O.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-14)  # unit RMS
    np.testing.assert_allclose(O.rms_norm(3.7 * x, np.ones(64), 0.0), y, rtol=1e-14)  # scale invariance
    assert abs(O.rms_norm(np.array([1e-3]), np.ones(1), 1e-6)[0] - 1e-3 / math.sqrt(1e-6 + 1e-6)) < 1e-15  # eps


def test_rope_closed_forms_and_invariants():
    # D = 2: (1, 0) at position p is (cos p, sin p); D = 4: the second pair turns by p theta^(-1/2)
    for p in (0, 1, 5, 1000):
        np.testing.assert_allclose(O.rope(np.array([[[1.0, 0.0]]]), np.array([p]), 10000.0)[0, 0],
                                   [math.cos(p), math.sin(p)], atol=1e-12)
    x = np.array([[[0.0, 2.0, 0.0, 0.0]]])  # feature 1 pairs with feature 3
    a = 7 * 100.0 ** -0.5
    np.testing.assert_allclose(O.rope(x, np.array([7]), 100.0)[0, 0], [0.0, 2 * math.cos(a), 0.0, 2 * math.sin(a)],
                               atol=1e-12)
    rng = np.random.default_rng(52)
    q = rng.standard_normal((1, 3, 16))
    k = rng.standard_normal((1, 3, 16))
    np.testing.assert_allclose(O.rope(q, np.array([0]), 500000.0), q, atol=0)  # position 0: identity
    r = O.rope(q, np.array([123]), 500000.0)
    np.testing.assert_allclose(np.linalg.norm(r[..., :8] ** 2 + r[..., 8:] ** 2),
                               np.linalg.norm(q[..., :8] ** 2 + q[..., 8:] ** 2), rtol=1e-12)  # pair norms kept
    # relative positions: <rope(q, m), rope(k, n)> depends on m - n only
    for m, n, t in ((5, 2, 40), (100, 300, 7)):
        a1 = np.sum(O.rope(q, np.array([m]), 10000.0) * O.rope(k, np.array([n]), 10000.0), axis=-1)
        a2 = np.sum(O.rope(q, np.array([m + t]), 10000.0) * O.rope(k, np.array([n + t]), 10000.0), axis=-1)
        np.testing.assert_allclose(a1, a2, rtol=1e-10, atol=1e-12)


def test_swiglu_closed_forms():
    assert O.swiglu(np.array([0.0]), np.array([5.0]))[0] == 0.0
    assert abs(O.swiglu(np.array([1.0]), np.array([2.0]))[0] - 2.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(O.swiglu(np.array([40.0]), np.array([3.0]))[0] - 120.0) < 1e-12  # SiLU(g) -> g
    assert abs(O.swiglu(np.array([-40.0]), np.array([3.0]))[0]) < 1e-15  # SiLU(g) -> 0


def _layer_weights(rng, d, Hq, Hkv, D, dff, scale=1.0):
    return {"wq": rng.standard_normal((Hq * D, d)) * scale, "wk": rng.standard_normal((Hkv * D, d)) * scale,
            "wv": rng.standard_normal((Hkv * D, d)) * scale, "wo": rng.standard_normal((d, Hq * D)) * scale,
            "wg": rng.standard_normal((dff, d)) * scale, "wu": rng.standard_normal((dff, d)) * scale,
            "wd": rng.standard_normal((d, dff)) * scale, "gamma1": 1.0 + 0.1 * rng.standard_normal(d),
            "gamma2": 1.0 + 0.1 * rng.standard_normal(d)}


def _brute_layer(x_src, idx, kc0, vc0, W, Hq, Hkv, D, theta, eps):
    """Index-by-index restatement of the layer (explicit sums over (output, input) weight
    indices), for tiny shapes."""
    L, d = len(x_src), len(x_src[0])
    dff = len(W["wg"])
    g = Hq // Hkv

    def norm(v, gam):
        ms = sum(t * t for t in v) / len(v)
        return [v[i] / math.sqrt(ms + eps) * gam[i] for i in range(len(v))]

    def mat(Wm, v):  # (W v)_j = sum_i W[j][i] v[i]
        return [sum(Wm[j][i] * v[i] for i in range(len(v))) for j in range(len(Wm))]

    def rot(vec, pos):  # one head
        h = D // 2
        out = list(vec)
        for i in range(h):
            ang = pos * theta ** (-2.0 * i / D)
            out[i] = vec[i] * math.cos(ang) - vec[i + h] * math.sin(ang)
            out[i + h] = vec[i + h] * math.cos(ang) + vec[i] * math.sin(ang)
        return out

    kc = [[list(kc0[p][j]) for j in range(Hkv)] for p in range(L)]
    vc = [[list(vc0[p][j]) for j in range(Hkv)] for p in range(L)]
    qs, hs, xs = [], [], []
    for p in idx:
        x = list(x_src[p])
        h = norm(x, W["gamma1"])
        q, k, v = mat(W["wq"], h), mat(W["wk"], h), mat(W["wv"], h)
        qs.append([rot(q[a * D:(a + 1) * D], p) for a in range(Hq)])
        kc[p] = [rot(k[a * D:(a + 1) * D], p) for a in range(Hkv)]
        vc[p] = [v[a * D:(a + 1) * D] for a in range(Hkv)]
        xs.append(x)
    ys = []
    for r, p in enumerate(idx):
        o = []
        for a in range(Hq):
            s = [sum(qs[r][a][e] * kc[j][a // g][e] for e in range(D)) / math.sqrt(D) for j in range(L)]
            m = max(s)
            w = [math.exp(t - m) for t in s]
            z = sum(w)
            o.extend(sum(w[j] / z * vc[j][a // g][e] for j in range(L)) for e in range(D))
        x2 = [xs[r][i] + t for i, t in enumerate(mat(W["wo"], o))]
        h2 = norm(x2, W["gamma2"])
        gg, uu = mat(W["wg"], h2), mat(W["wu"], h2)
        act = [gg[j] / (1 + math.exp(-gg[j])) * uu[j] for j in range(dff)]
        ys.append([x2[i] + t for i, t in enumerate(mat(W["wd"], act))])
    return np.array(ys), np.array(kc), np.array(vc)


def test_layer_forward_brute_force_tiny():
    rng = np.random.default_rng(53)
    for trial in range(6):
        L, d, Hq, Hkv, D, dff = 6, 4, 2, (1, 2)[trial % 2], 2, 3
        x_src = rng.standard_normal((L, d))
        kc = rng.standard_normal((L, Hkv, D))
        vc = rng.standard_normal((L, Hkv, D))
        W = _layer_weights(rng, d, Hq, Hkv, D, dff, scale=0.5)
        idx = np.sort(rng.choice(L, size=int(rng.integers(1, L + 1)), replace=False))
        got = O.layer_forward(x_src=x_src, idx=idx, k_cache=kc, v_cache=vc, weights=W, Hq=Hq, Hkv=Hkv,
                              theta=10.0, eps=1e-5)
        y, kc2, vc2 = _brute_layer(x_src, idx, kc, vc, W, Hq, Hkv, D, 10.0, 1e-5)
        np.testing.assert_allclose(got["y"], y, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(got["k_cache"], kc2, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(got["v_cache"], vc2, rtol=1e-12, atol=1e-14)


def test_layer_forward_residual_paths_and_sampled_rows():
    rng = np.random.default_rng(54)
    L, d, Hq, Hkv, D, dff = 9, 8, 2, 2, 4, 6
    x_src = rng.standard_normal((L, d))
    kc = rng.standard_normal((L, Hkv, D))
    vc = rng.standard_normal((L, Hkv, D))
    W = _layer_weights(rng, d, Hq, Hkv, D, dff)
    idx = np.array([1, 4, 5, 8])
    # zero output projections: both residual paths carry x through unchanged
    Z = dict(W, wo=np.zeros_like(W["wo"]), wd=np.zeros_like(W["wd"]))
    got = O.layer_forward(x_src=x_src, idx=idx, k_cache=kc, v_cache=vc, weights=Z, Hq=Hq, Hkv=Hkv, theta=100.0,
                          eps=1e-6)
    np.testing.assert_allclose(got["y"], x_src[idx], rtol=0, atol=0)
    # a sample of rows gives the same rows as the whole set
    full = O.layer_forward(x_src=x_src, idx=idx, k_cache=kc, v_cache=vc, weights=W, Hq=Hq, Hkv=Hkv, theta=100.0,
                           eps=1e-6)
    part = O.layer_forward(x_src=x_src, idx=idx, k_cache=kc, v_cache=vc, weights=W, Hq=Hq, Hkv=Hkv, theta=100.0,
                           eps=1e-6, rows=np.array([2, 0]))
    np.testing.assert_allclose(part["y"], full["y"][[2, 0]], rtol=1e-14)
    # the recomputed rows' attention reads the refreshed cache rows (not the stale ones)
    assert not np.allclose(full["k_cache"][idx], kc[idx])
    np.testing.assert_array_equal(full["k_cache"][[0, 2, 3, 6, 7]], kc[[0, 2, 3, 6, 7]])
