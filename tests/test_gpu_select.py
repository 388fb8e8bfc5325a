"""GPU parity of stages (b)+(c): commit, max-entropy gate, decode history, recompute set and
the K/V scatter. Both sides receive the same fp32 entropies and confidences, so every
decision is taken on identical values and every output must match bit for bit."""
import numpy as np
import pytest

import oracle as O
from tests._helpers import bf16_bits, bf16_tensor, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import entropy_gated_kv_gb300 as E

    E.lib()
    return E


def make_case(rng, B, L, C_max, k, n_dec, tau):
    tokens = rng.integers(0, 1000, size=(B, L)).astype(np.int32)
    mask = np.zeros((B, L), np.uint8)
    cand_pos = np.zeros((B, C_max), np.int32)
    cand_count = np.zeros(B, np.int32)
    ring = np.zeros((B, k), np.int32)
    head = np.zeros(B, np.int32)
    count = np.zeros(B, np.int32)
    for b in range(B):
        nm = int(rng.integers(1, min(L, 3 * C_max) + 1))
        masked = np.sort(rng.choice(L, size=nm, replace=False))
        mask[b, masked] = 1
        tokens[b, masked] = -1
        c = int(rng.integers(0, min(C_max, nm) + 1))
        cp = rng.permutation(masked)[:c]
        cand_pos[b, :c] = cp
        cand_count[b] = c
        decoded = [p for p in range(L) if not mask[b, p]]
        rng.shuffle(decoded)
        nh = int(rng.integers(0, len(decoded) + 1))
        r, h, n = O.history_push(np.zeros(k, np.int64), 0, 0, decoded[:nh])
        ring[b], head[b], count[b] = r, h, n
    rows = B * C_max
    ids = rng.integers(0, 50000, size=rows).astype(np.int32)
    ent = (rng.integers(0, 8, size=rows) * 0.25).astype(np.float32)  # many exactly equal to tau
    conf = (-rng.integers(0, 4, size=rows) * 0.5).astype(np.float32)  # many ties
    return dict(tokens=tokens, mask=mask, cand_pos=cand_pos, cand_count=cand_count, ring=ring, ring_head=head,
                ring_count=count, ids=ids, ent=ent, conf=conf)


def oracle_select(c, b, C_max, n_dec, tau, L, gamma=0.0):
    rows = slice(b * C_max, (b + 1) * C_max)
    cp = c["cand_pos"][b]
    cnt = int(c["cand_count"][b])
    conf = c["conf"][rows].astype(np.float64)
    ent = c["ent"][rows].astype(np.float64)
    dec = O.select_decoded(cp, cnt, conf, n_dec, gamma)
    tokens = c["tokens"][b].astype(np.int64).copy()
    mask = c["mask"][b].copy()
    for i in dec:
        tokens[cp[i]] = c["ids"][rows][i]
        mask[cp[i]] = 0
    E_ = O.max_entropy(ent, dec)
    full = O.recompute_flag(E_, np.float32(tau))
    ring, head, count = O.history_push(c["ring"][b], int(c["ring_head"][b]), int(c["ring_count"][b]),
                                       [int(cp[i]) for i in dec])
    idx = O.recompute_set(mask, O.history_last(ring, head, count), full)
    return dict(tokens=tokens, mask=mask, dec_pos=[int(cp[i]) for i in dec], E=E_, flag=full, ring=ring,
                ring_head=head, ring_count=count, idx=idx)


# gamma: the confidence-threshold commit (0 = the n_dec most confident). The generated
# log-confidences lie on a grid of 0.5 (0, -0.5, -1, -1.5), so ln(gamma) is well clear of every
# value: -0.75 between grid points, and ln(0.999) just below 0 (only certain candidates pass).
@pytest.mark.parametrize("gamma", [0.0, float(np.exp(-0.75)), 0.999])
@pytest.mark.parametrize("seed,B,L,C_max,k,n_dec,tau", [
    (0, 4, 16, 8, 4, 1, 1.0),
    (1, 8, 64, 16, 8, 3, 0.75),
    (2, 3, 1000, 32, 64, 1, 1.0),
    (3, 2, 100, 32, 5, 12, 0.5),   # n_dec > k: only the last k decoded stay in the history
    (4, 5, 4097, 64, 64, 2, 1.25),
    (5, 1, 32768, 32, 64, 1, 1.0),
    (6, 2, 12, 12, 12, 12, 0.0),
])
def test_select_recompute_matches_oracle(E, seed, B, L, C_max, k, n_dec, tau, gamma):
    import torch

    rng = np.random.default_rng(seed)
    c = make_case(rng, B, L, C_max, k, n_dec, tau)
    p = E.Params(B=B, L=L, Hq=1, Hkv=1, D=64, V=50000, C_max=C_max, k=k, n_dec=n_dec, tau=tau,
                 conf_threshold=gamma)
    st = E.DecodeState.from_arrays(p, tokens=c["tokens"], mask=c["mask"], ring=c["ring"], ring_head=c["ring_head"],
                                   ring_count=c["ring_count"])
    E.select_recompute(p, st, to_dev(c["cand_pos"]), to_dev(c["cand_count"]), to_dev(c["ids"]), to_dev(c["ent"]),
                       to_dev(c["conf"]))
    torch.cuda.synchronize()
    got = {f: getattr(st, f).cpu().numpy() for f in st.FIELDS}
    assert got["dev_err"][0] == 0
    for b in range(B):
        o = oracle_select(c, b, C_max, n_dec, tau, L, gamma)
        np.testing.assert_array_equal(got["tokens"][b], o["tokens"])
        np.testing.assert_array_equal(got["mask"][b], o["mask"])
        nd = len(o["dec_pos"])
        assert got["dec_pos"][b, :nd].tolist() == o["dec_pos"]
        assert (got["dec_pos"][b, nd:] == -1).all()
        assert float(got["E"][b]) == o["E"]
        assert bool(got["flag"][b]) == o["flag"]
        assert int(got["ring_head"][b]) == o["ring_head"] and int(got["ring_count"][b]) == o["ring_count"]
        np.testing.assert_array_equal(got["ring"][b], o["ring"])
        R = int(got["R"][b])
        assert R == len(o["idx"])
        np.testing.assert_array_equal(got["idx"][b, :R], o["idx"])


def test_select_reports_bad_candidates(E):
    import torch

    p = E.Params(B=1, L=16, Hq=1, Hkv=1, D=64, V=100, C_max=4, k=4, n_dec=1, tau=1.0)
    mask = np.zeros((1, 16), np.uint8)
    mask[0, 10:] = 1
    st = E.DecodeState.from_arrays(p, mask=mask)
    cand = np.array([[3, 99, 12, 12]], np.int32)  # decoded, out of range, valid, duplicate
    E.select_recompute(p, st, to_dev(cand), to_dev(np.array([4], np.int32)), to_dev(np.arange(4, dtype=np.int32)),
                       to_dev(np.zeros(4, np.float32)), to_dev(np.zeros(4, np.float32)))
    status, word = E.read_device_error(st.dev_err)
    assert status == 4 and word & 0x1  # EC_ERR_DEVICE_CHECK, EC_DEVERR_BAD_CAND_POS
    torch.cuda.synchronize()
    assert st.dec_pos.cpu().numpy()[0, 0] == 12 and st.mask.cpu().numpy()[0, 12] == 0


@pytest.mark.parametrize("by_position", [False, True])
def test_kv_scatter_bit_exact(E, by_position):
    import torch

    rng = np.random.default_rng(7)
    B, L, Hkv, D = 3, 300, 4, 128
    p = E.Params(B=B, L=L, Hq=Hkv, Hkv=Hkv, D=D, V=10, C_max=1, k=1)
    cache_k = rng.integers(0, 65535, size=(B, L, Hkv, D), dtype=np.uint16)
    cache_v = rng.integers(0, 65535, size=(B, L, Hkv, D), dtype=np.uint16)
    new_k = rng.integers(0, 65535, size=(B, L, Hkv, D), dtype=np.uint16)
    new_v = rng.integers(0, 65535, size=(B, L, Hkv, D), dtype=np.uint16)
    Rs = np.array([0, 17, L], np.int32)
    idx = np.zeros((B, L), np.int32)
    for b in range(B):
        idx[b, : Rs[b]] = np.sort(rng.choice(L, size=Rs[b], replace=False))
    kc, vc = bf16_tensor(cache_k), bf16_tensor(cache_v)
    E.kv_scatter(p, kc, vc, bf16_tensor(new_k), bf16_tensor(new_v), to_dev(idx), to_dev(Rs), src_by_position=by_position)
    torch.cuda.synchronize()
    want_k, want_v = cache_k.copy(), cache_v.copy()
    for b in range(B):
        for r in range(Rs[b]):
            src = idx[b, r] if by_position else r
            want_k[b, idx[b, r]] = new_k[b, src]
            want_v[b, idx[b, r]] = new_v[b, src]
    np.testing.assert_array_equal(bf16_bits(kc), want_k)
    np.testing.assert_array_equal(bf16_bits(vc), want_v)


def test_kv_scatter_reports_bad_idx(E):
    import torch

    B, L, Hkv, D = 1, 8, 1, 64
    p = E.Params(B=B, L=L, Hq=1, Hkv=1, D=D, V=10, C_max=1, k=1)
    z = np.zeros((B, L, Hkv, D), np.uint16)
    kc, vc = bf16_tensor(z), bf16_tensor(z)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = np.array([[0, 9, -1, 3, 0, 0, 0, 0]], np.int32)
    E.kv_scatter(p, kc, vc, bf16_tensor(z + 1), bf16_tensor(z + 1), to_dev(idx), to_dev(np.array([4], np.int32)),
                 dev_err=dev_err)
    status, word = E.read_device_error(dev_err)
    assert status == 4 and word & 0x2
    got = bf16_bits(kc)[0, :, 0, 0]
    assert got.tolist() == [1, 0, 0, 1, 0, 0, 0, 0]
