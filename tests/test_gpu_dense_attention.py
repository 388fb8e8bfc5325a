"""GPU parity of the dense attention for full steps (ec_dense_attention: two query tiles per
CTA, one softmax warpgroup per tile) against the float64 oracle.

Tolerance as for the partial attention (bf16 outputs): per head ||O - O_ref||_F <= 2e-2
||O_ref||_F and per element |O - O_ref| <= 2e-2 (|O_ref| + rms(O_ref)). Every row must be
written. Cases: the LLaDA-8B layer (MHA 32 x 128, L 1024) and the Dream-7B batch (B 8, GQA
28 / 4 x 128, L 2048, the shape the bench times) on sampled rows, grouped queries with
a ragged key block and an odd tile count (the last item's second tile past the end), several
sequences, a tile count that needs several items per CTA, a single ragged block, a single
position, 16 query heads per KV head (8 positions per tile), and a sharp softmax
(the lazy rescale).
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import attention_close, bf16_bits, bf16_tensor

pytestmark = pytest.mark.gpu

SENTINEL = 0x7F7F  # a bf16 bit pattern the kernel never writes


@pytest.fixture(scope="module")
def E():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import entropy_gated_kv_gb300 as E

    E.lib()
    return E


def run_dense(E, B, L, Hq, Hkv, seed=0, q_scale=1.0, rows=None):
    import torch

    D = 128
    rng = np.random.default_rng(seed)
    q = W.to_bf16_bits(rng.standard_normal((B, L, Hq, D), dtype=np.float32) * np.float32(q_scale))
    k = W.to_bf16_bits(rng.standard_normal((B, L, Hkv, D), dtype=np.float32))
    v = W.to_bf16_bits(rng.standard_normal((B, L, Hkv, D), dtype=np.float32))
    sc = 1.0 / math.sqrt(D)
    p = E.Params(B=B, L=L, Hq=Hq, Hkv=Hkv, D=D, V=8, C_max=1, k=1)
    out = torch.full((B, L, Hq, D), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.dense_attention(p, bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), out, dev_err=dev_err)
    torch.cuda.synchronize()
    assert int(dev_err.item()) == 0
    got = bf16_bits(out)
    assert not (got == SENTINEL).all(axis=-1).any(), "a row was left unwritten"
    sel = np.arange(L) if rows is None else np.asarray(rows)
    for b in range(B):
        ref = O.attention(O.widen(q[b, sel], "bf16"), O.widen(k[b], "bf16"), O.widen(v[b], "bf16"), sc)
        ok, msg = attention_close(O.widen(got[b, sel], "bf16"), ref)
        assert ok, f"b={b}: {msg}"
    return got


def tile_edges(L, nr, step=7):
    """Sampled rows: every step-th position plus the first and last position of every tile."""
    s = set(range(0, L, step))
    for t0 in range(0, L, nr):
        s.update((t0, min(L, t0 + nr) - 1))
    return sorted(s)


def test_llada_layer_shape(E):
    run_dense(E, B=1, L=1024, Hq=32, Hkv=32, seed=1, rows=tile_edges(1024, 128))


def test_dream_batch_shape(E):
    # g = 7: 18 positions per tile, 114 tiles per (sequence, KV head), 57 items each, 1824 items
    # over the persistent CTAs
    run_dense(E, B=8, L=2048, Hq=28, Hkv=4, seed=10, rows=tile_edges(2048, 128 // 7, step=13))


def test_gqa_ragged_block_odd_tiles(E):
    # g = 7: 18 positions per tile, ceil(520 / 18) = 29 tiles per head (the last item's second
    # tile lies past the end); 520 = 4 * 128 + 8 keys (a ragged last block)
    run_dense(E, B=2, L=520, Hq=28, Hkv=4, seed=2)


def test_mha_odd_tiles_three_sequences(E):
    run_dense(E, B=3, L=384, Hq=2, Hkv=2, seed=3)


def test_many_items_per_cta(E):
    # 4 sequences x 8 heads x 8 tile pairs = 256 items: more than one per SM, so CTAs take
    # several items (the Q, S and O buffers are reused across items)
    run_dense(E, B=4, L=2048, Hq=8, Hkv=8, seed=4, rows=tile_edges(2048, 128, step=11))


def test_single_ragged_block(E):
    run_dense(E, B=1, L=100, Hq=8, Hkv=2, seed=5)


def test_single_position(E):
    # L = 1: one item whose first tile holds one row and whose second tile is past the end; one
    # key, so every output row is that key's V row
    got = run_dense(E, B=2, L=1, Hq=4, Hkv=2, seed=8)
    assert got.shape == (2, 1, 4, 128)


def test_sixteen_query_heads_per_kv_head(E):
    # g = 16 packs 8 positions per tile; L = 37 gives 5 tiles (3 items, the last one half empty)
    # and a single ragged key block
    run_dense(E, B=2, L=37, Hq=32, Hkv=2, seed=9)


def test_sharp_softmax_rescale(E):
    run_dense(E, B=1, L=640, Hq=4, Hkv=4, seed=6, q_scale=8.0)


def test_matches_partial_attention_with_every_row(E):
    # the same attention through the partial-attention kernel with R = L: both within the
    # oracle's tolerance, and close to each other
    import torch

    B, L, Hq, Hkv, D = 1, 768, 16, 16, 128
    rng = np.random.default_rng(7)
    q = bf16_tensor(W.to_bf16_bits(rng.standard_normal((B, L, Hq, D), dtype=np.float32)))
    k = bf16_tensor(W.to_bf16_bits(rng.standard_normal((B, L, Hkv, D), dtype=np.float32)))
    v = bf16_tensor(W.to_bf16_bits(rng.standard_normal((B, L, Hkv, D), dtype=np.float32)))
    p = E.Params(B=B, L=L, Hq=Hq, Hkv=Hkv, D=D, V=8, C_max=1, k=1)
    a = torch.empty(B, L, Hq, D, dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    E.dense_attention(p, q, k, v, a)
    R = torch.full((B,), L, dtype=torch.int32, device="cuda")
    E.partial_attention(p, q, k, v, R, b)
    torch.cuda.synchronize()
    ok, msg = attention_close(O.widen(bf16_bits(a)[0], "bf16"), O.widen(bf16_bits(b)[0], "bf16"))
    assert ok, msg
