"""GPU parity of the output projection fused with the decode (ec_lm_head_entropy) against the
float64 oracle: logits = hidden @ weight.T, then ids / entropy / log_conf.

Tolerances: the tensor cores multiply bf16 exactly and accumulate in fp32, so a logit is off
by about d_model * 2^-24 * sum_k |h_k w_k| at most (1e-5 typical here). Entropy and
log-confidence are held to 1e-3 absolute, as for the decode kernels. The id must match
exactly unless the oracle's two best logits are closer than the accumulation bound: then
the GPU's id must be one whose oracle logit lies within that bound of the maximum (where
several ids are correct, check that the chosen one is valid).
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module")
def E():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import entropy_gated_kv_gb300 as E

    E.lib()
    return E


def _dev(bits):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def run_case(E, h_bits, w_bits):
    ids, ent, conf = (t.cpu().numpy() for t in E.lm_head_entropy(_dev(h_bits), _dev(w_bits)))
    h = O.widen(h_bits, "bf16")
    w = O.widen(w_bits, "bf16")
    ids_o, ent_o, conf_o = O.lm_head_entropy(h, w)
    logits = h @ w.T
    bound = 2.0 * h.shape[1] * 2.0 ** -24 * (np.abs(h) @ np.abs(w).T).max(axis=1)
    for r in range(h.shape[0]):
        if ids[r] != ids_o[r]:
            gap = logits[r, ids_o[r]] - logits[r, ids[r]]
            assert 0 <= gap <= bound[r], (r, ids[r], ids_o[r], gap, bound[r])
    assert np.max(np.abs(ent - ent_o)) <= TOL, np.max(np.abs(ent - ent_o))
    assert np.max(np.abs(conf - conf_o)) <= TOL, np.max(np.abs(conf - conf_o))
    return ids, ent, conf


@pytest.mark.parametrize("n_rows,d_model,V,peaked", [
    (1, 64, 1, 0),           # one vocabulary entry: entropy 0
    (5, 128, 1000, 2),       # few rows (N padded to 32), ragged last vocabulary tile
    (32, 1024, 50257, 8),    # GPT-2-sized vocabulary, ragged
    (40, 512, 8192, 4),      # two 32-candidate chunks
    (64, 128, 777, 4),       # seven vocabulary tiles over few CTAs, the last one ragged
    (256, 256, 3000, 16),    # the most rows (N = 256, eight chunks)
])
def test_matches_oracle(E, n_rows, d_model, V, peaked):
    h, w = W.lm_head_inputs(n_rows, d_model, V, seed=n_rows + V, peaked=peaked)
    ids, ent, _ = run_case(E, h, w)
    if V == 1:
        assert np.all(ids == 0) and np.all(np.abs(ent) <= TOL)


def test_llada_output_projection(E):
    # LLaDA-8B's output layer: d_model 4096, V 126464 (1.04 GB of bf16 weight), 32 candidates
    h, w = W.lm_head_inputs(32, 4096, 126464, seed=5, peaked=8)
    run_case(E, h, w)


def test_zero_weight_gives_uniform(E):
    # all logits 0: H = ln V, the first index, log_conf = -ln V
    V, d = 50000, 64
    h = W.to_bf16_bits(np.random.default_rng(3).standard_normal((7, d)).astype(np.float32))
    w = np.zeros((V, d), dtype=np.uint16)
    ids, ent, conf = (t.cpu().numpy() for t in E.lm_head_entropy(_dev(h), _dev(w)))
    assert np.all(ids == 0)
    assert np.max(np.abs(ent - math.log(V))) <= TOL
    assert np.max(np.abs(conf + math.log(V))) <= TOL
