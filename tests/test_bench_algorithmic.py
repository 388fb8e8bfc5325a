"""The roofline's algorithmic work per launch (bench.algorithmic) against hand-computed values.

`achieved` in the bench's roofline object is these bytes or flops divided by a measured launch
time, so a slip here would misstate every fraction. The expected values are written out from the
shapes, term by term: the decode reads every candidate logit once and writes 12 bytes per row;
attention reads K and V of the whole cache once, reads the recompute rows' queries and writes
their outputs, and does 2 flops per multiply-add in QK^T and in PV.
"""
import bench
import workloads as W


def test_llada_layer_partial_step():
    w = W.workload(2)  # B 1, 32 x 128 MHA, L 1024, 32 candidates, V 126464 bf16
    a = bench.algorithmic(w, 95)
    assert a["entropy_decode_bytes"] == 32 * 126464 * 2 + 32 * 12  # 8.09 MB
    kv = 1024 * 32 * 128 * 2  # one cache, bf16
    q_out = 95 * 32 * 128 * 2  # the recompute rows' queries (and, again, outputs)
    assert a["partial_attention_bytes"] == 2 * kv + 2 * q_out  # 18.3 MB
    assert a["partial_attention_flops"] == 2 * (2 * 32 * 95 * 1024 * 128)  # 1.59 GFLOP
    assert round(a["partial_attention_bytes"] / 1e6, 1) == 18.3


def test_llada_layer_full_step():
    w = W.workload(2)
    a = bench.algorithmic(w, 1024)
    assert a["partial_attention_bytes"] == 4 * 1024 * 32 * 128 * 2  # K, V, Q and O: 33.6 MB
    assert a["partial_attention_flops"] == 4 * 32 * 1024 * 1024 * 128  # 17.2 GFLOP


def test_dream_batch_full_step():
    w = W.workload(3)  # B 8, 28 query / 4 KV heads x 128, L 2048, V 152064 bf16
    R = 8 * 2048  # every position of every sequence
    a = bench.algorithmic(w, R)
    assert a["entropy_decode_bytes"] == 8 * 32 * 152064 * 2 + 8 * 32 * 12  # 77.9 MB
    assert a["partial_attention_flops"] == 4 * 28 * R * 2048 * 128  # 481 GFLOP
    assert round(a["partial_attention_flops"] / 1e9) == 481
    kv = 8 * 2048 * 4 * 128 * 2
    assert a["partial_attention_bytes"] == 2 * kv + 2 * R * 28 * 128 * 2


def test_tiny_fp32_logits():
    w = W.workload(1)  # V 32000 fp32 logits
    a = bench.algorithmic(w, 47)
    assert a["entropy_decode_bytes"] == 32 * 32000 * 4 + 32 * 12
