"""The benchmark's algorithmic byte count (the numerator of its roofline)
against the weight and cache shapes of the workloads, counted another way:
from the per-tensor shapes that generate the weights."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_every_weight_is_counted_once_and_every_cached_key_once():
    m = synth.workload("dense4b").model
    per_layer = sum(2 * int(np.prod(s)) for s in synth.layer_shapes(m).values())
    head = 2 * m.vocab * m.hidden + 2 * m.hidden  # tied LM head (the embedding) + final norm gain
    w, kv = bench.bytes_per_step(m, [511, 600], B=1, head=True)
    assert w == m.n_layers * per_layer + head
    # K and V, 36 layers, 8 KV heads, 128 dims, bf16: 147,456 bytes per cached token
    assert 2 * m.n_layers * m.n_kv_heads * m.head_dim * 2 == 147_456
    assert kv == 147_456 * (512 + 601)
    assert round(w / 1e9, 3) == 8.045


def test_one_layer_without_head():
    m = synth.workload("layer4b").model
    w, kv = bench.bytes_per_step(m, [4096], B=1, head=False)
    assert w == sum(2 * int(np.prod(s)) for s in synth.layer_shapes(m).values())
    assert kv == 2 * m.n_kv_heads * m.head_dim * 2 * 4097
    # 201.9 MB of weights and 16.8 MB of cache
    assert round(w / 1e6, 1) == 201.9 and round(kv / 1e6, 1) == 16.8
