"""dec_gqa_decode_attn_noalloc: attention for callers that cannot hand the
library any device memory (a host application whose pool owns every device
allocation, or a latency-critical loop that must not call cudaMalloc).  It
runs on the library's built-in scratch array and must give the result of the
workspace entry point, call after call (the array keeps the previous call's
contents, so whatever must start at zero has to be cleared each time).

Kept in a file of its own, collected last."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import TOL, assert_close, dev_bf16, dev_f32, dev_i32

pytestmark = pytest.mark.gpu

gd = pytest.importorskip("greedy_decode_step_gb300")


def _case(seed, B, Hq, Hkv, D, S_max, pos):
    Kb = synth.normal_bf16(seed, "K", (B, Hkv, S_max, D))
    Vb = synth.normal_bf16(seed, "V", (B, Hkv, S_max, D))
    qh = synth.bf16_to_f32(synth.normal_bf16(seed + 1, "q", (B, Hq, D)))
    return (dev_f32(qh), dev_bf16(Kb), dev_bf16(Vb), dev_i32(pos)), (qh, Kb, Vb)


def test_noalloc_attention_matches_workspace_entry_point_twice_in_a_row():
    """Two calls in a row (two shapes, two split plans): each is bit for bit
    the workspace call's result (the same kernel and plan), and the first
    also matches the fp64 oracle's attention row by row."""
    gd.lib()
    gd.device_error(clear=True)
    cases = [
        (11, 3, 32, 8, 128, 3000, [2999, 0, 1500]),   # several splits per group, ragged rows
        (12, 2, 12, 3, 128, 9000, [8191, 77]),        # a second call with another shape and plan
    ]
    for i, (seed, B, Hq, Hkv, D, S_max, pos) in enumerate(cases):
        (q, K, V, p), (qh, Kb, Vb) = _case(seed, B, Hq, Hkv, D, S_max, pos)
        ref = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
        gd.dec_gqa_decode_attn(q, K, V, p, ref)
        got = torch.full_like(ref, float("nan"))
        gd.dec_gqa_decode_attn_noalloc(q, K, V, p, got)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
        if i == 0:
            g = got.cpu().numpy()
            for b in range(B):
                o = oracle.attention(qh[b], Kb[b], Vb[b], pos[b] + 1)
                assert_close(g[b], o, TOL, f"row {b} against the oracle")
    assert gd.device_error(clear=True) == 0


def test_noalloc_attention_refuses_plans_beyond_its_scratch():
    gd.lib()
    # 16 rows x 16 KV heads x many splits x 16 query heads per group needs far more than 4 MiB
    q = torch.zeros((16, 256, 128), dtype=torch.float32, device="cuda")
    K = torch.zeros((16, 16, 64, 128), dtype=torch.bfloat16, device="cuda")
    p = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(gd.DecError, match="built-in scratch"):
        gd.dec_gqa_decode_attn_noalloc(q, K, K, p, torch.empty_like(q), num_splits=2)
