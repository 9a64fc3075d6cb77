"""Shared helpers of the parity tests: the same seeded host buffers (from
``synth``) become CUDA tensors for the library and numpy arrays for the
oracle.  Nothing here computes any part of the decode step."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Bar of the parity tests: max relative error 2e-2 on floating-point outputs,
# where the error of element i is |gpu_i - ref_i| / max(|ref_i|, rms(ref)).
# The rms floor keeps elements near zero from dividing by ~0; it is the
# vector's own scale, so the bar stays relative.
TOL = 2e-2
# Greedy tokens must agree wherever the oracle's top-2 logit margin exceeds this.
MARGIN = 1e-2


def rel_err(gpu, ref) -> float:
    g = np.asarray(gpu, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    if r.size == 0:
        return 0.0
    scale = np.sqrt(np.mean(r * r))
    den = np.maximum(np.abs(r), scale if scale > 0 else 1.0)
    return float(np.max(np.abs(g - r) / den))


def assert_close(gpu, ref, tol=TOL, what=""):
    e = rel_err(gpu, ref)
    assert e <= tol, f"{what}: max relative error {e:.3e} > {tol:.1e}"
    return e


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 CUDA tensor (exact)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_f32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def dev_i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


class HostModel:
    """Seeded host weights of a workload (uint16 bf16 bits), shared by both sides."""

    def __init__(self, m: synth.ModelShape, seed: int = 0, embed: bool = True, head: bool = True):
        self.m = m
        self.seed = seed
        self.layers = [synth.make_layer(seed, m, l) for l in range(m.n_layers)]
        self.embed = synth.make_embedding(seed, m) if (embed or head) else None
        self.final_norm = synth.make_final_norm(seed, m) if head else None
        self.lm_head = self.embed if head else None
        self.use_embed = embed

    def to_gpu(self):
        import greedy_decode_step_gb300 as gd
        m = self.m
        layers = [{k: dev_bf16(v) for k, v in l.items()} for l in self.layers]
        E = dev_bf16(self.embed) if self.embed is not None else None
        fn = dev_bf16(self.final_norm) if self.final_norm is not None else None
        self._gpu = gd.Model(m.n_layers, m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate, m.vocab,
                             m.rms_eps, m.rope_theta, layers, embed=E if self.use_embed else None,
                             final_norm=fn, lm_head=E if self.lm_head is not None else None)
        return self._gpu


def make_caches(m: synth.ModelShape, seed: int, batch: int, S_max: int, kv_len):
    """Per-layer [B, Hkv, S_max, D] uint16 caches, slots < kv_len[b] filled with bf16 N(0,1)."""
    K, V = [], []
    for l in range(m.n_layers):
        k = np.zeros((batch, m.n_kv_heads, S_max, m.head_dim), dtype=np.uint16)
        v = np.zeros_like(k)
        for b in range(batch):
            if kv_len[b] > 0:
                synth.make_kv_prefix(seed, m, l, b, kv_len[b], "k", k[b])
                synth.make_kv_prefix(seed, m, l, b, kv_len[b], "v", v[b])
        K.append(k)
        V.append(v)
    return K, V
