"""Seeded synthetic inputs shared by the oracle tests, the CUDA parity tests and
the benchmark.

Nothing here computes any part of the decode step: this module draws random
numbers (Philox4x32-10 in ``synth.c``), rounds them to bf16 and lays them out
as the workloads below describe.  Both sides of every parity check receive the
same host buffers from here; neither side imports the other.

Workloads (dense GQA decoder shapes of the rollout decode benchmark on the
segment-KI pull request, with synthetic values):

* ``tiny``      one layer + LM head, H=256, Hq=4, Hkv=2, D=64, I=704, V=1024,
                128-token N(0,1) KV cache, residual N(0,1), gains 1+N(0,0.1)
* ``layer4b``   one 4B-class layer, H=2560, Hq=32, Hkv=8, D=128, I=9728,
                4096-token N(0,1) KV cache
* ``dense4b``   36 such layers, V=151936, tied LM head, b=1, 512-token prompt
* ``dense4b_b8`` the same model at b=8, KV lengths U{1024..32768}
* ``gqa12x3``   24 layers, H=1536, Hq=12, Hkv=3, D=128, I=8960, V=151936,
                b=16, KV length 8192
* ``gqa6x3``    one layer with Hq=6, Hkv=3 (query-to-KV-group mapping check)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import zlib
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` beside it (host code, any CPU)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        lib.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_float, ctypes.c_float, ctypes.c_void_p, ctypes.c_int]
        lib.synth_normal_bf16.restype = None
        lib.synth_uniform_int.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        lib.synth_uniform_int.restype = None
        lib.synth_philox4x32_10.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_philox4x32_10.restype = None
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def stream_id(name: str) -> int:
    """Stable 64-bit stream number for a tensor name."""
    b = name.encode()
    return (zlib.crc32(b) << 32) | zlib.crc32(b[::-1] + b"#")


def philox4x32_10(ctr, key):
    """One Philox4x32-10 block (for the generator's own known-answer test)."""
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().synth_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def normal_bf16(seed: int, name: str, shape, mean: float = 0.0, std: float = 1.0, out: np.ndarray | None = None,
                offset: int = 0) -> np.ndarray:
    """bf16(mean + std*N(0,1)) as raw uint16 bits, C-contiguous, of ``shape``."""
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    if n:
        _load().synth_normal_bf16(seed, stream_id(name), offset, n, mean, std, out.ctypes.data, _threads())
    return out


def uniform_int(seed: int, name: str, shape, low: int, high: int) -> np.ndarray:
    """int32 uniform on [low, high] inclusive."""
    n = int(np.prod(shape))
    out = np.empty(shape, dtype=np.int32)
    if n:
        _load().synth_uniform_int(seed, stream_id(name), 0, n, low, high, out.ctypes.data, _threads())
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_to_f32(bits).astype(np.float64)


# --------------------------------------------------------------------------- workloads


@dataclass
class ModelShape:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rope_theta: float = 1e6
    rms_eps: float = 1e-6
    weight_std: float = 0.02
    gain_std: float = 0.02     # norm gains are 1 + N(0, gain_std)
    tied: bool = True


@dataclass
class Workload:
    name: str
    model: ModelShape
    batch: int
    kv_len: list            # per-sequence KV prefix length (synthetic N(0,1) entries) or prompt-filled
    steps: int
    prompt_len: int = 0     # >0: the KV cache is filled by a teacher-forced prompt instead of N(0,1)
    eos_id: int = -1
    seed: int = 0
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def max_seq(self) -> int:
        return max(self.kv_len) + self.prompt_len + self.steps + 1


def workload(name: str, **over) -> Workload:
    """The named workload; keyword overrides (e.g. ``steps=4``) give reduced variants."""
    if name == "tiny":
        m = ModelShape(1, 256, 4, 2, 64, 704, 1024, gain_std=0.1)
        w = Workload("tiny", m, 1, [128], 1, description="one layer + LM head, 128-token KV, one step")
    elif name == "layer4b":
        m = ModelShape(1, 2560, 32, 8, 128, 9728, 151936)
        w = Workload("layer4b", m, 1, [4096], 1, description="one 4B-class layer, 4096-token KV, one step",
                     extra={"lm_head": False})
    elif name == "dense4b":
        m = ModelShape(36, 2560, 32, 8, 128, 9728, 151936)
        w = Workload("dense4b", m, 1, [0], 256, prompt_len=512, eos_id=0,
                     description="36-layer 4B-class, b=1, 512-token prompt, 256 greedy steps")
    elif name == "dense4b_b8":
        m = ModelShape(36, 2560, 32, 8, 128, 9728, 151936)
        seed = over.get("seed", 0)
        lens = uniform_int(seed, "dense4b_b8.kv_len", (8,), 1024, 32768).tolist()
        w = Workload("dense4b_b8", m, 8, lens, 64, eos_id=0,
                     description="36-layer 4B-class, b=8, KV lengths U{1024..32768}, 64 steps")
    elif name == "gqa12x3":
        m = ModelShape(24, 1536, 12, 3, 128, 8960, 151936)
        w = Workload("gqa12x3", m, 16, [8192] * 16, 128, eos_id=0,
                     description="24-layer Hq=12/Hkv=3, b=16, KV 8192, 128 greedy steps")
    elif name == "gqa6x3":
        m = ModelShape(1, 768, 6, 3, 128, 1024, 1024)
        w = Workload("gqa6x3", m, 1, [64], 1, description="Hq=6/Hkv=3 query-to-KV-group mapping check")
    else:
        raise KeyError(name)
    for k, v in over.items():
        if hasattr(w, k):
            setattr(w, k, v)
        elif hasattr(w.model, k):
            setattr(w.model, k, v)
        else:
            raise KeyError(k)
    return w


LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")


def layer_shapes(m: ModelShape) -> dict:
    H, Hq, Hkv, D, I = m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate
    return {"attn_norm": (H,), "wq": (Hq * D, H), "wk": (Hkv * D, H), "wv": (Hkv * D, H),
            "wo": (H, Hq * D), "mlp_norm": (H,), "wg": (I, H), "wu": (I, H), "wd": (H, I)}


def make_layer(seed: int, m: ModelShape, layer: int, alloc=None) -> dict:
    """bf16 bits of one layer's weights (nn.Linear layout [out, in]) and gains."""
    out = {}
    for name, shape in layer_shapes(m).items():
        buf = alloc(shape) if alloc is not None else None
        if name.endswith("norm"):
            out[name] = normal_bf16(seed, f"L{layer}.{name}", shape, 1.0, m.gain_std, out=buf)
        else:
            out[name] = normal_bf16(seed, f"L{layer}.{name}", shape, 0.0, m.weight_std, out=buf)
    return out


def make_gated_attention(seed: int, m: ModelShape, layer: int, rot_dim: int) -> dict:
    """bf16 bits of one layer's gated-attention parts: per-head q/k RMSNorm gains
    [D] of 1 + N(0, gain_std) and the output-gate projection [Hq*D, H] of
    N(0, weight_std), with the rotary width ``rot_dim``."""
    D = m.head_dim
    return {"rot_dim": int(rot_dim),
            "q_norm": normal_bf16(seed, f"L{layer}.q_norm", (D,), 1.0, m.gain_std),
            "k_norm": normal_bf16(seed, f"L{layer}.k_norm", (D,), 1.0, m.gain_std),
            "wgate": normal_bf16(seed, f"L{layer}.wgate", (m.n_heads * D, m.hidden), 0.0, m.weight_std)}


def make_embedding(seed: int, m: ModelShape, alloc=None) -> np.ndarray:
    shape = (m.vocab, m.hidden)
    return normal_bf16(seed, "embed", shape, 0.0, m.weight_std, out=alloc(shape) if alloc else None)


def make_final_norm(seed: int, m: ModelShape) -> np.ndarray:
    return normal_bf16(seed, "final_norm", (m.hidden,), 1.0, m.gain_std)


def make_kv_prefix(seed: int, m: ModelShape, layer: int, b: int, length: int, which: str, out: np.ndarray) -> None:
    """Fill ``out`` ([Hkv, length, D] view rows) with bf16 N(0,1) for sequence b of layer ``layer``."""
    Hkv, D = m.n_kv_heads, m.head_dim
    for g in range(Hkv):
        normal_bf16(seed, f"L{layer}.{which}.b{b}.g{g}", (length, D), 0.0, 1.0, out=out[g, :length])


def make_residual(seed: int, batch: int, hidden: int) -> np.ndarray:
    """Residual-stream input as fp32 holding bf16 N(0,1) values."""
    return bf16_to_f32(normal_bf16(seed, "residual", (batch, hidden)))


def make_tokens(seed: int, name: str, shape, vocab: int) -> np.ndarray:
    return uniform_int(seed, name, shape, 0, vocab - 1)


def make_logits(seed: int, name: str, batch: int, vocab: int, std: float = 1.0, fine: bool = True) -> np.ndarray:
    """float32 logits [batch, vocab]: a bf16 draw of std * N(0,1) plus, with
    ``fine``, a second bf16 draw of std/256 * N(0,1), so that values rarely tie
    (without it, bf16-valued logits tie in large groups)."""
    a = bf16_to_f32(normal_bf16(seed, name, (batch, vocab), 0.0, std))
    if fine:
        a = a + bf16_to_f32(normal_bf16(seed, name + ".fine", (batch, vocab), 0.0, std / 256.0))
    return np.ascontiguousarray(a, dtype=np.float32)


def make_uniforms(seed: int, name: str, n: int) -> np.ndarray:
    """float32 draws k / 2^24 on [0, 1), k uniform integers."""
    return (uniform_int(seed, name, (n,), 0, (1 << 24) - 1).astype(np.float64) / float(1 << 24)).astype(np.float32)
