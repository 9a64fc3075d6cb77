"""fp64 CPU oracle for the greedy decode step (plain C in ``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg are the only callers.  It shares
no code with the CUDA path and does not import it.

Inputs are bf16 bit patterns (numpy ``uint16``) for weights and caches and
float64 (or anything convertible) for activations.  Every function here is a
thin ctypes wrapper; all arithmetic is in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int64
_D = ctypes.c_double


class Dims(ctypes.Structure):
    _fields_ = [("H", _I), ("Hq", _I), ("Hkv", _I), ("D", _I), ("I", _I), ("S_max", _I),
                ("eps", _D), ("theta", _D)]


class Taps(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("y_attn", "q", "k", "v", "o", "y_mlp", "h")]


class AttnVariant(ctypes.Structure):
    _fields_ = [("rot_dim", _I), ("q_norm", _P), ("k_norm", _P), ("Wgate", _P)]


def build(force: bool = False) -> str:
    """Compile the oracle (plain -O2, no fast-math) into ``liboracle.so``."""
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        sig = {
            "orc_bf16_to_f64": (_D, [ctypes.c_uint16]),
            "orc_f64_to_bf16": (ctypes.c_uint16, [_D]),
            "orc_rmsnorm": (None, [_P, _P, _I, _D, _P]),
            "orc_add_rmsnorm": (None, [_P, _P, _P, _I, _D, _P]),
            "orc_linear": (None, [_P, _P, _I, _I, _P]),
            "orc_rope": (None, [_P, _I, _I, _D]),
            "orc_kv_head": (_I, [_I, _I, _I]),
            "orc_attention": (None, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
            "orc_attention_splitk": (None, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
            "orc_silu": (_D, [_D]),
            "orc_glu": (None, [_P, _P, _P, _I, _I, _P]),
            "orc_argmax": (_I, [_P, _I]),
            "orc_layer": (None, [ctypes.POINTER(Dims)] + [_P] * 11 + [_I, _P, ctypes.POINTER(Taps)]),
            "orc_layer_ex": (None, [ctypes.POINTER(Dims), ctypes.POINTER(AttnVariant)] + [_P] * 11
                             + [_I, _P, ctypes.POINTER(Taps)]),
            "orc_rope_partial": (None, [_P, _I, _I, _I, _D]),
            "orc_head_rmsnorm": (None, [_P, _I, _I, _P, _D]),
            "orc_sigmoid": (_D, [_D]),
            "orc_head": (_I, [_P, _P, _P, _I, _I, _D, _P]),
            "orc_step": (_I, [ctypes.POINTER(Dims), _I, _P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _P, _P]),
            "orc_step_ex": (_I, [ctypes.POINTER(Dims), _I, _P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _P, _P]),
            "orc_select": (_I, [_P, _I, _P, _I, _D, _D, _I, _D, _D, _P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    assert a.dtype == np.uint16 and a.flags.c_contiguous, "bf16 inputs are C-contiguous uint16 bit patterns"
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


# ----------------------------------------------------------------------------- primitives

def bf16_to_f64(v: int) -> float:
    return lib().orc_bf16_to_f64(int(v))


def f64_to_bf16(x: float) -> int:
    return int(lib().orc_f64_to_bf16(float(x)))


def round_bf16(a) -> np.ndarray:
    """Element-wise fp64 -> bf16 bits (nearest, ties to even)."""
    a = _f64(a)
    f = lib().orc_f64_to_bf16
    return np.array([f(float(x)) for x in a.ravel()], dtype=np.uint16).reshape(a.shape)


def rmsnorm(r, gamma, eps: float, x=None):
    """Returns (r_after_add, y)."""
    r = _f64(r).copy()
    gamma = _u16(gamma)
    H = r.shape[-1]
    y = np.empty_like(r)
    xs = None if x is None else _f64(x)
    for b in range(r.size // H):
        lib().orc_add_rmsnorm(None if xs is None else xs.reshape(-1, H)[b].ctypes.data,
                              r.reshape(-1, H)[b].ctypes.data, gamma.ctypes.data, H, eps,
                              y.reshape(-1, H)[b].ctypes.data)
    return r, y


def linear(W, x):
    W = _u16(W)
    x = _f64(x)
    N, K = W.shape
    X = x.reshape(-1, K)
    y = np.empty((X.shape[0], N))
    for b in range(X.shape[0]):
        xb = np.ascontiguousarray(X[b])
        lib().orc_linear(W.ctypes.data, xb.ctypes.data, N, K, y[b].ctypes.data)
    return y.reshape(x.shape[:-1] + (N,))


def rope(v, p: int, theta: float):
    """RoPE of head vectors v[..., D] at absolute position p."""
    v = _f64(v).copy()
    D = v.shape[-1]
    flat = v.reshape(-1, D)
    for i in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[i])
        lib().orc_rope(row.ctypes.data, D, int(p), float(theta))
        flat[i] = row
    return flat.reshape(v.shape)


def rope_partial(v, rot_dim: int, p: int, theta: float):
    """RoPE of the first rot_dim dims of head vectors v[..., D] at position p; the rest unchanged."""
    v = _f64(v).copy()
    D = v.shape[-1]
    flat = v.reshape(-1, D)
    for i in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[i])
        lib().orc_rope_partial(row.ctypes.data, D, int(rot_dim), int(p), float(theta))
        flat[i] = row
    return flat.reshape(v.shape)


def head_rmsnorm(v, gain, eps: float):
    """RMSNorm of each head vector v[..., D] with the shared effective gain [D] (bf16 bits)."""
    v = _f64(v).copy()
    D = v.shape[-1]
    flat = np.ascontiguousarray(v.reshape(-1, D))
    lib().orc_head_rmsnorm(flat.ctypes.data, flat.shape[0], D, _u16(gain).ctypes.data, float(eps))
    return flat.reshape(v.shape)


def sigmoid(z: float) -> float:
    return float(lib().orc_sigmoid(float(z)))


def kv_head(h: int, Hq: int, Hkv: int) -> int:
    return int(lib().orc_kv_head(h, Hq, Hkv))


def attention(q, Kc, Vc, S: int, n_splits: int | None = None):
    """q [Hq, D] (f64); Kc/Vc [Hkv, S_max, D] bf16 bits of one sequence; keys 0..S-1."""
    q = _f64(q)
    Kc, Vc = _u16(Kc), _u16(Vc)
    Hq, D = q.shape
    Hkv, S_max, D2 = Kc.shape
    assert D2 == D and Vc.shape == Kc.shape
    o = np.empty((Hq, D))
    if n_splits is None:
        lib().orc_attention(q.ctypes.data, Kc.ctypes.data, Vc.ctypes.data, S, Hq, Hkv, D, S_max, o.ctypes.data)
    else:
        lib().orc_attention_splitk(q.ctypes.data, Kc.ctypes.data, Vc.ctypes.data, S, Hq, Hkv, D, S_max, n_splits,
                                   o.ctypes.data)
    return o


def silu(z: float) -> float:
    return float(lib().orc_silu(float(z)))


def glu(Wg, Wu, y):
    Wg, Wu = _u16(Wg), _u16(Wu)
    I, H = Wg.shape
    Y = _f64(y).reshape(-1, H)
    out = np.empty((Y.shape[0], I))
    for b in range(Y.shape[0]):
        yb = np.ascontiguousarray(Y[b])
        lib().orc_glu(Wg.ctypes.data, Wu.ctypes.data, yb.ctypes.data, I, H, out[b].ctypes.data)
    return out.reshape(np.shape(y)[:-1] + (I,))


def argmax(x) -> int:
    x = _f64(x)
    return int(lib().orc_argmax(x.ctypes.data, x.size))


def head(r, final_norm, lm_head, eps: float):
    """Final norm + logits + greedy token of one sequence: (token, logits)."""
    r = _f64(r)
    lm_head = _u16(lm_head)
    V, H = lm_head.shape
    logits = np.empty(V)
    t = lib().orc_head(r.ctypes.data, _u16(final_norm).ctypes.data, lm_head.ctypes.data, H, V, eps,
                       logits.ctypes.data)
    return int(t), logits


# ----------------------------------------------------------------------------- layer / step

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")


def dims(m, S_max: int) -> Dims:
    return Dims(m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate, S_max, m.rms_eps, m.rope_theta)


def layer(m, w: dict, Kc, Vc, p: int, r, taps: bool = False, variant: dict | None = None):
    """One layer of one sequence at position p.  Kc/Vc ([Hkv, S_max, D] bf16, this
    sequence's slice) are updated in place.  Returns (r_new, taps dict or None).

    variant (the gated attention layer): optional keys ``rot_dim`` (rotary dims
    per head), ``q_norm`` / ``k_norm`` (per-head RMSNorm gains [D], bf16 bits)
    and ``wgate`` (output-gate projection [Hq*D, H], bf16 bits)."""
    Kc, Vc = _u16(Kc), _u16(Vc)
    d = dims(m, Kc.shape[1])
    r = _f64(r).copy()
    t = None
    tp = None
    if taps:
        H, Hq, Hkv, D, I = m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate
        t = {"y_attn": np.empty(H), "q": np.empty(Hq * D), "k": np.empty(Hkv * D), "v": np.empty(Hkv * D),
             "o": np.empty(Hq * D), "y_mlp": np.empty(H), "h": np.empty(I)}
        tp = Taps(*[t[n].ctypes.data for n in ("y_attn", "q", "k", "v", "o", "y_mlp", "h")])
    ws = [_u16(w[k]) for k in LAYER_KEYS]
    if variant is None:
        lib().orc_layer(ctypes.byref(d), *[a.ctypes.data for a in ws], Kc.ctypes.data, Vc.ctypes.data, int(p),
                        r.ctypes.data, ctypes.byref(tp) if tp is not None else None)
        return r, t
    keep = {k: _u16(variant[k]) for k in ("q_norm", "k_norm", "wgate") if variant.get(k) is not None}
    var = AttnVariant(int(variant.get("rot_dim", 0)), *[keep[k].ctypes.data if k in keep else None
                                                        for k in ("q_norm", "k_norm", "wgate")])
    lib().orc_layer_ex(ctypes.byref(d), ctypes.byref(var), *[a.ctypes.data for a in ws], Kc.ctypes.data,
                       Vc.ctypes.data, int(p), r.ctypes.data, ctypes.byref(tp) if tp is not None else None)
    return r, t


class Model:
    """Host-side model for the oracle: lists of bf16 weight arrays and per-sequence caches.

    layers: list of dicts (LAYER_KEYS -> uint16 arrays); kcache/vcache: per layer
    arrays [B, Hkv, S_max, D] (uint16), owned and updated by the oracle only;
    variants: None, or one gated-attention dict per layer (see ``layer``).
    """

    def __init__(self, m, layers, embed, final_norm, lm_head, kcache, vcache, variants=None):
        self.m = m
        self.layers = layers
        self.embed = embed
        self.final_norm = final_norm
        self.lm_head = lm_head
        self.kcache = kcache
        self.vcache = vcache
        self._wptr = (ctypes.c_void_p * (9 * len(layers)))(
            *[_u16(l[k]).ctypes.data for l in layers for k in LAYER_KEYS])
        self._var = None
        if variants is not None:
            assert len(variants) == len(layers)
            self._keep = [{k: _u16(v[k]) for k in ("q_norm", "k_norm", "wgate") if v.get(k) is not None}
                          for v in variants]
            self._var = (AttnVariant * len(layers))(
                *[AttnVariant(int(v.get("rot_dim", 0)), *[kp[k].ctypes.data if k in kp else None
                                                          for k in ("q_norm", "k_norm", "wgate")])
                  for v, kp in zip(variants, self._keep)])

    def step(self, b: int, p: int, token: int | None = None, x_in=None):
        """One decode step of sequence b at position p.  Returns (token, logits, r_final)."""
        m = self.m
        L = len(self.layers)
        S_max = self.kcache[0].shape[2]
        d = dims(m, S_max)
        kc = (ctypes.c_void_p * L)(*[self.kcache[l][b].ctypes.data for l in range(L)])
        vc = (ctypes.c_void_p * L)(*[self.vcache[l][b].ctypes.data for l in range(L)])
        for l in range(L):
            assert self.kcache[l][b].flags.c_contiguous
        r_out = np.empty(m.hidden)
        has_head = self.lm_head is not None
        logits = np.empty(m.vocab) if has_head else None
        x = None if x_in is None else _f64(x_in)
        tok = lib().orc_step_ex(ctypes.byref(d), L, self._wptr, self._var, kc, vc,
                                None if self.embed is None else self.embed.ctypes.data,
                                _ptr(x), -1 if token is None else int(token), int(p),
                                None if self.final_norm is None else self.final_norm.ctypes.data,
                                self.lm_head.ctypes.data if has_head else None, m.vocab,
                                _ptr(logits), r_out.ctypes.data)
        return int(tok), logits, r_out


# ----------------------------------------------------------------------------- token selection

def select_token(logits, prev=None, penalty: float = 1.0, temperature: float = 0.0, top_k: int = 0,
                 top_p: float = 1.0, u: float = 0.0):
    """Token chosen from one float32 logits row (repetition penalty, temperature,
    top-k, top-p, then the draw ``u`` in [0, 1)); ``temperature == 0`` is greedy.

    Returns ``(token, margin_p, margin_u)``: the relative distances of the
    top-p cut and of ``u * M`` from the nearest cumulative boundary.
    """
    z = np.ascontiguousarray(logits, dtype=np.float32)
    assert z.ndim == 1
    pv = np.ascontiguousarray(prev if prev is not None else np.zeros(0), dtype=np.int32)
    mg = np.empty(2)
    t = lib().orc_select(z.ctypes.data, z.size, pv.ctypes.data if pv.size else None, pv.size, float(penalty),
                         float(temperature), int(top_k), float(top_p), float(u), mg.ctypes.data)
    return int(t), float(mg[0]), float(mg[1])


def top2_margin(logits) -> float:
    s = np.sort(np.asarray(logits, dtype=np.float64))
    return float(s[-1] - s[-2]) if s.size > 1 else float("inf")
