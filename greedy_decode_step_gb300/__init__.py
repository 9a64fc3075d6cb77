"""Python binding of libdec (the C-ABI in include/libdec.h).

Argument marshalling only: every function here checks tensor dtypes and
shapes, passes raw device pointers and sizes to the library and turns a
non-zero status into ``DecError``.  All arithmetic runs in the CUDA kernels of
``libdec.so``; if the library is missing, every call raises.

PyTorch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdec.so")

DEC_OK, DEC_EINVAL, DEC_ECAPACITY, DEC_ECUDA, DEC_EUNSUPPORTED, DEC_EDEVICE = range(6)
_NAMES = {1: "DEC_EINVAL", 2: "DEC_ECAPACITY", 3: "DEC_ECUDA", 4: "DEC_EUNSUPPORTED", 5: "DEC_EDEVICE"}

_lib = None


class DecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_NAMES.get(code, code)}: {msg}")
        self.code = code


class DecLayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")] + \
               [("rot_dim", ctypes.c_int), ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p),
                ("w_gate", ctypes.c_void_p)]


class DecModel(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("intermediate", ctypes.c_int),
                ("vocab", ctypes.c_int), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("layers", ctypes.POINTER(DecLayerWeights))]


class DecState(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("max_seq", ctypes.c_int),
                ("k_cache", ctypes.POINTER(ctypes.c_void_p)), ("v_cache", ctypes.POINTER(ctypes.c_void_p)),
                ("pos", ctypes.c_void_p), ("token", ctypes.c_void_p), ("residual", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("internal", ctypes.c_void_p)]


_P, _I, _F, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGNATURES = {
    "dec_last_error": (ctypes.c_char_p, []),
    "dec_version": (ctypes.c_char_p, []),
    "dec_device_error": (_I, [ctypes.POINTER(ctypes.c_uint32), _I]),
    "dec_add_rmsnorm": (_I, [_P, _P, _P, _P, _I, _I, _F, _P]),
    "dec_qkv_gemv_rope": (_I, [_P, _P, _P, _P, _P, _F, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "dec_attn_workspace_size": (_S, [_I, _I, _I, _I, _I, _I]),
    "dec_gqa_decode_attn": (_I, [_P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _I, _I, _P]),
    "dec_gqa_decode_attn_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "dec_glu_gemv": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "dec_down_gemv": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "dec_lmhead_workspace_size": (_S, [_I]),
    "dec_lmhead_argmax": (_I, [_P, _P, _F, _P, _P, _P, _P, _S, _I, _I, _I, _P]),
    "dec_select_tokens": (_I, [_P, _P, _I, _F, _F, _I, _F, _P, _P, _I, _I, _P]),
    "dec_state_workspace_size": (_S, [ctypes.POINTER(DecModel), _I, _I]),
    "dec_state_init": (_I, [ctypes.POINTER(DecModel), ctypes.POINTER(DecState), _P]),
    "dec_state_release": (_I, [ctypes.POINTER(DecState)]),
    "dec_state_set_wait": (_I, [ctypes.POINTER(DecModel), ctypes.POINTER(DecState), ctypes.c_ulonglong, _I, _P]),
    "dec_step": (_I, [ctypes.POINTER(DecModel), ctypes.POINTER(DecState), _P]),
    "dec_step_launches": (_I, [ctypes.POINTER(DecModel), ctypes.POINTER(DecState), ctypes.POINTER(_I)]),
    "dec_prefill": (_I, [ctypes.POINTER(DecModel), ctypes.POINTER(DecState), _P, _I, _P]),
    "dec_decode": (_I, [ctypes.POINTER(DecModel), ctypes.POINTER(DecState), _I, _I, _P, ctypes.POINTER(_I), _P]),
    "dec_generate": (_I, [ctypes.POINTER(DecModel), ctypes.POINTER(DecState), _P, _I, _I, _I, _P,
                          ctypes.POINTER(_I), _P]),
}


def build(force: bool = False) -> str:
    """Compile libdec.so for sm_103a in place (nvcc)."""
    return _build.build(force=force)


def lib():
    """The loaded libdec.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdec.so is not built ({LIB_PATH}); run greedy_decode_step_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(rc: int):
    if rc != DEC_OK:
        raise DecError(rc, lib().dec_last_error().decode())


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


_bf16, _f32, _i32 = torch.bfloat16, torch.float32, torch.int32


def version() -> str:
    return lib().dec_version().decode()


def device_error(clear: bool = False) -> int:
    v = ctypes.c_uint32(0)
    _check(lib().dec_device_error(ctypes.byref(v), int(clear)))
    return v.value


# ----------------------------------------------------------------------------- single ops

def dec_add_rmsnorm(x, residual, gamma, out, eps: float, stream=None):
    B, H = residual.shape
    _check(lib().dec_add_rmsnorm(_ptr(x, _f32, "x"), _ptr(residual, _f32, "residual"), _ptr(gamma, _bf16, "gamma"),
                                 _ptr(out, _f32, "out"), B, H, eps, _stream(stream)))


def dec_qkv_gemv_rope(y, Wq, Wk, Wv, pos, rope_theta: float, q_out, k_cache, v_cache, stream=None):
    B, H = y.shape
    Bc, Hkv, S_max, D = k_cache.shape
    Hq = Wq.shape[0] // D
    _check(lib().dec_qkv_gemv_rope(_ptr(y, _f32, "y"), _ptr(Wq, _bf16, "Wq"), _ptr(Wk, _bf16, "Wk"),
                                   _ptr(Wv, _bf16, "Wv"), _ptr(pos, _i32, "pos"), rope_theta,
                                   _ptr(q_out, _f32, "q_out"), _ptr(k_cache, _bf16, "k_cache"),
                                   _ptr(v_cache, _bf16, "v_cache"), B, H, Hq, Hkv, D, S_max, _stream(stream)))


def attn_workspace_size(B, Hq, Hkv, D, S_max, num_splits=0) -> int:
    return int(lib().dec_attn_workspace_size(B, Hq, Hkv, D, S_max, num_splits))


def dec_gqa_decode_attn(q, k_cache, v_cache, pos, o, ws=None, num_splits: int = 0, stream=None):
    B, Hq, D = q.shape
    _, Hkv, S_max, _ = k_cache.shape
    need = attn_workspace_size(B, Hq, Hkv, D, S_max, num_splits)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib().dec_gqa_decode_attn(_ptr(q, _f32, "q"), _ptr(k_cache, _bf16, "k_cache"),
                                     _ptr(v_cache, _bf16, "v_cache"), _ptr(pos, _i32, "pos"), _ptr(o, _f32, "o"),
                                     _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), B, Hq, Hkv, D, S_max,
                                     num_splits, _stream(stream)))
    return ws


def dec_gqa_decode_attn_noalloc(q, k_cache, v_cache, pos, o, num_splits: int = 0, stream=None):
    """dec_gqa_decode_attn on the library's built-in scratch: for callers that
    cannot provide (or allocate) a workspace.  Calls that may overlap on the
    GPU share that scratch and must be serialised by the caller."""
    B, Hq, D = q.shape
    _, Hkv, S_max, _ = k_cache.shape
    _check(lib().dec_gqa_decode_attn_noalloc(_ptr(q, _f32, "q"), _ptr(k_cache, _bf16, "k_cache"),
                                             _ptr(v_cache, _bf16, "v_cache"), _ptr(pos, _i32, "pos"),
                                             _ptr(o, _f32, "o"), B, Hq, Hkv, D, S_max, num_splits, _stream(stream)))


def dec_glu_gemv(y, Wg, Wu, h, stream=None):
    B, H = y.shape
    I = Wg.shape[0]
    _check(lib().dec_glu_gemv(_ptr(y, _f32, "y"), _ptr(Wg, _bf16, "Wg"), _ptr(Wu, _bf16, "Wu"), _ptr(h, _f32, "h"),
                              B, H, I, _stream(stream)))


def dec_down_gemv(x, W, residual, stream=None):
    B, N_in = x.shape
    N_out = W.shape[0]
    _check(lib().dec_down_gemv(_ptr(x, _f32, "x"), _ptr(W, _bf16, "W"), _ptr(residual, _f32, "residual"),
                               B, N_in, N_out, _stream(stream)))


def dec_lmhead_argmax(residual, final_norm, eps: float, W_lm, token_out, logits_out=None, ws=None, stream=None):
    B, H = residual.shape
    V = W_lm.shape[0]
    if ws is None:
        ws = torch.empty(int(lib().dec_lmhead_workspace_size(B)), dtype=torch.uint8, device=residual.device)
    _check(lib().dec_lmhead_argmax(_ptr(residual, _f32, "residual"), _ptr(final_norm, _bf16, "final_norm"), eps,
                                   _ptr(W_lm, _bf16, "W_lm"), _ptr(token_out, _i32, "token_out"),
                                   _ptr(logits_out, _f32, "logits_out"), _ptr(ws, None, "ws"),
                                   ws.numel() * ws.element_size(), B, H, V, _stream(stream)))


def dec_select_tokens(logits, token_out, u=None, prev_tokens=None, repetition_penalty: float = 1.0,
                      temperature: float = 0.0, top_k: int = 0, top_p: float = 1.0, stream=None):
    """Token per row of fp32 ``logits`` [B, V]: repetition penalty over ``prev_tokens``
    (int32 [B, n_prev]), then greedy (``temperature == 0``) or a draw by ``u``
    (fp32 [B] in [0, 1)) from the top-k / top-p filtered softmax."""
    B, V = logits.shape
    n_prev = 0 if prev_tokens is None else prev_tokens.shape[1]
    _check(lib().dec_select_tokens(_ptr(logits, _f32, "logits"), _ptr(prev_tokens, _i32, "prev_tokens"), n_prev,
                                   repetition_penalty, temperature, top_k, top_p, _ptr(u, _f32, "u"),
                                   _ptr(token_out, _i32, "token_out"), B, V, _stream(stream)))


# ----------------------------------------------------------------------------- model / state

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")


class Model:
    """Device weights of a dense GQA decoder wrapped in a ``dec_model``.

    layers: list of dicts with LAYER_KEYS -> bf16 CUDA tensors; a gated-attention
    layer adds any of "rot_dim" (int), "q_norm", "k_norm" ([D] gains) and
    "w_gate" (or "wgate", [Hq*D, H]).
    embed / final_norm / lm_head: bf16 CUDA tensors (lm_head may be embed; any may be None).
    """

    def __init__(self, n_layers, hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab, rms_eps, rope_theta,
                 layers, embed=None, final_norm=None, lm_head=None):
        self.layers = layers
        self.embed, self.final_norm, self.lm_head = embed, final_norm, lm_head
        self._lw = (DecLayerWeights * n_layers)()
        for i, l in enumerate(layers):
            for k in LAYER_KEYS:
                setattr(self._lw[i], k, _ptr(l[k], _bf16, k))
            self._lw[i].rot_dim = int(l.get("rot_dim", 0) or 0)
            for k in ("q_norm", "k_norm", "w_gate"):
                t = l.get(k) if l.get(k) is not None else l.get(k.replace("_", ""))  # "wgate" as well
                setattr(self._lw[i], k, _ptr(t, _bf16, k))
        self.c = DecModel(n_layers, hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab, rms_eps, rope_theta,
                          _ptr(embed, _bf16, "embed"), _ptr(final_norm, _bf16, "final_norm"),
                          _ptr(lm_head, _bf16, "lm_head"), self._lw)

    @property
    def shape(self):
        c = self.c
        return dict(n_layers=c.n_layers, hidden=c.hidden, n_heads=c.n_heads, n_kv_heads=c.n_kv_heads,
                    head_dim=c.head_dim, intermediate=c.intermediate, vocab=c.vocab)


class State:
    """Decode state on the GPU: per-layer KV caches, positions, tokens,
    residual stream and workspace, wrapped in a ``dec_state``."""

    def __init__(self, model: Model, batch: int, max_seq: int, device=None, k_cache=None, v_cache=None):
        c = model.c
        dev = torch.device(device or "cuda")
        self.batch, self.max_seq = batch, max_seq
        shp = (batch, c.n_kv_heads, max_seq, c.head_dim)
        self.k_cache = k_cache if k_cache is not None else [torch.zeros(shp, dtype=_bf16, device=dev)
                                                            for _ in range(c.n_layers)]
        self.v_cache = v_cache if v_cache is not None else [torch.zeros(shp, dtype=_bf16, device=dev)
                                                            for _ in range(c.n_layers)]
        self.pos = torch.zeros(batch, dtype=_i32, device=dev)
        self.token = torch.zeros(batch, dtype=_i32, device=dev)
        self.residual = torch.zeros(batch, c.hidden, dtype=_f32, device=dev)
        nbytes = int(lib().dec_state_workspace_size(ctypes.byref(c), batch, max_seq))
        if nbytes == 0:
            raise DecError(DEC_EINVAL, "dec_state_workspace_size rejected the model/state sizes")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self._kc = (ctypes.c_void_p * c.n_layers)(*[_ptr(t, _bf16, "k_cache") for t in self.k_cache])
        self._vc = (ctypes.c_void_p * c.n_layers)(*[_ptr(t, _bf16, "v_cache") for t in self.v_cache])
        self.c = DecState(batch, max_seq, self._kc, self._vc, _ptr(self.pos), _ptr(self.token), _ptr(self.residual),
                          _ptr(self.workspace), nbytes, None)
        self.model = model

    def init(self, stream=None):
        _check(lib().dec_state_init(ctypes.byref(self.model.c), ctypes.byref(self.c), _stream(stream)))
        return self

    def release(self):
        if self.c.internal:
            _check(lib().dec_state_release(ctypes.byref(self.c)))

    def __del__(self):
        try:
            if _lib is not None and self.c.internal:
                _lib.dec_state_release(ctypes.byref(self.c))
        except Exception:
            pass


def dec_step(model: Model, state: State, stream=None):
    _check(lib().dec_step(ctypes.byref(model.c), ctypes.byref(state.c), _stream(stream)))


def dec_step_launches(model: Model, state: State) -> int:
    """Kernel launches one dec_step makes for this model and state (1: the persistent step kernel)."""
    n = ctypes.c_int(0)
    _check(lib().dec_step_launches(ctypes.byref(model.c), ctypes.byref(state.c), ctypes.byref(n)))
    return n.value


def dec_prefill(model: Model, state: State, prompt, stream=None):
    B, P = prompt.shape
    _check(lib().dec_prefill(ctypes.byref(model.c), ctypes.byref(state.c), _ptr(prompt, _i32, "prompt"), P,
                             _stream(stream)))


def _check_out(out_tokens, state: State, n_steps: int):
    """out_tokens must hold the packed [B][n_steps] int32 block the library
    writes (row b at offset b * n_steps): contiguous, at least B * n_steps
    elements."""
    if out_tokens is None:
        return
    if out_tokens.dtype != _i32 or not out_tokens.is_contiguous():
        raise DecError(DEC_EINVAL, "out_tokens must be a contiguous int32 tensor")
    if out_tokens.numel() < state.batch * n_steps:
        raise DecError(DEC_EINVAL, f"out_tokens holds {out_tokens.numel()} elements; the [B][n_steps] block "
                                   f"needs {state.batch * n_steps}")


def dec_state_set_wait(model: Model, state: State, limit_ns: int = 0, hold: bool = False, stream=None):
    """Limit (ns, 0 = default) of the step kernel's waits for other CTAs; ``hold``
    adds a wait nothing ends, to exercise the bounded-wait path."""
    _check(lib().dec_state_set_wait(ctypes.byref(model.c), ctypes.byref(state.c), int(limit_ns), int(bool(hold)),
                                    _stream(stream)))


def dec_decode(model: Model, state: State, n_steps: int, eos_id: int, out_tokens=None, stream=None) -> int:
    _check_out(out_tokens, state, n_steps)
    done = ctypes.c_int(0)
    _check(lib().dec_decode(ctypes.byref(model.c), ctypes.byref(state.c), n_steps, eos_id,
                            _ptr(out_tokens, _i32, "out_tokens"), ctypes.byref(done), _stream(stream)))
    return done.value


def dec_generate(model: Model, state: State, prompt, n_steps: int, eos_id: int, out_tokens, stream=None) -> int:
    _check_out(out_tokens, state, n_steps)
    B, P = prompt.shape
    done = ctypes.c_int(0)
    _check(lib().dec_generate(ctypes.byref(model.c), ctypes.byref(state.c), _ptr(prompt, _i32, "prompt"), P,
                              n_steps, eos_id, _ptr(out_tokens, _i32, "out_tokens"), ctypes.byref(done),
                              _stream(stream)))
    return done.value
