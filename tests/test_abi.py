"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every entry point that include/libdec.h declares, and rejects bad arguments
with an error code and a message before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "libdec.h")


@pytest.fixture(scope="module")
def gd():
    import greedy_decode_step_gb300 as gd
    gd.build()
    return gd


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(dec_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("dec_add_rmsnorm", "dec_qkv_gemv_rope", "dec_gqa_decode_attn", "dec_glu_gemv", "dec_down_gemv",
              "dec_lmhead_argmax", "dec_step", "dec_generate"):
        assert n in names


def test_library_exports_every_declared_symbol(gd):
    L = ctypes.CDLL(gd.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_version(gd):
    assert "sm_103a" in gd.version()


def _call(gd, name, *args):
    fn = getattr(gd.lib(), name)
    return fn(*args), gd.lib().dec_last_error().decode()


def test_null_and_misaligned_pointers_are_rejected(gd):
    rc, msg = _call(gd, "dec_add_rmsnorm", None, None, None, None, 1, 256, 1e-6, None)
    assert rc == gd.DEC_EINVAL and "residual" in msg
    rc, msg = _call(gd, "dec_add_rmsnorm", None, 0x1004, 0x2000, 0x3000, 1, 256, 1e-6, None)
    assert rc == gd.DEC_EINVAL and "aligned" in msg
    rc, msg = _call(gd, "dec_glu_gemv", 0x1000, None, 0x2000, 0x3000, 1, 256, 704, None)
    assert rc == gd.DEC_EINVAL and "Wg" in msg
    rc, msg = _call(gd, "dec_down_gemv", 0x1000, 0x2000, None, 1, 256, 256, None)
    assert rc == gd.DEC_EINVAL


def test_shapes_outside_the_supported_set(gd):
    p = 0x1000
    rc, msg = _call(gd, "dec_add_rmsnorm", None, p, p, p, 0, 256, 1e-6, None)
    assert rc == gd.DEC_EUNSUPPORTED and "batch" in msg
    rc, _ = _call(gd, "dec_add_rmsnorm", None, p, p, p, 17, 256, 1e-6, None)
    assert rc == gd.DEC_EUNSUPPORTED
    rc, msg = _call(gd, "dec_add_rmsnorm", None, p, p, p, 1, 250, 1e-6, None)
    assert rc == gd.DEC_EUNSUPPORTED and "multiple of 8" in msg
    rc, msg = _call(gd, "dec_qkv_gemv_rope", p, p, p, p, p, 1e6, p, p, p, 1, 256, 4, 2, 96, 128, None)
    assert rc == gd.DEC_EUNSUPPORTED and "head_dim" in msg
    rc, msg = _call(gd, "dec_qkv_gemv_rope", p, p, p, p, p, 1e6, p, p, p, 1, 256, 6, 4, 64, 128, None)
    assert rc == gd.DEC_EINVAL and "multiple" in msg
    rc, msg = _call(gd, "dec_gqa_decode_attn", p, p, p, p, p, p, 1 << 20, 1, 34, 2, 64, 128, 0, None)
    assert rc == gd.DEC_EUNSUPPORTED and "Hq/Hkv" in msg
    rc, _ = _call(gd, "dec_add_rmsnorm", None, p, p, p, 1, 256, -1.0, None)
    assert rc == gd.DEC_EINVAL


def test_model_checks_before_any_device_work(gd):
    import ctypes as C
    lw = (gd.DecLayerWeights * 1)()
    m = gd.DecModel(1, 256, 4, 2, 64, 704, 1024, 1e-6, 1e6, None, None, None, lw)
    s = gd.DecState()
    rc = gd.lib().dec_step(C.byref(m), C.byref(s), None)
    assert rc == gd.DEC_EINVAL and "layer 0" in gd.lib().dec_last_error().decode()
    m0 = gd.DecModel(0, 256, 4, 2, 64, 704, 1024, 1e-6, 1e6, None, None, None, lw)
    assert gd.lib().dec_step(C.byref(m0), C.byref(s), None) == gd.DEC_EINVAL


def test_missing_library_fails_loudly(monkeypatch, gd):
    monkeypatch.setattr(gd, "_lib", None)
    monkeypatch.setattr(gd, "LIB_PATH", "/nonexistent/libdec.so")
    with pytest.raises(RuntimeError, match="not built"):
        gd.lib()


def test_token_selection_arguments_are_checked_on_the_host(gd):
    p = 0x1000
    rc, msg = _call(gd, "dec_select_tokens", None, None, 0, 1.0, 0.0, 0, 1.0, None, p, 1, 1024, None)
    assert rc == gd.DEC_EINVAL and "logits" in msg
    rc, msg = _call(gd, "dec_select_tokens", p, None, 0, 1.0, 0.5, 0, 1.5, p, p, 1, 1024, None)
    assert rc == gd.DEC_EINVAL and "top_p" in msg
    rc, msg = _call(gd, "dec_select_tokens", p, None, 0, 1.0, 0.5, 0, 0.0, p, p, 1, 1024, None)
    assert rc == gd.DEC_EINVAL and "top_p" in msg
    rc, msg = _call(gd, "dec_select_tokens", p, None, 3, 1.0, 0.5, 0, 1.0, p, p, 1, 1024, None)
    assert rc == gd.DEC_EINVAL and "prev_tokens" in msg
    rc, msg = _call(gd, "dec_select_tokens", p, None, 0, 1.0, 0.5, 0, 1.0, None, p, 1, 1024, None)
    assert rc == gd.DEC_EINVAL and "u is NULL" in msg
    rc, msg = _call(gd, "dec_select_tokens", p, None, 0, 0.0, 0.5, 0, 1.0, p, p, 1, 1024, None)
    assert rc == gd.DEC_EINVAL and "repetition_penalty" in msg
    rc, msg = _call(gd, "dec_select_tokens", p, None, 0, 1.0, -1.0, 0, 1.0, p, p, 1, 1024, None)
    assert rc == gd.DEC_EINVAL and "temperature" in msg
    rc, msg = _call(gd, "dec_select_tokens", p, None, 0, 1.0, 0.5, -1, 1.0, p, p, 1, 1024, None)
    assert rc == gd.DEC_EINVAL and "top_k" in msg
    rc, msg = _call(gd, "dec_select_tokens", p, None, 0, 1.0, 0.5, 0, 1.0, p, p, 1, 1 << 19, None)
    assert rc == gd.DEC_EUNSUPPORTED and "shared memory" in msg
    rc, msg = _call(gd, "dec_select_tokens", p, None, 0, 1.0, 0.5, 0, 1.0, p, p, 1, 1020, None)
    assert rc == gd.DEC_EUNSUPPORTED and "multiple of 8" in msg
    rc, msg = _call(gd, "dec_select_tokens", p, None, 0, 1.0, 0.5, 0, 1.0, p, p, 0, 1024, None)
    assert rc == gd.DEC_EUNSUPPORTED and "batch" in msg
    # greedy needs no draws
    rc, msg = _call(gd, "dec_select_tokens", p, None, 0, 1.0, 0.0, 0, 1.0, None, None, 1, 1024, None)
    assert rc == gd.DEC_EINVAL and "token_out" in msg
