"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/sub_api.h declares, and rejects bad arguments
before touching the device."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "sub_api.h")).read()
    decl = r"^\s*(?:int32_t|const char\s*\*)\s*(sub_[a-z0-9_]+)\s*\("
    return sorted(set(re.findall(decl, src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import substitute_speculative_decoding_gb300 as s
    return s


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "sub_generate" in names and "sub_w4_gemm" in names
    for n in names:
        assert hasattr(lib._lib, n), n
    assert set(names) == set(lib.EXPORTED)


def test_version(lib):
    assert "sm_103a" in lib.version()


def test_bad_arguments_are_rejected_on_the_host(lib):
    s = lib
    # group != 64 -> unsupported, before any CUDA call
    r = s._w4_pack(None, 16, 64, 32, None, None, None, None)
    assert r == s.SUB_EUNSUPPORTED
    assert b"group" in s._lib.sub_last_error()
    # null pointers / bad sizes -> EINVAL
    assert s._w4_pack(None, 16, 64, 64, None, None, None, None) == s.SUB_EINVAL
    assert s._w4_pack(None, 16, 60, 64, None, None, None, None) == s.SUB_EINVAL
    assert s._bf16_gemm(None, 4, None, 16, 64, None, None) == s.SUB_EINVAL
    assert s._model_create(None, None) == s.SUB_EINVAL
    kv = s.KVCache()
    assert s._kv_compact(C.byref(kv), 0, None, None, 4, None) == s.SUB_EINVAL
    cfg = s.DecodeCfg(4, 2, 0.2, 0, 1.0, 0, 0)
    assert s._generate(None, None, 0, 0, C.byref(cfg), None, None) == s.SUB_EINVAL


def test_model_desc_validation(lib):
    s = lib
    d = s.ModelDesc()
    d.n_layers = 2
    d.hidden = 256
    d.head_dim = 96            # unsupported head size
    d.n_heads_q, d.n_heads_kv = 4, 2
    layers = (s.LayerDesc * 2)()
    d.layers = layers
    h = C.c_void_p()
    assert s._model_create(C.byref(d), C.byref(h)) == s.SUB_EINVAL
    assert b"head_dim" in s._lib.sub_last_error()
