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
    # 2/3/4-bit packing: the code width and the HQQ iteration count are checked first
    assert s._wq_pack(None, 16, 64, 64, 5, None, None, None, None) == s.SUB_EINVAL
    assert s._wq_pack(None, 16, 64, 64, 1, None, None, None, None) == s.SUB_EINVAL
    assert s._wq_pack(None, 16, 64, 32, 2, None, None, None, None) == s.SUB_EUNSUPPORTED
    assert s._wq_pack_hqq(None, 16, 64, 64, 3, 0, None, None, None, None) == s.SUB_EINVAL
    assert s._wq_dequant(None, None, None, 16, 64, 64, 6, None, None) == s.SUB_EINVAL
    assert s._wq_gemm(None, 1, None, None, None, 16, 64, 64, 2, None, None) == s.SUB_EINVAL


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


def test_struct_layouts_match_the_header(lib, tmp_path):
    """Every ctypes mirror of a struct in include/sub_api.h has the C layout:
    a small C program compiled against the header prints sizeof and the
    offset of each field, and the binding must agree field by field."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    s = lib
    mirrors = {"sub_kv_cache": s.KVCache, "sub_tree": s.Tree, "sub_w4": s.W4,
               "sub_layer_desc": s.LayerDesc, "sub_model_desc": s.ModelDesc,
               "sub_decode_cfg": s.DecodeCfg, "sub_stats": s.Stats}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "sub_api.h"',
             "int main(void) {"]
    for cname, py in mirrors.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for f in py._fields_:
            lines.append(f'  printf("{cname} {f[0]} %zu\\n", offsetof({cname}, {f[0]}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run([gcc, "-std=c11", "-I", inc, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {}
    for ln in out.splitlines():
        cname, field, val = ln.split()
        got[(cname, field)] = int(val)
    for cname, py in mirrors.items():
        assert got[(cname, "size")] == C.sizeof(py), cname
        for f in py._fields_:
            assert got[(cname, f[0])] == getattr(py, f[0]).offset, (cname, f[0])
