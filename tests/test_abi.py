"""The C ABI library on the host: it builds, loads without a GPU, exports every
entry point include/injectscale.h declares, and validates arguments before
touching the device.  No compute call is made here."""
import ctypes
import os
import re

import numpy as np
import pytest

from kv_cache_injection_gb300 import _lib, api, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "injectscale.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(is_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    for name in names:
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.is_status_string(code).decode() == name


def test_struct_layouts_match_header():
    assert ctypes.sizeof(_lib.StoreConfig) == 72
    assert ctypes.sizeof(_lib.RopeParams) == 48
    assert ctypes.sizeof(_lib.CacheDesc) == 20
    assert ctypes.sizeof(_lib.StoreInfo) == 64


def _create(**kw):
    base = dict(num_layers=2, num_kv_heads=4, head_dim=64, emb_dim=64, kv_dtype="bf16",
                emb_dtype="f16", max_facts=10, max_tokens=100, max_users=1)
    base.update(kw)
    return api.is_store_create(api.make_config(**base), 0, 0)


@pytest.mark.parametrize("kw,status", [
    (dict(num_layers=0), 1), (dict(emb_dtype="bf16"), 1), (dict(max_facts=0), 1),
    (dict(max_k=2000), 1), (dict(max_queries=5000), 1), (dict(head_dim=96), 8),
    (dict(num_kv_heads=1, head_dim=64), 8), (dict(emb_dim=60), 8), (dict(head_dim=1024), 8),
    (dict(kv_dtype=7), 1), (dict(kv_placement=2), 1), (dict(reserved=3), 1)])
def test_create_rejects_bad_configs_before_the_device(lib, kw, status):
    with pytest.raises(api.ISError) as e:
        _create(**kw)
    assert e.value.status == status


def test_null_handles_are_rejected(lib):
    assert lib.is_store_destroy(None) == 1
    bits = ctypes.c_uint32()
    assert lib.is_get_status(None, None, ctypes.byref(bits)) == 1
    assert lib.is_inject(None, 1, None, None, 1, None, None, None, None, 1, None, None, None,
                         None, None) == 1
    assert lib.is_retrieve_topk(None, 1, None, None, 1, None, None, None) == 1
    assert "NULL" in lib.is_last_error_message().decode()


def test_rope_frequencies_host_side(lib):
    from oracle import rope
    for theta, D, sc in [(1e4, 64, 0), (1e6, 128, 0), (5e5, 128, 1), (5e5, 256, 1)]:
        p = api.make_rope(theta, 0, sc, 8.0, 1.0, 4.0, 8192)
        got = api.is_rope_frequencies(p, D)
        want = rope.inv_freq(D, theta, sc, 8.0, 1.0, 4.0, 8192)
        assert np.allclose(got, want, rtol=1e-14, atol=0)
    with pytest.raises(api.ISError):
        api.is_rope_frequencies(api.make_rope(0.5), 64)
    with pytest.raises(api.ISError):
        api.is_rope_frequencies(api.make_rope(1e4, style=3), 64)


def test_binding_constants_match_the_header():
    """Every integer IS_* constant the binding defines equals the header's #define."""
    text = open(HEADER).read()
    defines = {}
    for name, val in re.findall(r"#define\s+(IS_[A-Z0-9_]+)\s+(\(1 << \d+\)|0x[0-9a-fA-F]+|\d+)u?\b", text):
        m = re.match(r"\(1 << (\d+)\)", val)
        defines[name] = (1 << int(m.group(1))) if m else int(val, 0)
    assert len(defines) >= 8
    checked = 0
    for name, value in defines.items():
        if hasattr(_lib, name):
            assert getattr(_lib, name) == value, name
            checked += 1
    assert checked >= 6


def test_host_call_prepare_checks_before_the_device(lib):
    """is_host_call_prepare refuses a missing store or output slot, and
    is_host_call_run a missing handle, without touching a device."""
    out = ctypes.c_void_p()
    rope = api.make_rope(1e4)
    cache = api.make_cache_desc(16, 1, "bf16")
    buf = np.zeros(4, dtype=np.int32)
    p = buf.ctypes.data
    assert lib.is_host_call_prepare(None, 1, p, p, 1, p, ctypes.byref(rope), p, 1, ctypes.byref(cache), p,
                                    None, None, None, None, ctypes.byref(out)) == 1
    assert out.value is None
    assert lib.is_host_call_prepare(None, 1, p, p, 1, p, ctypes.byref(rope), p, 1, ctypes.byref(cache), p,
                                    None, None, None, None, None) == 1
    assert lib.is_host_call_run(None) == 1
    assert lib.is_host_call_destroy(None) == 0
