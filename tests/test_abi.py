"""The C-ABI library loads without a GPU, exports every declared entry point and
rejects bad host arguments before touching the device."""
import ctypes
import os
import re

import pytest

import head_latent_attention_25_b300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", src)
    return names


def test_library_exports_every_declared_symbol():
    lib = mla.load()
    names = declared_symbols()
    assert set(names) >= set(mla.EXPORTED) and len(names) == len(set(names))
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings():
    assert mla.status_string(mla.MLA_OK) == "ok"
    for s in range(1, 5):
        assert mla.status_string(s) and mla.status_string(s) != "unknown status"


def _dims(**kw):
    base = dict(n_heads=4, d_h=16, d_c=32, d_r=8, hidden=64)
    base.update(kw)
    return mla.make_dims(**base)


@pytest.mark.parametrize("bad", [dict(d_c=31), dict(d_r=7), dict(n_heads=0), dict(d_h=0),
                                 dict(rope_base=0.0), dict(softmax_scale=-1.0)])
def test_bad_dims_rejected_on_host(bad):
    d = _dims(**bad)
    lib = mla.load()
    fake = 256  # never dereferenced: the checks fail first
    st = lib.mla_cache_append(ctypes.byref(d), 0, 1, 1, fake, fake, fake, fake, fake, fake, fake, 64, None, 0, fake, None)
    assert st == mla.MLA_ERR_INVALID_ARG
    st = lib.mla_project_out(ctypes.byref(d), 0, 1, fake, fake, fake, fake, None)
    assert st == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_workspace_size(ctypes.byref(d), 0, 1, 16, 4) == 0


def test_null_pointers_rejected_on_host():
    d = _dims()
    lib = mla.load()
    fake = 256
    assert lib.mla_cache_append(ctypes.byref(d), 0, 1, 1, None, fake, fake, fake, fake, fake, fake, 64, None, 0, fake,
                                None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_absorbed(ctypes.byref(d), 0, 1, fake, fake, fake, None, 64, fake, fake, 8, 1, fake,
                                   1 << 20, fake, None, fake, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_absorbed(ctypes.byref(d), 0, 1, fake, fake, fake, fake, 0, fake, fake, 8, 1, fake,
                                   1 << 20, fake, None, fake, None) == mla.MLA_ERR_INVALID_ARG
    for fn in (lib.mla_decode_prepare, lib.mla_decode_attend):
        assert fn(ctypes.byref(d), 0, 1, fake, fake, fake, None, 64, fake, fake, 8, 1, fake,
                  1 << 20, fake, None, fake, None) == mla.MLA_ERR_INVALID_ARG
        assert fn(ctypes.byref(d), 0, 1, fake, fake, fake, fake, 64, fake, fake, 8, 1, None,
                  1 << 20, fake, None, fake, None) == mla.MLA_ERR_WORKSPACE
    assert lib.mla_project_query(ctypes.byref(d), 0, 1, 64, fake, fake, None, fake, fake, fake,
                                 None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_project_query(ctypes.byref(d), 0, 1, 64, fake, fake, fake, fake, fake, None,
                                 None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_project_query_latent(ctypes.byref(d), 0, 1, 32, fake, None, None, 0, fake, fake,
                                        None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_query_latent_workspace_size(ctypes.byref(d), 0, 1, 32) == 0
    assert lib.mla_cache_append(None, 0, 1, 1, fake, fake, fake, fake, fake, fake, fake, 64, None, 0, fake,
                                None) == mla.MLA_ERR_INVALID_ARG


def test_misaligned_cache_and_bad_dtype_rejected():
    d = _dims()
    lib = mla.load()
    fake = 256
    assert lib.mla_cache_append(ctypes.byref(d), 0, 1, 1, fake, fake, fake, fake, fake, fake, fake + 4, 64, None, 0, fake,
                                None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_cache_append(ctypes.byref(d), 7, 1, 1, fake, fake, fake, fake, fake, fake, fake, 64, None, 0, fake,
                                None) == mla.MLA_ERR_INVALID_ARG
    # bf16 rows of 3 + 3 elements are 12 bytes: not a multiple of 16
    d2 = _dims(d_c=4, d_r=2)
    assert lib.mla_cache_append(ctypes.byref(d2), 1, 1, 1, fake, fake, fake, fake, fake, fake, fake, 64, None, 0, fake,
                                None) == mla.MLA_ERR_INVALID_ARG


def test_workspace_size_explicit_splits():
    d = _dims()
    a = mla.mla_decode_workspace_size(d, mla.MLA_F32, 1, 129, 1)
    b = mla.mla_decode_workspace_size(d, mla.MLA_F32, 1, 129, 7)
    assert 0 < a < b and a % 256 == 0 and b % 256 == 0
    assert mla.mla_decode_workspace_size(d, mla.MLA_F32, 0, 129, 1) == 0


def test_cache_layout_checks_on_host():
    """Layouts are checked before anything is enqueued: unsupported shapes, misaligned or
    too-short strides, block sizes that are not whole tiles."""
    lib = mla.load()
    fake = 1 << 12                              # 16-byte aligned, never dereferenced
    v3 = mla.make_dims(128, 128, 512, 64, 7168)
    good = mla.MlaCacheLayout(fake, fake, 512, 64, 1 << 16, None, 0, 0)
    bad_stride = mla.MlaCacheLayout(fake, fake, 500, 64, 1 << 16, None, 0, 0)
    bad_block = mla.MlaCacheLayout(fake, None, 576, 0, 1 << 16, fake, 96, 8)
    args = lambda lay: (ctypes.byref(v3), mla.MLA_BF16, 4, fake, fake, fake, ctypes.byref(lay), fake, fake, 4096,
                        0, fake, 1 << 30, fake, None, fake, None)
    assert lib.mla_decode_absorbed_ex(*args(bad_stride)) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_absorbed_ex(*args(bad_block)) == mla.MLA_ERR_INVALID_ARG
    small = mla.make_dims(4, 16, 32, 8, 64)
    assert lib.mla_decode_absorbed_ex(ctypes.byref(small), mla.MLA_BF16, 4, fake, fake, fake, ctypes.byref(good),
                                      fake, fake, 16, 0, fake, 1 << 30, fake, None, fake, None) == mla.MLA_ERR_UNSUPPORTED
    assert lib.mla_cache_append_ex(ctypes.byref(small), mla.MLA_BF16, 1, 1, fake, fake, fake, ctypes.byref(good),
                                   fake, fake, fake, fake, 1 << 20, fake, None) == mla.MLA_ERR_UNSUPPORTED
