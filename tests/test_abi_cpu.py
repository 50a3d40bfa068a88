"""The C-ABI library builds, loads on a machine without a GPU, exports every
function include/oscar.h declares, and answers its host-only calls."""

import ctypes

import pytest

from bit_rotated_kv_oscar_gb300 import abi, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.lib()


def test_every_declared_symbol_is_exported(lib):
    names = abi.header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(abi._SIGS)


def test_version_and_status_strings(lib):
    assert lib.oscar_version() == 1
    assert lib.oscar_status_string(0) == b"ok"
    assert lib.oscar_status_string(-5) == b"unsupported shape"
    assert lib.oscar_status_string(123) == b"unknown status"


def test_config_validation(lib):
    good = abi.make_config(32, 8, 4, 128, 16, 2049)
    assert abi.check_config(good) == 0
    assert abi.check_config(abi.make_config(32, 8, 4, 128, 16, 2049, head_dim=64)) == -5
    assert abi.check_config(abi.make_config(32, 8, 4, 128, 16, 2049, page_size=32)) == -5
    assert abi.check_config(abi.make_config(48, 8, 4, 128, 16, 2049)) == -5   # group of 6
    assert abi.check_config(abi.make_config(30, 8, 4, 128, 16, 2049)) == -1   # not a multiple
    assert abi.check_config(abi.make_config(32, 8, -1, 128, 16, 2049)) == -1
    assert abi.check_config(abi.make_config(32, 8, 4, 0, 16, 2049)) == -1
    assert abi.check_config(abi.make_config(32, 8, 4, 1021, 16, 2049)) == -5  # window too big
    assert lib.oscar_check_config(None) == -1


def test_cache_bytes(lib):
    cfg = abi.make_config(64, 8, 4, 128, 28, 6251)
    pool, win = abi.cache_bytes(cfg, 175000)
    assert pool == 175000 * 8 * 1536
    assert win == 28 * 8 * 2 * 132 * 128 * 2
    with pytest.raises(abi.OscarError):
        abi.cache_bytes(cfg, -1)


def test_null_handles_do_not_crash(lib):
    assert lib.oscar_bind_cache(None, None, 1, None) == -1
    assert lib.oscar_quant_append(None, None, None, None, None, 1, 1, None) == -1
    assert lib.oscar_decode_attn(None, None, None, None, None, 1, None) == -1
    assert lib.oscar_last_error(None) == b"null context"
    lib.oscar_destroy(None)
    out = ctypes.c_void_p()
    assert lib.oscar_create(None, ctypes.byref(out)) == -1 and not out.value
