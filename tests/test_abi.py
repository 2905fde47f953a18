"""Host-side checks of the C-ABI library; none of them needs a GPU."""

import ctypes

import pytest

from head_latent_attention_26_b300 import build, mla


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mla.load()


def test_library_exports_every_declared_symbol(lib):
    names = mla.header_symbols()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert missing == []
    # the binding declares a signature for every symbol of the header
    assert sorted(mla._SIGS) == names


def test_status_strings(lib):
    assert lib.mla_status_string(0) == b"ok"
    assert b"workspace" in lib.mla_status_string(3)
    assert lib.mla_status_string(99) == b"unknown status"


def test_null_handle_is_rejected_without_launching(lib):
    P = ctypes.c_void_p
    s = P(0)
    assert lib.mla_q_proj(None, None, None, None, None, 1, None, None, None, 0, s) == 1
    assert lib.mla_cache_append(None, None, None, None, None, 1, None, 1, 1, None, 1, s) == 1
    assert lib.mla_absorb_q(None, None, None, None, 1, None, None, s) == 1
    assert lib.mla_decode(None, None, None, 1, None, 1, None, None, 1, 1, 0, None, 0, None, None, s) == 1
    assert lib.mla_out(None, None, None, None, 1, None, None, 0, s) == 1
    assert lib.mla_check_device_status(None, s) == 1
    assert lib.mla_set_wait_limit(None, 5) == 1
    assert lib.mla_decode_workspace_bytes(None, 4, 0) == 0
    assert lib.mla_num_sms(None) == 0


def test_create_rejects_bad_dims(lib):
    out = ctypes.c_void_p()
    bad = mla._Dims(128, 128, 63, 512, 1536, 5120, 64, 10000.0, 0.07, 0)  # odd d_hr
    assert lib.mla_create(ctypes.byref(bad), 100, ctypes.byref(out)) == 1
    ok_dims = mla._Dims(128, 128, 64, 512, 1536, 5120, 64, 10000.0, 0.07, 0)
    assert lib.mla_create(ctypes.byref(ok_dims), 0, ctypes.byref(out)) == 1  # max_pos < 1
    big = mla._Dims(4, 8, 4, 1024, 24, 32, 64, 10000.0, 0.07, 1)  # d_c beyond the generic path
    assert lib.mla_create(ctypes.byref(big), 10, ctypes.byref(out)) == 2
