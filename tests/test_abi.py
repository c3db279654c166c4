"""The C-ABI library builds, loads and exports every entry point of
include/mk.h; host-only argument checks. No GPU needed (no compute calls)."""
import ctypes

import pytest

from decode_megakernel_llama_gb300 import _lib
from decode_megakernel_llama_gb300.build import build
from decode_megakernel_llama_gb300.configs import LLAMA_1B, TINY, ModelShape


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = _lib.declared_symbols()
    expected = {"mk_create", "mk_decode_step", "mk_decode_step_dev", "mk_decode_step_host",
                "mk_decode_step_unfused", "mk_get_status", "mk_set_wait_timeout", "mk_set_trace",
                "mk_read_trace", "mk_plan_size", "mk_plan_inspect", "mk_destroy", "mk_last_error"}
    assert expected <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_destroy_null_and_last_error(lib):
    lib.mk_destroy(None)
    assert isinstance(lib.mk_last_error(), bytes)


def test_null_handle_calls_are_rejected(lib):
    tok = ctypes.c_int32(0)
    assert lib.mk_decode_step(None, 0, 0, None, ctypes.addressof(tok), None) == _lib.MK_ERR_INVALID_ARG
    assert b"handle" in lib.mk_last_error()
    assert lib.mk_get_status(None) == _lib.MK_ERR_INVALID_ARG
    assert lib.mk_create(None, None, None, None) == _lib.MK_ERR_INVALID_ARG


@pytest.mark.parametrize("bad,code", [
    (dict(head_dim=96), _lib.MK_ERR_UNSUPPORTED),
    (dict(n_kv_heads=3), _lib.MK_ERR_INVALID_ARG),
    (dict(d_model=2000), _lib.MK_ERR_UNSUPPORTED),
    (dict(ffn_dim=100), _lib.MK_ERR_UNSUPPORTED),
    (dict(n_layers=0), _lib.MK_ERR_INVALID_ARG),
    (dict(vocab=0), _lib.MK_ERR_INVALID_ARG),
])
def test_plan_rejects_unsupported_configs(lib, bad, code):
    import dataclasses
    shape = dataclasses.replace(LLAMA_1B, **bad)
    cfg = _lib.make_config(shape, 256)
    qlen = (ctypes.c_int32 * 152)()
    n = ctypes.c_int32()
    assert lib.mk_plan_inspect(ctypes.byref(cfg), 152, None, 0, qlen, ctypes.byref(n)) == code
    assert lib.mk_last_error()


def test_plan_inspect_cap_too_small(lib):
    cfg = _lib.make_config(TINY, 40)
    qlen = (ctypes.c_int32 * 4)()
    buf = (ctypes.c_int32 * 16)()
    n = ctypes.c_int32()
    assert lib.mk_plan_inspect(ctypes.byref(cfg), 4, buf, 1, qlen, ctypes.byref(n)) == _lib.MK_ERR_INVALID_ARG


def test_w2_packing_layout_and_round_trip():
    # element 16w + 4j + i sits in bits [8i + 2j, 8i + 2j + 2) of word w as q + 1
    import numpy as np
    q = np.zeros((2, 32), dtype=np.int8)
    q[0, 5] = 1     # w 0, j 1, i 1 -> bits 10..11 = 2
    q[1, 16 + 14] = -1  # w 1, j 3, i 2 -> bits 22..23 = 0
    p = _lib.w2_pack(q)
    assert p[0, 0] == (0x55555555 & ~(3 << 10)) | (2 << 10)
    assert p[0, 1] == 0x55555555
    assert p[1, 1] == 0x55555555 & ~(3 << 22)
    rng = np.random.default_rng(0)
    r = (rng.integers(0, 3, (7, 2048)) - 1).astype(np.int8)
    assert (_lib.w2_unpack(_lib.w2_pack(r), 2048) == r).all()
    bad = r.copy()
    bad[3, 100] = 2
    with pytest.raises(_lib.MKError):
        _lib.w2_pack(bad)
