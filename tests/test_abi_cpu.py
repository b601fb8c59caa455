"""C ABI checks that need no GPU: the library builds, exports every function
declared in include/*.h, and rejects bad arguments before launching."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from flashattention_attention_backward_gb300.build import build
    import flashattention_attention_backward_gb300 as attn

    build()
    return attn


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?(?:long\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text,
                                flags=re.M))
    return sorted(names)


def test_header_declares_entry_points():
    names = _declared()
    for want in ("attn_fwd", "attn_fwd_ref", "attn_bwd_preprocess", "attn_bwd", "attn_bwd_finalize",
                 "attn_device_status", "attn_strerror"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    from flashattention_attention_backward_gb300.build import LIB_PATH

    so = ctypes.CDLL(LIB_PATH)
    for name in _declared():
        assert hasattr(so, name), name


def test_strerror(lib):
    for code in range(0, -9, -1):
        s = lib.attn_strerror(code)
        assert s and s != "unknown error code"
    assert lib.attn_strerror(-100) == "unknown error code"


FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced


def test_bwd_argument_validation(lib):
    a = FAKE
    ok = (a, a, a, a, a, a, a, a, a)
    # null pointer
    assert lib.attn_bwd(0, *ok[1:], 1, 2, 2, 128, 128, 0.1, 1, 0.0, a) == lib.ATTN_ERR_NULL
    assert lib.attn_bwd(*ok, 1, 2, 2, 128, 128, 0.1, 1, 0.0, 0) == lib.ATTN_ERR_NULL
    # bad shapes
    assert lib.attn_bwd(*ok, 1, 3, 2, 128, 128, 0.1, 1, 0.0, a) == lib.ATTN_ERR_SHAPE
    assert lib.attn_bwd(*ok, -1, 2, 2, 128, 128, 0.1, 1, 0.0, a) == lib.ATTN_ERR_SHAPE
    assert lib.attn_bwd(*ok, 1, 2, 0, 128, 128, 0.1, 1, 0.0, a) == lib.ATTN_ERR_SHAPE
    assert lib.attn_bwd(*ok, 1, 2, 2, 128, 128, float("nan"), 1, 0.0, a) == lib.ATTN_ERR_SHAPE
    assert lib.attn_bwd(*ok, 1, 2, 2, 128, 128, 0.0, 1, 0.0, a) == lib.ATTN_ERR_SHAPE
    # unsupported head dim
    assert lib.attn_bwd(*ok, 1, 2, 2, 128, 96, 0.1, 1, 0.0, a) == lib.ATTN_ERR_UNSUPPORTED
    # misaligned pointer
    bad = list(ok)
    bad[0] = a + 8
    assert lib.attn_bwd(*bad, 1, 2, 2, 128, 128, 0.1, 1, 0.0, a) == lib.ATTN_ERR_ALIGN
    # too large
    assert lib.attn_bwd(*ok, 1, 1, 1, 1 << 30, 128, 0.1, 1, 0.0, a) == lib.ATTN_ERR_TOO_LARGE
    # empty problems succeed without touching the device
    assert lib.attn_bwd(*ok, 0, 2, 2, 128, 128, 0.1, 1, 0.0, a) == lib.ATTN_OK
    assert lib.attn_bwd(*ok, 1, 2, 2, 0, 128, 0.1, 1, 0.0, a) == lib.ATTN_OK


def test_other_entry_points_validation(lib):
    a = FAKE
    for fwd in (lib.attn_fwd_ref, lib.attn_fwd):
        assert fwd(0, a, a, a, a, 1, 1, 1, 64, 64, 0.1, 0, 0.0) == lib.ATTN_ERR_NULL
        assert fwd(a, a, a, a, a, 1, 1, 1, 64, 80, 0.1, 0, 0.0) == lib.ATTN_ERR_UNSUPPORTED
        assert fwd(a, a, a, a, a, 1, 4, 3, 64, 64, 0.1, 0, 0.0) == lib.ATTN_ERR_SHAPE
        assert fwd(a, a, a, a + 4, a, 1, 1, 1, 64, 64, 0.1, 0, 0.0) == lib.ATTN_ERR_ALIGN
        assert fwd(a, a, a, a, a, 1, 0, 1, 64, 64, 0.1, 0, 0.0) == lib.ATTN_OK
    # the tensor-core forward takes tau > 0; the fp32 forward any finite nonzero tau
    assert lib.attn_fwd(a, a, a, a, a, 1, 1, 1, 64, 64, -0.1, 0, 0.0) == lib.ATTN_ERR_SHAPE
    assert lib.attn_fwd_local(a, a, a, a, a, 1, 1, 1, 64, 64, -0.1, 0, 0.0, 8, 8) == \
        lib.ATTN_ERR_SHAPE
    assert lib.attn_fwd_ref(a, a, a, a, a, 1, 0, 1, 64, 64, -0.1, 0, 0.0) == lib.ATTN_OK
    for fn in (lib.attn_fwd_local, lib.attn_fwd_ref_local):
        assert fn(0, a, a, a, a, 1, 1, 1, 64, 64, 0.1, 0, 0.0, 8, 8) == lib.ATTN_ERR_NULL
        assert fn(a, a, a, a, a, 1, 1, 1, 64, 96, 0.1, 0, 0.0, 8, 8) == lib.ATTN_ERR_UNSUPPORTED
        assert fn(a, a, a, a, a, 1, 0, 1, 64, 64, 0.1, 1, 0.0, 8, -1) == lib.ATTN_OK
    ok9 = (a, a, a, a, a, a, a, a, a)
    assert lib.attn_bwd_local(0, *ok9[1:], 1, 2, 2, 128, 128, 0.1, 1, 0.0, a, 64, -1) == \
        lib.ATTN_ERR_NULL
    assert lib.attn_bwd_local(*ok9, 1, 2, 2, 128, 96, 0.1, 1, 0.0, a, 64, -1) == \
        lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_bwd_local(*ok9, 0, 2, 2, 128, 128, 0.1, 1, 0.0, a, 64, -1) == lib.ATTN_OK
    assert lib.attn_fwd_ref(0, a, a, a, a, 1, 1, 1, 64, 64, 0.1, 0, 0.0) == lib.ATTN_ERR_NULL
    assert lib.attn_fwd_ref(a, a, a, a, a, 1, 1, 1, 64, 80, 0.1, 0, 0.0) == lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_fwd_ref(a, a, a, a, a, 1, 4, 3, 64, 64, 0.1, 0, 0.0) == lib.ATTN_ERR_SHAPE
    assert lib.attn_fwd_ref(a, a, a, a + 4, a, 1, 1, 1, 64, 64, 0.1, 0, 0.0) == lib.ATTN_ERR_ALIGN
    assert lib.attn_bwd_preprocess(a, a, 0, a, 1, 1, 64, 64) == lib.ATTN_ERR_NULL
    assert lib.attn_bwd_preprocess(a, a, a, a, 1, 1, 64, 66) == lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_bwd_preprocess(a, a, a, a + 2, 1, 1, 64, 64) == lib.ATTN_ERR_ALIGN
    assert lib.attn_bwd_preprocess(a, a, a, a, 1, 1, 0, 64) == lib.ATTN_OK
    assert lib.attn_bwd_finalize(a, 0, 0.1, 1, 1, 64, 64) == lib.ATTN_ERR_NULL
    assert lib.attn_bwd_finalize(a, a, float("inf"), 1, 1, 64, 64) == lib.ATTN_ERR_SHAPE
    assert lib.attn_bwd_finalize(a, a, 0.1, 1, 1, 64, 64 + 2) == lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_bwd_finalize(a, a, 0.1, 0, 1, 64, 64) == lib.ATTN_OK
    rc = lib.library().attn_device_status(None, 0, None)
    assert rc == lib.ATTN_ERR_NULL
    # deterministic-dQ entry points
    assert lib.attn_bwd_dq_partials_bytes(2, 32, 4096, 128, 1) == 2 * 32 * 528 * 128 * 128 * 4
    assert lib.attn_bwd_dq_partials_bytes(1, 2, 256, 64, 0) == 1 * 2 * 4 * 128 * 64 * 4
    assert lib.attn_bwd_dq_partials_bytes(1, 3, 256, 64, 0) == 3 * 4 * 128 * 64 * 4
    assert lib.attn_bwd_dq_partials_bytes(-1, 2, 256, 64, 0) == lib.ATTN_ERR_SHAPE
    assert lib.attn_bwd_finalize_partials(0, a, 0.1, 1, 1, 64, 64, 1) == lib.ATTN_ERR_NULL
    assert lib.attn_bwd_finalize_partials(a, a, 0.1, 1, 1, 64, 96, 1) == lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_bwd_finalize_partials(a, a, 0.1, 0, 1, 64, 64, 1) == lib.ATTN_OK
    ok = (a, a, a, a, a, a, a, a, a)
    assert lib.attn_bwd_deterministic(0, *ok[1:], 1, 2, 2, 128, 128, 0.1, 1, 0.0, a) == \
        lib.ATTN_ERR_NULL
    assert lib.attn_bwd_deterministic(*ok, 1, 2, 2, 128, 96, 0.1, 1, 0.0, a) == \
        lib.ATTN_ERR_UNSUPPORTED
    # preprocess may skip the accumulator
    assert lib.attn_bwd_preprocess(a, a, a, None, 1, 1, 0, 64) == lib.ATTN_OK


def test_dropout_and_d256_validation(lib):
    a = FAKE
    ok9 = (a, a, a, a, a, a, a, a, a)
    seed = 1234
    # drop probability outside [0, 1)
    for p in (-0.1, 1.0, 1.5, float("nan")):
        assert lib.attn_fwd_dropout(a, a, a, a, a, 1, 1, 1, 64, 64, 0.1, 0, 0.0, p, seed) == \
            lib.ATTN_ERR_SHAPE
        assert lib.attn_fwd_ref_dropout(a, a, a, a, a, 1, 1, 1, 64, 64, 0.1, 0, 0.0, p, seed) == \
            lib.ATTN_ERR_SHAPE
        assert lib.attn_bwd_dropout(*ok9, 1, 2, 2, 128, 128, 0.1, 1, 0.0, a, p, seed) == \
            lib.ATTN_ERR_SHAPE
    # null pointers
    assert lib.attn_fwd_dropout(0, a, a, a, a, 1, 1, 1, 64, 64, 0.1, 0, 0.0, 0.1, seed) == \
        lib.ATTN_ERR_NULL
    assert lib.attn_bwd_dropout(*ok9, 1, 2, 2, 128, 128, 0.1, 1, 0.0, 0, 0.1, seed) == \
        lib.ATTN_ERR_NULL
    # d = 256 is offered by the dropout, deterministic and local backward and
    # the fp32 forward with dropout; other head dimensions are not
    for d in (256,):
        assert lib.attn_fwd_ref_dropout(a, a, a, a, a, 0, 1, 1, 64, d, 0.1, 0, 0.0, 0.1, seed) == \
            lib.ATTN_OK
        assert lib.attn_bwd_dropout(*ok9, 0, 2, 2, 128, d, 0.1, 1, 0.0, a, 0.1, seed) == \
            lib.ATTN_OK
        assert lib.attn_bwd(*ok9, 0, 2, 2, 128, d, 0.1, 1, 0.0, a) == lib.ATTN_OK
        assert lib.attn_bwd_local(*ok9, 0, 2, 2, 128, d, 0.1, 1, 0.0, a, 64, -1) == lib.ATTN_OK
        assert lib.attn_bwd_deterministic(*ok9, 0, 2, 2, 128, d, 0.1, 1, 0.0, a) == lib.ATTN_OK
        assert lib.attn_bwd_finalize_partials(a, a, 0.1, 0, 1, 64, d, 1) == lib.ATTN_OK
    for d in (96, 192, 320):
        assert lib.attn_fwd_ref_dropout(a, a, a, a, a, 1, 1, 1, 64, d, 0.1, 0, 0.0, 0.1, seed) == \
            lib.ATTN_ERR_UNSUPPORTED
        assert lib.attn_bwd_dropout(*ok9, 1, 2, 2, 128, d, 0.1, 1, 0.0, a, 0.1, seed) == \
            lib.ATTN_ERR_UNSUPPORTED
        assert lib.attn_bwd_deterministic(*ok9, 1, 2, 2, 128, d, 0.1, 1, 0.0, a) == \
            lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_bwd_dq_partials_bytes(1, 2, 300, 256, 1) == 2 * 6 * 128 * 256 * 4
    # the tensor-core forwards take d = 256 too
    assert lib.attn_fwd(a, a, a, a, a, 0, 1, 1, 64, 256, 0.1, 0, 0.0) == lib.ATTN_OK
    assert lib.attn_fwd_local(a, a, a, a, a, 0, 1, 1, 64, 256, 0.1, 1, 0.0, 8, -1) == lib.ATTN_OK
    assert lib.attn_fwd_dropout(a, a, a, a, a, 0, 1, 1, 64, 256, 0.1, 0, 0.0, 0.1, seed) == \
        lib.ATTN_OK
    assert lib.attn_fwd(a, a, a, a, a, 1, 1, 1, 64, 192, 0.1, 0, 0.0) == lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_fwd(a, a, a, a, a, 1, 1, 1, 64, 256, -0.1, 0, 0.0) == lib.ATTN_ERR_SHAPE
    # empty problems succeed without touching the device
    assert lib.attn_fwd_dropout(a, a, a, a, a, 0, 1, 1, 64, 64, 0.1, 0, 0.0, 0.1, seed) == \
        lib.ATTN_OK
    assert lib.attn_bwd_dropout(*ok9, 1, 2, 2, 0, 128, 0.1, 1, 0.0, a, 0.1, seed) == lib.ATTN_OK


def test_noalloc_argument_validation(lib):
    """attn_bwd_noalloc runs every check of its three steps before its first
    launch, so each of these returns its code without touching a device."""
    a = FAKE
    ok9 = (a, a, a, a, a, a, a, a, a)
    shape = (1, 2, 2, 128, 128)
    assert lib.attn_bwd_noalloc(0, *ok9[1:], *shape, 0.1, 1, 0.0) == lib.ATTN_ERR_NULL
    for bad_scale in (float("nan"), float("inf"), -float("inf"), 0.0):
        assert lib.attn_bwd_noalloc(*ok9, *shape, bad_scale, 1, 0.0) == lib.ATTN_ERR_SHAPE
    assert lib.attn_bwd_noalloc(*ok9, *shape, 0.1, 1, float("nan")) == lib.ATTN_ERR_SHAPE
    # every one of the nine pointers is checked for 16-byte alignment, o and
    # the output dq included (the main kernel alone never sees them)
    for i in range(9):
        bad = list(ok9)
        bad[i] = a + 8
        assert lib.attn_bwd_noalloc(*bad, *shape, 0.1, 1, 0.0) == lib.ATTN_ERR_ALIGN, i
    assert lib.attn_bwd_noalloc(*ok9, 1, 2, 2, 128, 256, 0.1, 1, 0.0) == lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_bwd_noalloc(*ok9, 1, 3, 2, 128, 128, 0.1, 1, 0.0) == lib.ATTN_ERR_SHAPE
    # the array holds 8,388,608 floats and a problem needs B*H*N*(d + 1):
    # N = 65028 at B = H = 1, d = 128 is one row more than fits (65027 rows)
    assert 65027 * 129 <= 8388608 < 65028 * 129
    assert lib.attn_bwd_noalloc(*ok9, 1, 1, 1, 65028, 128, 0.1, 1, 0.0) == lib.ATTN_ERR_TOO_LARGE
    assert 129055 * 65 <= 8388608 < 129056 * 65
    assert lib.attn_bwd_noalloc(*ok9, 1, 1, 1, 129056, 64, 0.1, 0, 0.0) == lib.ATTN_ERR_TOO_LARGE
    assert lib.attn_bwd_noalloc(*ok9, 0, 2, 2, 128, 128, 0.1, 1, 0.0) == lib.ATTN_OK
