"""Host-only checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every function include/specverify.h declares, and
rejects invalid arguments synchronously without touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    import speculative_decoding_token_gb300 as sv
    sv.build()
    return sv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(specverify_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ["specverify_create", "specverify_verify", "specverify_verify_greedy",
                 "specverify_destroy", "specverify_device_status"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    import speculative_decoding_token_gb300 as sv
    assert sv.specverify_status_string(0) == "ok"
    assert "invalid" in sv.specverify_status_string(-1)
    assert sv.specverify_status_string(12345) == "unknown status"


def test_invalid_arguments_are_rejected_on_the_host(lib):
    import speculative_decoding_token_gb300 as sv
    # NULL out-pointer and out-of-range sizes fail before any CUDA call
    assert lib.specverify_create(None, 0, 1, 1, 1) == sv.ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert lib.specverify_create(ctypes.byref(h), 0, 0, 1, 1) == sv.ERR_INVALID_ARG
    assert lib.specverify_create(ctypes.byref(h), 0, 1, 257, 1) == sv.ERR_INVALID_ARG
    assert lib.specverify_create(ctypes.byref(h), 0, 1, 1, 0) == sv.ERR_INVALID_ARG
    assert lib.specverify_create(ctypes.byref(h), -1, 1, 1, 1) == sv.ERR_INVALID_ARG
    batch = sv.SpecverifyBatch()
    assert lib.specverify_verify(None, ctypes.byref(batch), 1.0, 0, None, None, None, None,
                                 None) == sv.ERR_INVALID_ARG
    assert lib.specverify_verify_greedy(None, ctypes.byref(batch), None, None, None) == \
        sv.ERR_INVALID_ARG
    assert lib.specverify_device_status(None, None, None) == sv.ERR_INVALID_ARG
    assert lib.specverify_destroy(None) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import speculative_decoding_token_gb300 as sv
    from speculative_decoding_token_gb300 import _build
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "nothing.so"))
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        sv.load()
