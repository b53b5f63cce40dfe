"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/gemm.h declares, and rejects bad arguments on the host before
touching any device (so these run on CPU-only machines too)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FAKE = 0x7F0000000000   # a 256-byte-aligned address; never dereferenced here


def _declared():
    text = open(os.path.join(ROOT, "include", "gemm.h")).read()
    return re.findall(r"GEMM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_documented_entry_points():
    names = _declared()
    assert "gemm" in names and "gemm_status_string" in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(libgemm):
    lib = libgemm.lib()
    for name in _declared():
        assert hasattr(lib, name), f"libgemm.so does not export {name}"
        assert name in libgemm.SIGNATURES, f"binding has no signature for {name}"


def test_status_strings(libgemm):
    for code in range(8):
        s = libgemm.status_string(code)
        assert s and s != "unknown status"
    assert libgemm.status_string(99) == "unknown status"
    assert libgemm.version() == 200
    assert libgemm.launch_count() >= 0


@pytest.mark.parametrize("mode", [-1, 6, 17])
def test_bad_mode(libgemm, mode):
    assert libgemm.gemm_raw(FAKE, FAKE + 4096, FAKE + 8192, 4, 4, 4, mode) == libgemm.ERR_INVALID_ARG


@pytest.mark.parametrize("dims", [(-1, 4, 4), (4, -1, 4), (4, 4, -1), (1 << 31, 1, 1),
                                  (1 << 30, 1 << 30, 1 << 30)])
def test_bad_dims(libgemm, dims):
    M, K, N = dims
    assert libgemm.gemm_raw(FAKE, FAKE, FAKE, M, K, N, 0) == libgemm.ERR_INVALID_ARG


def test_empty_output_needs_no_device(libgemm):
    # nothing to do: returns before any CUDA call, even with NULL pointers
    for mode in (0, 1, 2):
        assert libgemm.gemm_raw(0, 0, 0, 0, 5, 5, mode) == libgemm.OK
        assert libgemm.gemm_raw(0, 0, 0, 5, 5, 0, mode) == libgemm.OK


def test_null_pointers(libgemm):
    G = 1 << 20
    assert libgemm.gemm_raw(0, FAKE + G, FAKE + 2 * G, 4, 4, 4, 0) == libgemm.ERR_INVALID_ARG
    assert libgemm.gemm_raw(FAKE, 0, FAKE + 2 * G, 4, 4, 4, 1) == libgemm.ERR_INVALID_ARG
    assert libgemm.gemm_raw(FAKE, FAKE + G, 0, 4, 4, 4, 2) == libgemm.ERR_INVALID_ARG


def test_misaligned_pointers(libgemm):
    G = 1 << 20
    assert libgemm.gemm_raw(FAKE + 2, FAKE + G, FAKE + 2 * G, 4, 4, 4, 0) == libgemm.ERR_MISALIGNED
    assert libgemm.gemm_raw(FAKE, FAKE + G + 1, FAKE + 2 * G, 4, 4, 4, 1) == libgemm.ERR_MISALIGNED
    assert libgemm.gemm_raw(FAKE, FAKE + G, FAKE + 2 * G + 2, 4, 4, 4, 2) == libgemm.ERR_MISALIGNED
    assert libgemm.gemm_raw(FAKE + 1, FAKE + G, FAKE + 2 * G, 4, 4, 4, 2) == libgemm.ERR_MISALIGNED


def test_c_overlapping_a_or_b(libgemm):
    G = 1 << 20
    # C starts inside A
    assert libgemm.gemm_raw(FAKE, FAKE + G, FAKE + 16, 4, 4, 4, 0) == libgemm.ERR_INVALID_ARG
    # C ends inside B (bf16 B of 4x4 = 32 bytes at FAKE+G; C of 64 bytes before it)
    assert libgemm.gemm_raw(FAKE, FAKE + G, FAKE + G - 48, 4, 4, 4, 2) == libgemm.ERR_INVALID_ARG


def test_no_device_is_an_error_not_a_crash(libgemm):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    G = 1 << 20
    rc = libgemm.gemm_raw(FAKE, FAKE + G, FAKE + 2 * G, 4, 4, 4, 0)
    assert rc in (libgemm.ERR_CUDA, libgemm.ERR_UNSUPPORTED_DEVICE)


def test_gemm_ex_validates_like_gemm(libgemm):
    G = 1 << 20
    ex = libgemm.gemm_ex_raw
    assert ex(FAKE, FAKE + G, FAKE + 2 * G, 4, 4, 4, 2.0, 1.0, 6) == libgemm.ERR_INVALID_ARG
    assert ex(FAKE, FAKE, FAKE, -1, 4, 4, 2.0, 1.0, 0) == libgemm.ERR_INVALID_ARG
    assert ex(0, 0, 0, 0, 5, 5, 2.0, 1.0, 0) == libgemm.OK          # empty C: nothing to do
    assert ex(0, FAKE + G, FAKE + 2 * G, 4, 4, 4, 2.0, 1.0, 0) == libgemm.ERR_INVALID_ARG
    assert ex(FAKE, FAKE + G, FAKE + 2 * G + 2, 4, 4, 4, 2.0, 1.0, 1) == libgemm.ERR_MISALIGNED
    assert ex(FAKE, FAKE + G, FAKE + 16, 4, 4, 4, 2.0, 1.0, 0) == libgemm.ERR_INVALID_ARG
