"""The C-ABI library builds, loads without a GPU, and exports every entry point
include/*.h declares; the host-side argument checks reject bad calls before
any launch (no compute is attempted here)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from serving_draft_verify_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    return ctypes.CDLL(b.LIB)


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names.update(re.findall(r"\b(dspark_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_four_operations():
    names = _declared()
    for op in ("dspark_draft_block", "dspark_schedule_prefix", "dspark_verify", "dspark_accept_rate_tv"):
        assert op in names and op + "_workspace_size" in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    from serving_draft_verify_gb300 import _binding
    assert set(_declared()) <= set(_binding.exported_symbols())


def test_status_strings(lib):
    lib.dspark_status_string.restype = ctypes.c_char_p
    assert lib.dspark_status_string(0) == b"DSPARK_OK"
    assert lib.dspark_status_string(1) == b"DSPARK_ERR_INVALID_ARGUMENT"
    assert lib.dspark_status_string(99) == b"DSPARK_ERR_UNKNOWN"


def test_host_checks_reject_before_launch(lib):
    # invalid arguments are refused on the host: no device memory is touched
    f = lib.dspark_accept_rate_tv
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 4 + \
                 [ctypes.c_size_t, ctypes.c_void_p]
    fake = ctypes.c_void_p(0x1000)
    assert f(-1, 64, 1, fake, fake, fake, fake, 256, None) == 1        # rows < 0
    assert f(4, 60, 1, fake, fake, fake, fake, 256, None) == 1         # V % 8 != 0 for bf16
    assert f(4, 64, 7, fake, fake, fake, fake, 256, None) == 1         # bad dtype
    assert f(4, 64, 1, fake, fake, fake, None, 256, None) == 1         # no workspace
    assert f(4, 64, 1, fake, fake, fake, fake, 16, None) == 3          # workspace too small
    assert f(4, 64, 1, ctypes.c_void_p(0x1001), fake, fake, fake, 256, None) == 1   # misaligned d
    g = lib.dspark_schedule_prefix
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 6 + [ctypes.c_size_t, ctypes.c_void_p]
    assert g(0, 7, fake, fake, fake, fake, fake, fake, 256, None) == 1        # B = 0
    assert g(4, 33, fake, fake, fake, fake, fake, fake, 256, None) == 1       # gamma > 32
    assert g(1024, 17, fake, fake, fake, fake, fake, fake, 256, None) == 2    # more than 16384 pairs
