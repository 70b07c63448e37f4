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


def test_host_checks_of_the_other_entry_points(lib):
    # only arguments each entry point rejects in its first checks, before any CUDA call
    P = ctypes.c_void_p
    fake = P(0x1000)
    i, f32, u64, sz = ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t

    d = lib.dspark_draft_block
    d.restype = i
    d.argtypes = [i] * 6 + [P] * 5 + [f32, P, f32, u64] + [P] * 6 + [sz, P]

    def draft(B=4, G=7, V=64, H=8, r=16, dt=1, T=1.0):
        return d(B, G, V, H, r, dt, fake, fake, fake, fake, fake, 0.0, fake, T, 1,
                 fake, fake, fake, fake, fake, fake, 1 << 30, None)
    assert draft(B=0) == 1 and draft(B=65536) == 1
    assert draft(G=0) == 1 and draft(G=33) == 1
    assert draft(r=264) == 1 and draft(r=12) == 1               # r > 256, r % 8 != 0
    assert draft(dt=7) == 1
    assert draft(T=-1.0) == 1 and draft(T=float("nan")) == 1 and draft(T=float("inf")) == 1
    assert draft(V=60) == 1                                     # bf16 rows need V % 8 == 0

    v = lib.dspark_verify
    v.restype = i
    v.argtypes = [i] * 5 + [P] * 9 + [f32, u64] + [P] * 3 + [sz, P]

    def verify(B=4, G=7, V=64, r=16, dt=1, T=1.0):
        return v(B, G, V, r, dt, fake, fake, fake, fake, fake, fake, fake, fake, fake, T, 1,
                 fake, fake, fake, 1 << 30, None)
    assert verify(B=0) == 1 and verify(G=33) == 1 and verify(r=12) == 1 and verify(dt=7) == 1
    assert verify(B=65535, G=1) == 2                            # more than 65535 target rows
    assert verify(T=-0.5) == 1 and verify(V=60) == 1

    lo = lib.dspark_training_loss
    lo.restype = i
    lo.argtypes = [ctypes.c_int64, i, i] + [P] * 5 + [f32] * 3 + [P] * 5 + [sz, P]

    def loss(rows=4, V=64, dt=1, ws=fake, ws_bytes=1 << 20, out=fake):
        return lo(rows, V, dt, fake, fake, fake, fake, fake, 0.1, 0.9, 1.0, fake, out, None, None,
                  ws, ws_bytes, None)
    assert loss(rows=-1) == 1 and loss(V=60) == 1 and loss(dt=7) == 1
    assert loss(ws=None) == 1 and loss(ws=P(0x1010)) == 1        # workspace missing / not 256-byte aligned
    assert loss(ws_bytes=16) == 3
    assert loss(out=None) == 1                                  # no loss output

    r = lib.dspark_decode_rounds
    r.restype = i
    r.argtypes = [i] * 8 + [P] * 6 + [f32, P, P, f32, u64] + [P] * 5 + [sz, P]

    def rounds(n=2, pool=1, B=4, G=7, dt=1):
        return r(n, pool, B, G, 64, 8, 16, dt, fake, fake, fake, fake, fake, fake, 0.0, fake, fake, 1.0, 1,
                 fake, fake, fake, None, fake, 1 << 30, None)
    assert rounds(n=-1) == 1 and rounds(pool=0) == 1 and rounds(B=0) == 1 and rounds(G=0) == 1
    assert rounds(dt=7) == 1
