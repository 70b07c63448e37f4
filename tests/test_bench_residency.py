"""The benchmark's W2 residency setting: on for the headline run, off for the
one-kernel modes, unless --l2-residency on|off says otherwise."""
import argparse

import bench


class _FakeLib:
    def __init__(self):
        self.calls = []

    def dspark_set_l2_residency(self, nbytes):
        self.calls.append(nbytes)


def _apply(mode, default):
    lib = _FakeLib()
    kept = bench.apply_l2_residency(lib, argparse.Namespace(l2_residency=mode), default=default)
    return kept, lib.calls


def test_auto_follows_the_mode_default():
    kept, calls = _apply("auto", default=True)
    assert kept > 0 and calls == [kept]
    assert _apply("auto", default=False) == (0, [])


def test_explicit_setting_wins():
    assert _apply("off", default=True) == (0, [])
    kept, calls = _apply("on", default=False)
    assert kept > 0 and calls == [kept]


def test_flag_alone_means_on():
    ap = bench.arg_parser()
    assert ap.parse_args(["--l2-residency"]).l2_residency == "on"
    assert ap.parse_args(["--l2-residency", "off"]).l2_residency == "off"
    assert ap.parse_args([]).l2_residency == "auto"
