"""GPU parity of the draft block and verification at the degenerate and the
largest draft lengths: gamma = 1 (one position: the first is also the last)
and gamma = 32 (the largest the C ABI accepts; verification keeps one lane per
position), on the tensor-core (bf16) and CUDA-core (fp32) paths, with ragged
vocabularies."""
import numpy as np
import pytest

from serving_draft_verify_gb300 import workloads as wl
from tests.gpu_harness import (compare_draft, compare_verify, gpu_draft, gpu_verify, npy, oracle_draft,
                               oracle_verify)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    import serving_draft_verify_gb300 as m
    m.load()
    return m


EDGES = [
    ("g1_bf16", wl.QWEN3_8B, dict(B=12, gamma=1, V=1000, H=32)),
    ("g1_f32", wl.TINY, dict(B=5, gamma=1, V=600)),
    ("g32_bf16", wl.QWEN3_8B, dict(B=6, gamma=32, V=1000, H=32)),
    ("g32_f32", wl.TINY, dict(B=3, gamma=32, V=600)),
]


@pytest.mark.parametrize("name,cfg,changes", EDGES, ids=[c[0] for c in EDGES])
@pytest.mark.parametrize("temperature", [None, 0.0])
def test_draft_and_verify_at_edge_lengths(dsv, name, cfg, changes, temperature):
    cfg = wl.scaled(cfg, **changes)
    inp = wl.make_draft_inputs(cfg)
    d = gpu_draft(dsv, inp, temperature=temperature)
    dn = {k: npy(v) for k, v in d.items()}
    ref = oracle_draft(inp, dn["x"], temperature=temperature)
    exempt = compare_draft(dn, ref, cfg.dtype)
    assert exempt <= max(2, dn["x"].size // 50)
    assert np.all(np.diff(dn["a"], axis=1) <= 0) and np.all((dn["a"] >= 0) & (dn["a"] <= 1))
    rng = np.random.default_rng(cfg.B + cfg.gamma)
    for ell in (np.full(cfg.B, cfg.gamma), np.zeros(cfg.B, int), rng.integers(0, cfg.gamma + 1, cfg.B)):
        g = gpu_verify(dsv, inp, d, ell, temperature=temperature)
        vref = oracle_verify(inp, dn, ell, temperature=temperature)
        exempt += compare_verify(g, vref, exact=(temperature == 0.0))
        assert np.all((g["n_accept"] >= 0) & (g["n_accept"] <= ell))
        assert np.all((g["next_token"] >= 0) & (g["next_token"] < cfg.V))
    assert exempt <= max(2, (dn["x"].size + 3 * cfg.B) // 20)
