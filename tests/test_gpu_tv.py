"""GPU parity of dspark_accept_rate_tv against the oracle (float64 c*).

Tolerance (the parity bar): 2e-3 absolute for bf16 inputs, 1e-5 for fp32.
The kernel sums fp32 terms, so it is also held to a tighter 1e-4 / 2e-6 that
documents its expected accuracy."""
import numpy as np
import pytest
import torch

import oracle
from serving_draft_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-3, torch.float32: 1e-5}
TIGHT = {torch.bfloat16: 1e-4, torch.float32: 2e-6}


@pytest.fixture(scope="module")
def dsv():
    import serving_draft_verify_gb300 as m
    m.load()
    return m


def _check(dsv, d, t):
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    got = dsv.dspark_accept_rate_tv(d.cuda(), t.cuda(), workspace=ws)
    assert dsv.workspace_status(ws) == 0
    want = oracle.accept_rate_tv(wl.to_f64(d), wl.to_f64(t))
    err = np.abs(got.cpu().numpy().astype(np.float64) - want)
    assert err.max() < TOL[d.dtype], err.max()
    assert err.max() < TIGHT[d.dtype], err.max()
    return err.max()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V", [8, 1024, 5000, 151936, 262144])
def test_tv_parity_seeded_rows(dsv, dtype, V):
    cfg = wl.scaled(wl.TV_TRAIN, V=V)
    d, t = wl.make_tv_inputs(cfg, rows=37)
    _check(dsv, d.to(dtype), t.to(dtype))


def test_tv_special_cases(dsv):
    V = 4096
    rng = np.random.default_rng(0)
    d = torch.from_numpy(rng.normal(0, 2, (6, V))).float()
    t = d.clone()
    t[1] += 3.0                                   # shift invariance -> 1
    t[2] = -1e30                                  # disjoint halves -> 0
    t[2, V // 2:] = 0.0
    d[2] = -1e30
    d[2, : V // 2] = 0.0
    d[3] = 0.0                                    # uniform vs peaked
    t[3] = 0.0
    t[3, 7] = 50.0
    d[4] = float("-inf")                          # a single finite logit per row
    d[4, 100] = 1.0
    t[4] = float("-inf")
    t[4, 100] = -4.0
    for dt in (torch.float32, torch.bfloat16):
        got = dsv.dspark_accept_rate_tv(d.to(dt).cuda(), t.to(dt).cuda()).cpu().numpy()
        assert abs(got[0] - 1.0) < 1e-5
        if dt == torch.float32:      # d + 3 rounded to bf16 is not an exact shift of d in bf16
            assert abs(got[1] - 1.0) < 1e-5
        assert got[2] == 0.0
        assert abs(got[4] - 1.0) < 1e-6
        want = oracle.accept_rate_tv(wl.to_f64(d.to(dt)), wl.to_f64(t.to(dt)))
        assert np.max(np.abs(got - want)) < 1e-5


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("offset", [-120.0, 60.0, 100.0])
def test_tv_large_logits(dsv, dtype, offset):
    """Logits far from 0: the bf16 path forms its exponents as x log2e - L log2e in
    one fused step, so every term carries the rounding of L log2e (largest at large
    |L|); both dtypes must still meet the tight bound."""
    cfg = wl.scaled(wl.TV_TRAIN, V=151936)
    d, t = wl.make_tv_inputs(cfg, rows=9)
    _check(dsv, (d.float() + offset).to(dtype), (t.float() + offset).to(dtype))


def test_tv_empty_and_one_row(dsv):
    out = torch.full((0,), 7.0, device="cuda")
    d = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    dsv.dspark_accept_rate_tv(d, d, c_star=out)
    d, t = wl.make_tv_inputs(wl.scaled(wl.TV_TRAIN, V=151936), rows=1)
    _check(dsv, d, t)


def test_tv_full_size_sampled(dsv):
    """16384 x 151936 bf16 rows (the training accept-rate workload), generated on
    the GPU; 48 sampled rows are checked one by one against the oracle, and every
    row is checked against properties that hold at any size."""
    cfg = wl.TV_TRAIN
    d, t = wl.make_tv_inputs(cfg, device="cuda")
    got = dsv.dspark_accept_rate_tv(d, t)
    torch.cuda.synchronize()
    g = got.cpu().numpy()
    assert np.all(np.isfinite(g)) and np.all(g >= -1e-6) and np.all(g <= 1 + 1e-6)
    rows = np.random.default_rng(1).choice(cfg.rows, 48, replace=False)
    rows[:2] = [0, cfg.rows - 1]
    idx = torch.from_numpy(rows).cuda()
    want = oracle.accept_rate_tv(wl.to_f64(d[idx]), wl.to_f64(t[idx]))
    err = np.abs(g[rows] - want)
    assert err.max() < TOL[torch.bfloat16] and err.max() < TIGHT[torch.bfloat16], err.max()
    del d, t
    torch.cuda.empty_cache()
