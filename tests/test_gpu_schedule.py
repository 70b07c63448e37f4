"""GPU parity of dspark_schedule_prefix against the oracle's literal Algorithm 1:
l*, N and Theta_best must be bit-identical (the survival sum is exact on both
sides and Theta is one IEEE division and one multiplication)."""
import numpy as np
import pytest
import torch

from oracle import schedule

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    import serving_draft_verify_gb300 as m
    m.load()
    return m


def _sps(B, G, alpha=20.0, beta=0.05):
    N = np.arange(B * (G + 1) + 1, dtype=np.float64)
    return N / (alpha + beta * N)


def _run(dsv, a, sps):
    a = np.asarray(a, np.float32)
    ws = torch.empty(dsv.load().dspark_schedule_prefix_workspace_size(*a.shape), dtype=torch.uint8, device="cuda")
    out = dsv.dspark_schedule_prefix(torch.from_numpy(a).cuda(), torch.from_numpy(np.asarray(sps)).cuda(),
                                     workspace=ws)
    assert dsv.workspace_status(ws) == 0
    ell, n, th = schedule.schedule_prefix(a, sps)
    assert np.array_equal(out["ell"].cpu().numpy(), ell)
    assert int(out["n_sched"].item()) == n
    assert out["theta"].item() == th                     # bit-exact double
    return ell


def _survival(c):
    return np.cumprod(np.asarray(c, np.float32), axis=1, dtype=np.float32)


@pytest.mark.parametrize("B,G", [(1, 1), (4, 7), (3, 2), (64, 7), (100, 3), (256, 7), (1024, 16),
                                 (16384, 1), (512, 32)])
def test_schedule_random(dsv, B, G):
    rng = np.random.default_rng(B * 131 + G)
    for alpha, beta in ((20.0, 0.05), (2.0, 0.5), (200.0, 0.001)):
        c = rng.beta(5, 2, (B, G))
        _run(dsv, _survival(c), _sps(B, G, alpha, beta))


def test_schedule_constant_confidence_per_request(dsv):
    rng = np.random.default_rng(7)
    B, G = 1024, 16
    q = rng.beta(5, 2, B)
    _run(dsv, _survival(np.repeat(q[:, None], G, axis=1)), _sps(B, G))


def test_schedule_ties_and_extremes(dsv):
    B, G = 300, 7
    _run(dsv, np.ones((B, G)), _sps(B, G))                          # every pair ties at 1
    _run(dsv, np.zeros((B, G)), _sps(B, G))                         # nothing worth verifying
    _run(dsv, np.full((B, G), 0.5), _sps(B, G, 2.0, 0.3))           # ties broken by (b, j)
    a = np.repeat(np.array([[1.0, 0.75, 0.5, 0.5, 0.25, 0.25, 0.0]]), B, axis=0)
    _run(dsv, a, _sps(B, G, 0.5, 0.1))
    rng = np.random.default_rng(3)
    tiny = _survival(rng.uniform(1e-8, 1e-3, (B, G)))               # deep denormals
    _run(dsv, tiny, _sps(B, G))


def test_schedule_rounding_ties(dsv):
    # E = 1 + 2^-53 is halfway between two doubles (rounds to even, 1.0);
    # 1 + 2^-53 + 2^-100 is just above halfway (rounds up); whether the pair is
    # taken depends on that rounding, so both sides must round the same way
    for a in ([[1.0, 2.0 ** -53]], [[2.0 ** -53, 2.0 ** -100]], [[1.0, 2.0 ** -53, 2.0 ** -100]],
              [[1.0, 2.0 ** -52, 2.0 ** -53]], [[2.0 ** -24, 2.0 ** -60, 2.0 ** -126]],
              [[1e-45, 1e-45, 1e-45]]):
        a = np.array(a, np.float32)
        B, G = a.shape
        rising = np.arange(B * (G + 1) + 1, dtype=np.float64) * 3.0
        _run(dsv, a, rising)


def test_schedule_non_concave_table_stops_at_first_drop(dsv):
    B, G = 2, 2
    a = np.full((B, G), 0.9, np.float32)
    ell = _run(dsv, a, np.array([0.0, 1.0, 1.0, 0.5, 5.0, 5.0, 5.0]))
    assert list(ell) == [0, 0]
    rng = np.random.default_rng(11)
    for _ in range(20):
        B, G = int(rng.integers(1, 60)), int(rng.integers(1, 9))
        table = rng.uniform(0.5, 2.0, B * (G + 1) + 1)
        _run(dsv, _survival(rng.uniform(0.2, 1.0, (B, G))), table)


def test_schedule_rejects_out_of_range_survival(dsv):
    a = torch.tensor([[0.5, float("nan")], [1.5, 0.2]], device="cuda")
    ws = torch.empty(dsv.load().dspark_schedule_prefix_workspace_size(2, 2), dtype=torch.uint8, device="cuda")
    dsv.dspark_schedule_prefix(a, torch.ones(7, dtype=torch.float64, device="cuda"), workspace=ws)
    assert dsv.workspace_status(ws) == 6        # DSPARK_ERR_DEVICE_CHECK


def test_schedule_workspace_reuse_and_late_chunk_error(dsv):
    """One workspace through calls of different sizes: the per-chunk sums, flags and
    counters are cleared by each call; an out-of-range survival in the last chunk of
    a many-chunk batch is reported, and the next valid call reports a clear status."""
    lib = dsv.load()
    ws = torch.empty(lib.dspark_schedule_prefix_workspace_size(1024, 16), dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(21)

    def call(a, sps):
        out = dsv.dspark_schedule_prefix(torch.from_numpy(a).cuda(), torch.from_numpy(sps).cuda(), workspace=ws)
        torch.cuda.synchronize()
        return out

    for B, G in ((1024, 16), (37, 3), (1000, 9), (5, 1)):
        a = _survival(rng.beta(5, 2, (B, G)))
        sps = _sps(B, G, 2.0, 0.01)
        out = call(a, sps)
        assert dsv.workspace_status(ws) == 0
        ell, n, th = schedule.schedule_prefix(a, sps)
        assert np.array_equal(out["ell"].cpu().numpy(), ell) and int(out["n_sched"].item()) == n
        assert out["theta"].item() == th
    B, G = 1000, 9
    a = _survival(rng.beta(5, 2, (B, G)))
    bad = a.copy()
    bad[B - 1, G - 1] = np.float32(np.nan)                  # pair 8999: the last of 71 chunks
    call(bad, _sps(B, G))
    assert dsv.workspace_status(ws) == 6
    out = call(a, _sps(B, G))
    assert dsv.workspace_status(ws) == 0
    assert np.array_equal(out["ell"].cpu().numpy(), schedule.schedule_prefix(a, _sps(B, G))[0])
