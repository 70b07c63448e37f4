"""GPU checks of the sampler's noise routines, the pieces every draw shares.

  * E = -ln u on the device for every one of the 2^23 uniforms
    u = (m + 1/2) 2^-23 the generator can give, against float64: the draws
    compare lw_v - ln E_v (or e_v / E_v), so E must keep its relative
    accuracy where it is small (u near 1).  The bound asserted, 4e-6, keeps
    the error of a Gumbel key (ln E) far below the 1e-4 decision margin that
    parity tests exempt.
  * The per-row Philox4x32-10 of the draws (two constant rounds hoisted)
    against the oracle's generator, which is pinned to the published
    known-answer vectors.
"""
import numpy as np
import pytest
import torch

from oracle import philox

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    import serving_draft_verify_gb300 as m
    m.load()
    return m


def test_exponential_variate_every_uniform(dsv):
    m = torch.arange(1 << 23, dtype=torch.int64, device="cuda")
    # the low 9 bits of a word do not enter u: vary them to check that too
    low = torch.randint(0, 512, m.shape, generator=torch.Generator(device="cuda").manual_seed(1), device="cuda")
    words = (m << 9) | low
    words = torch.where(words >= 2 ** 31, words - 2 ** 32, words)        # int32 bit patterns
    E = dsv._binding.exp_draws(words).double().cpu().numpy()
    u = (np.arange(1 << 23, dtype=np.float64) + 0.5) * 2.0 ** -23
    ref = -np.log(u)
    rel = np.abs(E - ref) / ref
    worst = int(np.argmax(rel))
    print(f"exp_draws: max relative error {rel.max():.3e} at u = {u[worst]!r}")
    assert np.all(E > 0)
    assert rel.max() < 4e-6, (rel.max(), u[worst])


@pytest.mark.parametrize("seed,k,b,stream,q0", [
    (0, 1, 0, 0, 0),
    (0x0123456789ABCDEF, 7, 63, 2, 37980),
    (2 ** 64 - 1, 32, 65535, 1, 2 ** 32 - 100),        # counter wrap-around of the first word
    (4, 16, 1023, 0, 12345),
])
def test_philox_rows_match_the_generator(dsv, seed, k, b, stream, q0):
    n = 200
    got = dsv._binding.philox_rows(seed, k, b, stream, q0, n).cpu().numpy().astype(np.uint64)
    q = (np.arange(n, dtype=np.uint64) + np.uint64(q0)) & np.uint64(0xFFFFFFFF)
    ref = philox.philox4x32_10(q, k, b, stream, seed & 0xFFFFFFFF, seed >> 32)
    for j in range(4):
        assert np.array_equal(got[:, j], ref[j]), j
