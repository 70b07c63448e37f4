"""GPU parity of dspark_verify against the oracle, stage-isolated: the oracle
verifies the GPU draft's own tokens, lse_d and logp_d with the same l*.
n_accept and next_token must match exactly except requests whose smallest
oracle decision margin (|u - ratio| of an acceptance test, or the top-2 gap
of the final draw) is below 1e-4; those are counted.  A chi-square test over
many identical requests checks losslessness of the GPU path directly."""
import numpy as np
import pytest
import torch
from scipy import stats

from serving_draft_verify_gb300 import workloads as wl
from tests.gpu_harness import gpu_draft, gpu_verify, npy, oracle_verify, compare_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    import serving_draft_verify_gb300 as m
    m.load()
    return m


CASES = [
    ("tiny", wl.TINY, {}),                                                    # fp32: CUDA-core residual
    ("qwen_small", wl.QWEN3_8B, dict(B=24, V=5000, H=64)),                    # bf16: tensor-core residual
    ("two_mtiles", wl.DRAFT_27B, dict(B=140, gamma=4, V=2048, H=96)),
    ("r16_bf16", wl.QWEN3_8B, dict(B=6, gamma=4, V=1000, H=32, r=16)),
]


def _ells(B, G, rng):
    return [np.full(B, G), np.zeros(B, int), rng.integers(0, G + 1, B)]


@pytest.mark.parametrize("name,cfg,changes", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("temperature", [None, 0.0])
def test_verify_parity_small(dsv, name, cfg, changes, temperature):
    cfg = wl.scaled(cfg, **changes)
    inp = wl.make_draft_inputs(cfg)
    d = gpu_draft(dsv, inp, temperature=temperature)
    dn = {k: npy(v) for k, v in d.items()}
    rng = np.random.default_rng(cfg.B)
    exempt = 0
    for ell in _ells(cfg.B, cfg.gamma, rng):
        g = gpu_verify(dsv, inp, d, ell, temperature=temperature)
        ref = oracle_verify(inp, dn, ell, temperature=temperature)
        exempt += compare_verify(g, ref, exact=(temperature == 0.0))
        assert np.all((g["n_accept"] >= 0) & (g["n_accept"] <= ell))
        assert np.all((g["next_token"] >= 0) & (g["next_token"] < cfg.V))
    assert exempt <= max(2, 3 * cfg.B // 20)


def test_verify_many_rejections(dsv):
    """Strong Markov bias and noisy targets: most requests reject early, so the
    residual path runs for many rows."""
    cfg = wl.scaled(wl.QWEN3_8B, B=64, gamma=5, V=4096, H=32, target_noise=2.0)
    inp = wl.make_draft_inputs(cfg)
    g = torch.Generator().manual_seed(9)
    inp["W1"] = (torch.randn(inp["W1"].shape, generator=g) * 0.5).bfloat16()
    inp["W2"] = (torch.randn(inp["W2"].shape, generator=g) * 0.5).bfloat16()
    for T in (0.7, 1.3):
        d = gpu_draft(dsv, inp, temperature=T)
        dn = {k: npy(v) for k, v in d.items()}
        ell = np.full(cfg.B, cfg.gamma)
        gv = gpu_verify(dsv, inp, d, ell, temperature=T)
        compare_verify(gv, oracle_verify(inp, dn, ell, temperature=T))
        assert np.mean(gv["n_accept"] < cfg.gamma) > 0.5


def test_verify_lossless_chi_square(dsv):
    """20000 requests with identical logits: the first emitted token must follow
    softmax(t_1 / T), whatever the draft proposed (section 8.2: lossless)."""
    R, G, V, H, r, T = 20000, 2, 64, 8, 64, 1.0
    gen = torch.Generator().manual_seed(3)
    U1 = torch.randn((G, V), generator=gen) * 1.5
    t1 = torch.cat([U1, torch.randn((1, V), generator=gen)]) + torch.randn((G + 1, V), generator=gen)
    inp = dict(U=U1.expand(R, G, V).contiguous().bfloat16(), t=t1.expand(R, G + 1, V).contiguous().bfloat16(),
               W1=(torch.randn((V, r), generator=gen) * 0.3).bfloat16(),
               W2=(torch.randn((V, r), generator=gen) * 0.3).bfloat16(),
               w=torch.zeros(H + r).bfloat16(), bias=0.0, h=torch.zeros((R, G, H)).bfloat16(),
               x0=torch.full((R,), 5, dtype=torch.int32), temperature=T, seed=11)
    d = gpu_draft(dsv, inp)
    gv = gpu_verify(dsv, inp, d, np.full(R, G))
    x = npy(d["x"])
    first = np.where(gv["n_accept"] >= 1, x[:, 0], gv["next_token"])
    tb = t1.bfloat16().double().numpy()[0] / T
    p = np.exp(tb - tb.max())
    p /= p.sum()
    counts = np.bincount(first, minlength=V).astype(float)
    keep = p * R >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(p[keep] * R, p[~keep].sum() * R)
    if exp[-1] < 5:
        obs, exp = obs[:-1], exp[:-1]
        obs[-1] += counts[~keep].sum()
        exp[-1] += p[~keep].sum() * R
    assert stats.chisquare(obs, exp).pvalue > 1e-3


@pytest.mark.parametrize("key,temperature", [("qwen3_8b", 0.7), ("qwen3_8b", 0.0), ("draft_27b", None),
                                             ("high_conc", None)])
def test_verify_full_size(dsv, key, temperature):
    """Full-size round (draft -> schedule -> verify) on the GPU; requests are
    verified again by the oracle from the GPU's draft outputs (all of them up to
    B = 256; at B = 1024, 152 spread over every M-tile and CTA residue plus the
    request with the longest prefix)."""
    from tests.test_gpu_draft import full_size_rows
    cfg = wl.DRAFT_CONFIGS[key]
    inp = wl.make_draft_inputs(cfg, device="cuda")
    d = gpu_draft(dsv, inp, temperature=temperature)
    sch = dsv.dspark_schedule_prefix(d["a"], inp["sps"])
    ell = npy(sch["ell"])
    gv = gpu_verify(dsv, inp, d, ell, temperature=temperature)
    dn = {k: npy(v) for k, v in d.items()}
    rows = full_size_rows(cfg.B, key)
    if rows.size < cfg.B:
        rows = np.unique(np.append(rows, int(np.argmax(ell))))
    ref = oracle_verify(inp, dn, ell, temperature=temperature, rows=rows)
    exempt = compare_verify(gv, ref, rows=rows, exact=(temperature == 0.0))
    assert exempt <= max(2, rows.size // 20)
    assert np.all((gv["n_accept"] >= 0) & (gv["n_accept"] <= ell))
    del inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("temperature", [None, 0.0])
def test_verify_reads_target_rows_from_pinned_host_memory(dsv, temperature):
    """t_logits in pinned host memory: the same outputs, bit for bit, as from device memory."""
    cfg = wl.scaled(wl.QWEN3_8B, B=32, V=8192, H=64)
    inp = wl.make_draft_inputs(cfg)
    d = gpu_draft(dsv, inp, temperature=temperature)
    T = cfg.temperature if temperature is None else temperature
    g = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    rng = np.random.default_rng(3)
    ell = torch.as_tensor(rng.integers(0, cfg.gamma + 1, cfg.B), dtype=torch.int32).cuda()
    a = dsv.dspark_verify(g["t"], g["U"], g["W1"], g["W2"], g["x0"], d["x"], d["lse_d"], d["logp_d"], ell, T,
                          cfg.seed)
    t_host = inp["t"].clone().pin_memory()
    b = dsv.dspark_verify(t_host, g["U"], g["W1"], g["W2"], g["x0"], d["x"], d["lse_d"], d["logp_d"], ell, T,
                          cfg.seed)
    torch.cuda.synchronize()
    assert torch.equal(a["n_accept"], b["n_accept"]) and torch.equal(a["next_token"], b["next_token"])
