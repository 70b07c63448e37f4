"""GPU parity of dspark_decode_rounds (several draft -> schedule -> verify
rounds with the anchor carried) against the oracle, round by round: the oracle
starts each round from the GPU's anchor and is teacher-forced on the GPU's
draft tokens and survivals (so a decision inside the 1e-4 margin in one round
does not derail the next).  Tokens, l*, n_accept and next_token must match
exactly (outside the margin); the emitted tokens, the carried anchor and the
realised tokens per request are integer bookkeeping and match exactly; E[tau]
matches the exact sum to 1e-12.  The multi-round call must also equal the
three single-round calls chained by hand, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from oracle import rounds as orounds
from serving_draft_verify_gb300 import workloads as wl
from tests.gpu_harness import MARGIN, FTOL, npy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    import serving_draft_verify_gb300 as m
    m.load()
    return m


CASES = [
    ("tiny", wl.TINY, {}),
    ("qwen_small", wl.QWEN3_8B, dict(B=24, V=5000, H=64)),
]


def _run(dsv, g, rounds, T, seed, trace=True):
    anchor = g["x0"].clone().cuda()
    cu = {k: g[k].cuda() for k in ("U", "h", "t", "W1", "W2", "w", "sps")}
    ws = torch.empty(dsv.load().dspark_decode_rounds_workspace_size(*g["U"].shape[1:4], g["W1"].shape[1]),
                     dtype=torch.uint8, device="cuda")
    out = dsv.dspark_decode_rounds(cu["U"], cu["h"], cu["t"], cu["W1"], cu["W2"], cu["w"], g["bias"], cu["sps"],
                                   anchor, rounds, T, seed, trace=trace, workspace=ws)
    assert dsv.workspace_status(ws) == 0
    return {k: npy(v) for k, v in out.items()}, npy(anchor)


@pytest.mark.parametrize("name,cfg,changes", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("temperature", [None, 0.0])
def test_rounds_parity(dsv, name, cfg, changes, temperature):
    cfg = wl.scaled(cfg, **changes)
    g = wl.make_round_pool(cfg, 3)
    T = cfg.temperature if temperature is None else temperature
    R = 5
    got, final = _run(dsv, g, R, T, cfg.seed)
    B, G = cfg.B, cfg.gamma
    dtype = cfg.dtype
    pool = [dict(U=wl.to_f64(g["U"][p]), h=wl.to_f64(g["h"][p]), t=wl.to_f64(g["t"][p])) for p in range(3)]
    anchors = [npy(g["x0"])] + [got["next_token"][i] for i in range(R - 1)]
    forced = [dict(anchor=anchors[i], x=got["x"][i], a=got["a"][i], lse_d=got["lse_d"][i], logp_d=got["logp_d"][i])
              for i in range(R)]
    ref, _ = orounds.decode_rounds(pool, wl.to_f64(g["W1"]), wl.to_f64(g["W2"]), wl.to_f64(g["w"]), g["bias"],
                                   npy(g["sps"]), npy(g["x0"]), T, cfg.seed, R, forced=forced)
    exempt = 0
    for i, o in enumerate(ref):
        ex_d = o["draft_margin"] < MARGIN
        assert not ((got["x"][i] != o["x"]) & ~ex_d).any(), ("round", i, "draft tokens")
        for k in ("c", "a"):
            assert np.abs(got[k][i] - o[k]).max() <= FTOL[dtype], ("round", i, k)
        assert np.array_equal(got["ell"][i], o["ell"]), ("round", i, "ell")
        ex_v = o["verify_margin"] < MARGIN
        bad = ((got["n_accept"][i] != o["n_accept"]) | (got["next_token"][i] != o["next_token"])) & ~ex_v
        assert not bad.any(), ("round", i, "verify")
        exempt += int(ex_d.sum()) + int(ex_v.sum())
        # bookkeeping of the GPU's own round, exactly
        want_tok = orounds.emitted_tokens(got["x"][i], got["n_accept"][i], got["next_token"][i])
        assert np.array_equal(got["tokens"][i], want_tok), ("round", i, "tokens")
        assert np.array_equal(got["n_emitted"][i], got["n_accept"][i] + 1)
        assert got["stats"][i, 1] == np.mean(got["n_accept"][i] + 1.0)
        e = orounds.expected_tau(got["a"][i], got["ell"][i])
        assert abs(got["stats"][i, 0] - e) <= 1e-12 * e, ("round", i, "E[tau]")
    assert np.array_equal(final, got["next_token"][R - 1])
    assert exempt <= max(2, 3 * B * G * R // 100)


def test_rounds_equal_chained_single_calls(dsv):
    """Bit-exact against dspark_draft_block / dspark_schedule_prefix / dspark_verify
    called round by round with seed + i and the anchor set to the last emitted token."""
    cfg = wl.scaled(wl.QWEN3_8B, B=16, V=4096, H=64)
    g = wl.make_round_pool(cfg, 2)
    R, T = 4, 0.7
    got, final = _run(dsv, g, R, T, 1234, trace=False)
    cu = {k: g[k].cuda() for k in ("U", "h", "t", "W1", "W2", "w", "sps")}
    anchor = g["x0"].clone().cuda()
    for i in range(R):
        p = i % 2
        d = dsv.dspark_draft_block(cu["U"][p], cu["h"][p], cu["W1"], cu["W2"], cu["w"], g["bias"], anchor, T,
                                   1234 + i)
        s = dsv.dspark_schedule_prefix(d["a"], cu["sps"])
        v = dsv.dspark_verify(cu["t"][p], cu["U"][p], cu["W1"], cu["W2"], anchor, d["x"], d["lse_d"], d["logp_d"],
                              s["ell"], T, 1234 + i)
        tok = orounds.emitted_tokens(npy(d["x"]), npy(v["n_accept"]), npy(v["next_token"]))
        assert np.array_equal(got["tokens"][i], tok), ("round", i)
        anchor = v["next_token"].clone()
    assert np.array_equal(final, npy(anchor))


def test_rounds_zero_and_pool_of_one(dsv):
    cfg = wl.scaled(wl.TINY, B=3)
    g = wl.make_round_pool(cfg, 1)
    got, final = _run(dsv, g, 0, 1.0, 5, trace=False)
    assert got["tokens"].shape == (0, 3, cfg.gamma + 1)
    assert np.array_equal(final, npy(g["x0"]))
    got, final = _run(dsv, g, 3, 1.0, 5, trace=True)
    assert np.all(got["n_emitted"] >= 1) and np.all(got["n_emitted"] <= cfg.gamma + 1)
    assert np.array_equal(final, got["next_token"][2])


def test_rounds_full_qwen3_size_sampled_requests(dsv):
    """Two rounds of the Qwen3-8B-shaped workload (B = 64, V = 151936, bf16, T = 0.7, pool of
    2): four sampled requests of each round against the teacher-forced oracle, and the whole
    batch's bookkeeping exactly."""
    cfg = wl.QWEN3_8B
    g = wl.make_round_pool(cfg, 2, device="cuda")
    R, T = 2, cfg.temperature
    anchor = g["x0"].clone()
    out = dsv.dspark_decode_rounds(g["U"], g["h"], g["t"], g["W1"], g["W2"], g["w"], 0.0, g["sps"], anchor, R, T,
                                   cfg.seed, trace=True)
    torch.cuda.synchronize()
    got = {k: npy(v) for k, v in out.items()}
    rows = np.array([0, 21, 42, 63])
    idx = torch.from_numpy(rows).cuda()
    anchors = [npy(g["x0"])] + [got["next_token"][i] for i in range(R - 1)]
    W1, W2, w = wl.to_f64(g["W1"]), wl.to_f64(g["W2"]), wl.to_f64(g["w"])
    for i in range(R):
        s = orounds.round_seed(cfg.seed, i)
        U = wl.to_f64(g["U"][i][idx])
        d = oracle.draft_block(U, wl.to_f64(g["h"][i][idx]), W1, W2, w, 0.0, anchors[i][rows], T, s,
                               forced_tokens=got["x"][i][rows], requests=rows)
        assert not ((got["x"][i][rows] != d["x"]) & ~(d["margin"] < MARGIN)).any(), ("round", i)
        assert np.abs(got["a"][i][rows] - d["a"]).max() <= FTOL["bf16"]
        # the scheduler over the whole batch, on the GPU's survivals: exact
        ell, _, _ = oracle.schedule_prefix(got["a"][i], npy(g["sps"]))
        assert np.array_equal(ell, got["ell"][i]), ("round", i, "ell")
        v = oracle.verify_round(wl.to_f64(g["t"][i][idx]), U, W1, W2, anchors[i][rows], got["x"][i][rows],
                                got["lse_d"][i][rows], got["logp_d"][i][rows], ell[rows], T, s, requests=rows)
        bad = ((got["n_accept"][i][rows] != v["n_accept"]) | (got["next_token"][i][rows] != v["next_token"])) \
            & ~(v["margin"] < MARGIN)
        assert not bad.any(), ("round", i, "verify")
        tok = orounds.emitted_tokens(got["x"][i], got["n_accept"][i], got["next_token"][i])
        assert np.array_equal(got["tokens"][i], tok)
    assert np.array_equal(npy(anchor), got["next_token"][R - 1])


def test_rounds_with_target_logits_in_pinned_host_memory(dsv):
    """The target-logit pool in pinned host memory: bit-identical rounds."""
    cfg = wl.scaled(wl.QWEN3_8B, B=16, V=4096, H=64)
    g = wl.make_round_pool(cfg, 2)
    cu = {k: g[k].cuda() for k in ("U", "h", "t", "W1", "W2", "w", "sps")}
    outs = []
    for t in (cu["t"], g["t"].clone().pin_memory()):
        anchor = g["x0"].clone().cuda()
        o = dsv.dspark_decode_rounds(cu["U"], cu["h"], t, cu["W1"], cu["W2"], cu["w"], 0.0, cu["sps"], anchor, 3,
                                     0.7, 99)
        torch.cuda.synchronize()
        outs.append((npy(o["tokens"]), npy(anchor)))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
