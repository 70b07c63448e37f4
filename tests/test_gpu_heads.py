"""GPU parity of the gated and recurrent heads (dspark_draft_block_ex /
dspark_verify_ex) against the oracle.  The oracle draft is teacher-forced on the
GPU's tokens and forms its own e_k (float64, rounded to bf16 for bf16 weights);
the GPU's E must match it (bf16: within one bf16 step, and equal for all but
1 % of the entries; fp32: 1e-5 relative), and
the draft outputs hold to the bars of the Markov-head tests.  Verification is
stage-isolated: the oracle verifies the GPU's tokens with the GPU's E."""
import numpy as np
import pytest
import torch

import oracle
from oracle import heads as oheads
from serving_draft_verify_gb300 import workloads as wl
from tests.gpu_harness import MARGIN, FTOL, npy, compare_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv():
    import serving_draft_verify_gb300 as m
    m.load()
    return m


CASES = [
    ("tiny", wl.TINY, {}),                                                    # fp32: CUDA-core phases
    ("qwen_small", wl.QWEN3_8B, dict(B=24, V=5000, H=64)),                    # bf16: tensor-core phases
]


def _run(dsv, inp, kind, Wg, Wc, T):
    d = torch.device("cuda")
    g = {k: (v.to(d) if torch.is_tensor(v) else v) for k, v in inp.items()}
    head = dict(kind=kind, Wg=Wg.to(d), Wc=None if Wc is None else Wc.to(d))
    out = dsv.dspark_draft_block_ex(g["U"], g["h"], g["W1"], g["W2"], g["w"], inp["bias"], g["x0"], T, inp["seed"],
                                    head)
    return g, out


@pytest.mark.parametrize("name,cfg,changes", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("kind", [1, 2], ids=["gated", "rnn"])
@pytest.mark.parametrize("temperature", [None, 0.0])
def test_heads_draft_and_verify_parity(dsv, name, cfg, changes, kind, temperature):
    cfg = wl.scaled(cfg, **changes)
    inp = wl.make_draft_inputs(cfg)
    Wg, Wc = wl.make_head_weights(cfg, kind)
    T = cfg.temperature if temperature is None else temperature
    g, out = _run(dsv, inp, kind, Wg, Wc, T)
    gx = npy(out["x"])
    head = oheads.Head(kind, Wg=wl.to_f64(Wg), Wc=None if Wc is None else wl.to_f64(Wc), bf16=cfg.dtype == "bf16")
    ref = oracle.draft_block(wl.to_f64(inp["U"]), wl.to_f64(inp["h"]), wl.to_f64(inp["W1"]), wl.to_f64(inp["W2"]),
                             wl.to_f64(inp["w"]), inp["bias"], npy(inp["x0"]), T, inp["seed"], forced_tokens=gx,
                             head=head)
    gE = wl.to_f64(out["E"])
    if cfg.dtype == "bf16":
        # one bf16 step (8 significant bits) of the larger magnitude: the float32 and
        # float64 values may round to neighbouring bf16 values
        mag = np.maximum(np.abs(gE), np.abs(ref["E"]))
        ulp = np.exp2(np.floor(np.log2(np.maximum(mag, 1e-30))) - 7)
        assert np.all(np.abs(gE - ref["E"]) <= ulp)
        assert np.mean(gE != ref["E"]) < 0.01
    else:
        assert np.all(np.abs(gE - ref["E"]) <= 1e-5 * np.abs(ref["E"]) + 1e-7)
    exempt = ref["margin"] < MARGIN
    assert not ((gx != ref["x"]) & ~exempt).any()
    same = gx == ref["x"]
    for k in ("c", "a"):
        assert np.abs(npy(out[k]) - ref[k]).max() <= FTOL[cfg.dtype], k
    for k in ("lse_d", "logp_d"):
        assert np.abs(npy(out[k]) - ref[k])[same].max(initial=0.0) <= FTOL["bf16"], k
    assert exempt.sum() <= max(2, 3 * cfg.B * cfg.gamma // 100)
    # verification of the GPU draft, with the GPU's E
    rng = np.random.default_rng(cfg.B + kind)
    ehead = dict(kind=kind, E=out["E"])
    for ell in (np.full(cfg.B, cfg.gamma), rng.integers(0, cfg.gamma + 1, cfg.B)):
        ell_t = torch.as_tensor(ell, dtype=torch.int32).cuda()
        v = dsv.dspark_verify_ex(g["t"], g["U"], g["W1"], g["W2"], g["x0"], out["x"], out["lse_d"], out["logp_d"],
                                 ell_t, T, inp["seed"], ehead)
        vref = oracle.verify_round(wl.to_f64(inp["t"]), wl.to_f64(inp["U"]), wl.to_f64(inp["W1"]),
                                   wl.to_f64(inp["W2"]), npy(inp["x0"]), gx, npy(out["lse_d"]), npy(out["logp_d"]),
                                   ell, T, inp["seed"], E=gE)
        compare_verify({k: npy(t) for k, t in v.items()}, vref)


def test_markov_kind_is_the_plain_call(dsv):
    cfg = wl.scaled(wl.QWEN3_8B, B=8, V=2048, H=32)
    inp = wl.make_draft_inputs(cfg)
    d = torch.device("cuda")
    g = {k: (v.to(d) if torch.is_tensor(v) else v) for k, v in inp.items()}
    a = dsv.dspark_draft_block(g["U"], g["h"], g["W1"], g["W2"], g["w"], 0.0, g["x0"], 0.7, 4)
    b = dsv.dspark_draft_block_ex(g["U"], g["h"], g["W1"], g["W2"], g["w"], 0.0, g["x0"], 0.7, 4, dict(kind=0))
    for k in ("x", "lse_d", "logp_d", "c", "a"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("kind", [1, 2], ids=["gated", "rnn"])
def test_heads_full_qwen3_size_sampled_requests(dsv, kind):
    """B = 64, gamma = 7, V = 151936, H = 4096, r = 256, bf16, T = 0.7: four sampled
    requests against the teacher-forced oracle (each keyed by its own index)."""
    cfg = wl.QWEN3_8B
    inp = wl.make_draft_inputs(cfg, device="cuda")
    Wg, Wc = wl.make_head_weights(cfg, kind, device="cuda")
    out = dsv.dspark_draft_block_ex(inp["U"], inp["h"], inp["W1"], inp["W2"], inp["w"], 0.0, inp["x0"],
                                    cfg.temperature, cfg.seed, dict(kind=kind, Wg=Wg, Wc=Wc))
    torch.cuda.synchronize()
    rows = np.array([0, 17, 40, 63])
    idx = torch.from_numpy(rows).cuda()
    gx = npy(out["x"])
    head = oheads.Head(kind, Wg=wl.to_f64(Wg), Wc=None if Wc is None else wl.to_f64(Wc), bf16=True)
    ref = oracle.draft_block(wl.to_f64(inp["U"][idx]), wl.to_f64(inp["h"][idx]), wl.to_f64(inp["W1"]),
                             wl.to_f64(inp["W2"]), wl.to_f64(inp["w"]), 0.0, npy(inp["x0"])[rows], cfg.temperature,
                             cfg.seed, forced_tokens=gx[rows], requests=rows, head=head)
    gE = wl.to_f64(out["E"][idx])
    mag = np.maximum(np.abs(gE), np.abs(ref["E"]))
    assert np.all(np.abs(gE - ref["E"]) <= np.exp2(np.floor(np.log2(np.maximum(mag, 1e-30))) - 7))
    exempt = ref["margin"] < MARGIN
    assert not ((gx[rows] != ref["x"]) & ~exempt).any()
    same = gx[rows] == ref["x"]
    for k in ("c", "a"):
        assert np.abs(npy(out[k])[rows] - ref[k]).max() <= FTOL["bf16"], k
    for k in ("lse_d", "logp_d"):
        assert np.abs(npy(out[k])[rows] - ref[k])[same].max(initial=0.0) <= FTOL["bf16"], k
