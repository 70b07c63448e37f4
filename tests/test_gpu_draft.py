"""GPU parity of dspark_draft_block against the oracle.

Integer outputs (tokens) must match exactly except decisions whose oracle
margin (top-2 gap of the perturbed logits over the vocabulary; greedy: of the
logits) is below 1e-4; those are counted and reported.  The oracle is run teacher-
forced on the GPU's tokens so every position is checked on its own.
Float outputs: |err| <= 2e-3 for bf16 inputs and 1e-5 for fp32 (c, a); the
same bars hold for lse_d / logp_d.  The tensor-core bias itself is checked
against a float64 matmul at 1e-5 relative.
"""
import numpy as np
import pytest
import torch

import oracle
from serving_draft_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

from tests.gpu_harness import MARGIN, FTOL, npy as _np, oracle_draft, compare_draft as compare  # noqa: E402


@pytest.fixture(scope="module")
def dsv():
    import serving_draft_verify_gb300 as m
    m.load()
    return m


def gpu_draft(dsv, inp, temperature=None, seed=None):
    from tests.gpu_harness import gpu_draft as run
    return {k: _np(v) for k, v in run(dsv, inp, temperature, seed).items()}


@pytest.mark.parametrize("B,V,r", [(1, 1024, 64), (20, 5000, 256), (130, 2048, 128), (300, 1000, 192)])
def test_tensor_core_logits(dsv, B, V, r):
    """z = U_k + W2 . W1[prev] from the tcgen05 path vs a float64 matmul."""
    g = torch.Generator().manual_seed(B + V + r)
    U = (torch.randn((B, V), generator=g) * 2).bfloat16()
    W1 = (torch.randn((V, r), generator=g) * 0.5).bfloat16()
    W2 = (torch.randn((V, r), generator=g) * 0.5).bfloat16()
    prev = torch.randint(0, V, (B,), generator=g).int()
    z, ws = dsv._binding.dspark_debug_draft_logits(U.cuda(), W1.cuda(), W2.cuda(), prev.cuda())
    assert dsv.workspace_status(ws) == 0
    ref = U.double() + W1.double()[prev.long()] @ W2.double().T
    err = (z.cpu().double() - ref).abs() / (1.0 + ref.abs())
    assert err.max().item() < 1e-5, err.max().item()


SMALL = [
    ("tiny", wl.TINY, {}),                                                        # fp32, CUDA-core path
    ("qwen_small", wl.QWEN3_8B, dict(B=20, V=5000, H=64)),                        # bf16, tensor cores
    ("two_mtiles", wl.DRAFT_27B, dict(B=130, gamma=3, V=2048, H=96)),            # ragged second M-tile
    ("r64_bf16", wl.QWEN3_8B, dict(B=9, gamma=5, V=1000, H=32, r=64)),
    ("r16_bf16", wl.QWEN3_8B, dict(B=5, gamma=4, V=1000, H=32, r=16)),            # CUDA-core, bf16
]


@pytest.mark.parametrize("name,cfg,changes", SMALL, ids=[c[0] for c in SMALL])
@pytest.mark.parametrize("temperature", [None, 0.0, 1.7])
def test_draft_parity_small(dsv, name, cfg, changes, temperature):
    cfg = wl.scaled(cfg, **changes)
    inp = wl.make_draft_inputs(cfg)
    gpu = gpu_draft(dsv, inp, temperature=temperature)
    ref = oracle_draft(inp, gpu["x"], temperature=temperature)
    exempt = compare(gpu, ref, cfg.dtype)
    assert exempt <= max(2, gpu["x"].size // 50)
    T = cfg.temperature if temperature is None else temperature
    if T == 0.0:
        assert np.all(gpu["lse_d"] == 0) and np.all(gpu["logp_d"] == 0)


def test_draft_strong_bias_chain(dsv):
    """Markov weights N(0, 0.5^2) make the bias O(1): tokens then depend on x_{k-1}."""
    cfg = wl.scaled(wl.QWEN3_8B, B=16, gamma=6, V=3000, H=32)
    inp = wl.make_draft_inputs(cfg)
    g = torch.Generator().manual_seed(5)
    inp["W1"] = (torch.randn(inp["W1"].shape, generator=g) * 0.5).bfloat16()
    inp["W2"] = (torch.randn(inp["W2"].shape, generator=g) * 0.5).bfloat16()
    for T in (0.7, 0.0):
        gpu = gpu_draft(dsv, inp, temperature=T)
        compare(gpu, oracle_draft(inp, gpu["x"], temperature=T), "bf16")


def test_draft_rejects_bad_anchor(dsv):
    cfg = wl.scaled(wl.QWEN3_8B, B=4, gamma=2, V=1024, H=16)
    inp = wl.make_draft_inputs(cfg)
    inp["x0"][2] = cfg.V + 5
    dev = torch.device("cuda")
    ws = torch.empty(dsv.load().dspark_draft_block_workspace_size(4, 2, 1024, 256), dtype=torch.uint8, device=dev)
    dsv.dspark_draft_block(inp["U"].to(dev), inp["h"].to(dev), inp["W1"].to(dev), inp["W2"].to(dev),
                           inp["w"].to(dev), 0.0, inp["x0"].to(dev), 1.0, 3, workspace=ws)
    assert dsv.workspace_status(ws) == 6


def full_size_rows(B, key):
    """Requests checked one by one at full size: every request up to B = 256; at
    B = 1024, 152 requests, one for every residue b mod 152 (the finalizing CTA of
    request b is b mod grid, grid = 152 SMs) spread over all eight 128-row M-tiles,
    and the last request."""
    if B <= 256:
        return np.arange(B)
    i = np.arange(152)
    rows = i + 152 * (i % 6)
    rows[-1] = B - 1
    return np.unique(rows)


@pytest.mark.parametrize("key,temperature", [("qwen3_8b", 0.7), ("qwen3_8b", 0.0), ("draft_27b", None),
                                             ("high_conc", None)])
def test_draft_full_size(dsv, key, temperature):
    """Full-size configs on the GPU; requests checked one by one (all of them up to
    B = 256, 152 covering every finalizing CTA at B = 1024)."""
    cfg = wl.DRAFT_CONFIGS[key]
    inp = wl.make_draft_inputs(cfg, device="cuda")
    gpu = gpu_draft(dsv, inp, temperature=temperature)
    rows = full_size_rows(cfg.B, key)
    ref = oracle_draft(inp, gpu["x"], temperature=temperature, rows=rows)
    exempt = compare(gpu, ref, cfg.dtype, rows=rows)
    assert exempt <= max(2, rows.size * cfg.gamma // 20)
    a = gpu["a"]
    assert np.all(np.diff(a, axis=1) <= 0) and np.all((a >= 0) & (a <= 1))
    del inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("key,changes,temperature", [
    ("qwen3_8b", dict(B=20, V=5000, H=64), 0.7),
    ("qwen3_8b", dict(B=20, V=5000, H=64), 0.0),
    ("draft_27b", dict(B=130, gamma=3, V=2048, H=96), 1.0),
    ("qwen3_8b", {}, 0.7),
])
def test_draft_one_launch_equals_per_position(dsv, key, changes, temperature):
    """The single cooperative launch (grid barriers between positions) and the
    per-position launches (engine kernel + winner kernel each) compute the same
    values in the same order: every output must agree bit for bit."""
    cfg = wl.scaled(wl.DRAFT_CONFIGS[key], **changes)
    inp = wl.make_draft_inputs(cfg, device="cuda")
    one = gpu_draft(dsv, inp, temperature=temperature)
    dsv._binding.force_phase_launches(True)
    try:
        per = gpu_draft(dsv, inp, temperature=temperature)
    finally:
        dsv._binding.force_phase_launches(False)
    for name in one:
        assert np.array_equal(one[name], per[name]), name
    del inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", [40, 5])                   # the tcgen05 engine; the small-batch path
@pytest.mark.parametrize("temperature", [None, 0.0])
def test_draft_reads_inputs_from_pinned_host_memory(dsv, temperature, B):
    """U, h and x0 in pinned host memory: the same outputs, bit for bit, as from device
    memory -- with U and h copied to the device by the call (dspark_draft_block), and
    with every input read by the kernels over the host link (the no-allocation entry
    point, which does not stage)."""
    cfg = wl.scaled(wl.QWEN3_8B, B=B, V=8192, H=64)
    inp = wl.make_draft_inputs(cfg)
    T = cfg.temperature if temperature is None else temperature
    g = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    a = dsv.dspark_draft_block(g["U"], g["h"], g["W1"], g["W2"], g["w"], 0.0, g["x0"], T, cfg.seed)
    host = {k: inp[k].clone().pin_memory() for k in ("U", "h", "x0")}
    staged0 = dsv._binding.staged_bytes()
    b = dsv.dspark_draft_block(host["U"], host["h"], g["W1"], g["W2"], g["w"], 0.0, host["x0"], T, cfg.seed)
    staged1 = dsv._binding.staged_bytes()
    out = {k: torch.empty_like(a[k]) for k in ("x", "lse_d", "logp_d", "c", "a")}
    c = dsv._binding.dspark_draft_block_noalloc(host["U"], host["h"], g["W1"], g["W2"], g["w"], 0.0, host["x0"], T,
                                               cfg.seed, out=out)
    torch.cuda.synchronize()
    # U and h went by copy engine in the first call, nothing in the no-allocation one
    assert staged1 - staged0 == (host["U"].numel() + host["h"].numel()) * 2
    assert dsv._binding.staged_bytes() == staged1
    for k in a:
        assert torch.equal(a[k], b[k]), k
        assert torch.equal(a[k], c[k]), k


def test_l2_residency_changes_no_result(dsv):
    """W2 held in L2 by a persisting access-policy window (opt-in): the same outputs,
    bit for bit, on both draft paths and the residual launch of verification; turning it
    off again restores the context's previous persisting-L2 limit."""
    for B in (40, 5):                                     # the tcgen05 engine; the small-batch path
        cfg = wl.scaled(wl.QWEN3_8B, B=B, V=8192, H=64)
        inp = wl.make_draft_inputs(cfg)
        g = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
        run = lambda: dsv.dspark_draft_block(g["U"], g["h"], g["W1"], g["W2"], g["w"], 0.0, g["x0"],  # noqa: E731
                                             cfg.temperature, cfg.seed)
        a = run()
        dsv.dspark_set_l2_residency(g["W2"].numel() * 2)
        try:
            b = run()
            torch.cuda.synchronize()
        finally:
            dsv.dspark_set_l2_residency(0)
        for k in a:
            assert torch.equal(a[k], b[k]), (B, k)
    # verification with many rejections (its residual launch reads W2 through the window)
    from tests.gpu_harness import gpu_draft as draft_run, gpu_verify
    cfg = wl.scaled(wl.QWEN3_8B, B=64, gamma=5, V=4096, H=32, target_noise=2.0)
    inp = wl.make_draft_inputs(cfg)
    d = draft_run(dsv, inp)
    ell = np.full(cfg.B, cfg.gamma)
    v0 = gpu_verify(dsv, inp, d, ell)
    dsv.dspark_set_l2_residency(inp["W2"].numel() * 2)
    try:
        v1 = gpu_verify(dsv, inp, d, ell)
    finally:
        dsv.dspark_set_l2_residency(0)
    for k in v0:
        assert np.array_equal(v0[k], v1[k]), k
    assert np.mean(v0["n_accept"] < cfg.gamma) > 0.3
