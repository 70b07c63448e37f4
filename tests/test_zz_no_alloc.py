"""dspark_draft_block_noalloc: the draft block for callers that cannot allocate
device memory (hosts that own all GPU memory in their own pool and forbid
cudaMalloc from plug-in code).  It is called through the C ABI three times in a
row, with different inputs (the last two of equal shape), and each result is
checked against dspark_draft_block on the same inputs: the same kernels run on
the same data, so every output must agree bit for bit.  This file is collected
last."""
import numpy as np
import pytest
import torch

from serving_draft_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _out(B, G):
    dev = torch.device("cuda")
    return dict(x=torch.full((B, G), -7, dtype=torch.int32, device=dev),
                **{k: torch.full((B, G), float("nan"), dtype=torch.float32, device=dev)
                   for k in ("lse_d", "logp_d", "c", "a")})


def test_noalloc_matches_draft_block_twice():
    import serving_draft_verify_gb300 as dsv
    dsv.load()
    cases = [(wl.scaled(wl.QWEN3_8B, B=40, gamma=5, V=5000, H=64), 0.7, 11),
             (wl.scaled(wl.QWEN3_8B, B=24, gamma=7, V=3000, H=32, seed=5), 1.3, 12),
             # the same B and gamma as the call before, other inputs and seed: every slot of
             # the shared scratch that call wrote is reused
             (wl.scaled(wl.QWEN3_8B, B=24, gamma=7, V=3000, H=32, seed=9), 0.9, 13)]
    runs = []
    for cfg, T, seed in cases:        # two no-allocation calls in a row, sharing the internal scratch
        inp = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in wl.make_draft_inputs(cfg).items()}
        args = (inp["U"], inp["h"], inp["W1"], inp["W2"], inp["w"], 0.0, inp["x0"], T, seed)
        runs.append((args, dsv._binding.dspark_draft_block_noalloc(*args, out=_out(cfg.B, cfg.gamma))))
    torch.cuda.synchronize()
    for args, got in runs:
        ref = dsv.dspark_draft_block(*args)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: every output bit for bit
        for k in ("x", "lse_d", "logp_d", "c", "a"):
            assert torch.equal(got[k], ref[k]), k


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import serving_draft_verify_gb300 as dsv
    cfg = wl.scaled(wl.QWEN3_8B, B=1024, gamma=16, V=1024, H=8)
    dev = torch.device("cuda")
    U = torch.zeros((cfg.B, cfg.gamma, cfg.V), dtype=torch.bfloat16, device=dev)
    h = torch.zeros((cfg.B, cfg.gamma, cfg.H), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((cfg.V, cfg.r), dtype=torch.bfloat16, device=dev)
    w = torch.zeros(cfg.H + cfg.r, dtype=torch.bfloat16, device=dev)
    x0 = torch.zeros(cfg.B, dtype=torch.int32, device=dev)
    with pytest.raises(dsv.DSparkError) as e:
        dsv._binding.dspark_draft_block_noalloc(U, h, W, W, w, 0.0, x0, 1.0, 1, out=_out(cfg.B, cfg.gamma))
    assert e.value.status == 2     # DSPARK_ERR_UNSUPPORTED
