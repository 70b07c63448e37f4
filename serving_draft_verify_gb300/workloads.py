"""Seeded synthetic workloads for the draft / schedule / verify / TV path.

This module only draws inputs; it holds none of the method's arithmetic, and
it is the one module both the CUDA library's tests and the oracle's tests use.

The shapes follow the pages: Qwen3 vocabulary V = 151936, serving block
gamma = 7 (verify width 8 with the bonus row), Markov rank r = 256, hidden
size 4096 / 5120, confidence-head input H + r (model card, config.json
fields), training block 16.  Value recipe (same for every config unless the
config overrides it):

  U[b, k, :]   ~ N(0, 2^2) per logit, plus +8 on one uniformly drawn token of
                 the row with probability `peak_rate` (a peaked draft row);
  t[b, k, :]   = U[b, k, :] + N(0, target_noise^2) for k = 1..gamma, and row
                 gamma+1 is a fresh U-like row plus the same noise;
  W1, W2 [V, r], w [H + r] ~ N(0, 0.05^2);  bias = 0;  h ~ N(0, 1);
  x0[b]        ~ uniform over the vocabulary;
  SPS(N)       = N / (20 + 0.05 N), tabulated for N = 0..B (gamma + 1).

The high-concurrency config draws one peak rate per request from Beta(5, 2).
TV rows: d like U (peak rate 0.7), t = d + N(0, sigma_row^2) with sigma_row ~
U(0.1, 2.0) per row.  Training-loss rows add a uniform target token, a
N(0, 2^2) confidence logit and the block position (row mod 16) + 1.
"""
from dataclasses import dataclass, field, replace

import numpy as np
import torch


@dataclass(frozen=True)
class DraftConfig:
    name: str
    B: int
    gamma: int
    V: int
    H: int
    r: int
    dtype: str            # "f32" or "bf16"
    temperature: float
    seed: int
    peak_rate: float = 0.7
    target_noise: float = 0.5
    peak_rate_beta: tuple = field(default=None)   # (alpha, beta): per-request rate


@dataclass(frozen=True)
class TVConfig:
    name: str
    rows: int
    V: int
    dtype: str
    seed: int


TINY = DraftConfig("tiny fp32", B=4, gamma=7, V=1024, H=64, r=16, dtype="f32",
                   temperature=1.0, seed=0)
QWEN3_8B = DraftConfig("Qwen3-8B-shaped serving", B=64, gamma=7, V=151936, H=4096, r=256,
                       dtype="bf16", temperature=0.7, seed=1)
DRAFT_27B = DraftConfig("27B-draft-shaped serving", B=256, gamma=7, V=151936, H=5120, r=256,
                        dtype="bf16", temperature=1.0, seed=2, peak_rate=0.5, target_noise=1.0)
TV_TRAIN = TVConfig("training accept-rate TV", rows=16384, V=151936, dtype="bf16", seed=3)
HIGH_CONC = DraftConfig("high-concurrency scheduling", B=1024, gamma=16, V=151936, H=4096, r=256,
                        dtype="bf16", temperature=1.0, seed=4, peak_rate_beta=(5.0, 2.0))

DRAFT_CONFIGS = {"tiny": TINY, "qwen3_8b": QWEN3_8B, "draft_27b": DRAFT_27B, "high_conc": HIGH_CONC}


def scaled(cfg, **changes):
    """A copy of a config with some sizes changed (parity tests at small sizes)."""
    return replace(cfg, **changes)


def _torch_dtype(name):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _logit_rows(gen, n_rows, V, peak_rates, device, out_dtype, chunk=1 << 24):
    """n_rows rows of N(0, 4) logits with +8 on one random token of a row with
    probability peak_rates[row]; drawn in float32 and cast."""
    out = torch.empty((n_rows, V), dtype=out_dtype, device=device)
    rows_per_chunk = max(1, chunk // V)
    for r0 in range(0, n_rows, rows_per_chunk):
        r1 = min(n_rows, r0 + rows_per_chunk)
        blk = torch.randn((r1 - r0, V), generator=gen, device=device) * 2.0
        coin = torch.rand((r1 - r0,), generator=gen, device=device)
        tok = torch.randint(0, V, (r1 - r0,), generator=gen, device=device)
        hit = coin < peak_rates[r0:r1].to(device)
        blk[torch.arange(r1 - r0, device=device)[hit], tok[hit]] += 8.0
        out[r0:r1] = blk.to(out_dtype)
    return out


def make_draft_inputs(cfg, device="cpu"):
    """All inputs of one draft -> schedule -> verify round, as torch tensors on
    `device` (float inputs in the config's dtype; x0 int32; sps float64)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed)
    rng = np.random.default_rng(cfg.seed)
    dt = _torch_dtype(cfg.dtype)
    B, G, V, H, r = cfg.B, cfg.gamma, cfg.V, cfg.H, cfg.r
    if cfg.peak_rate_beta is not None:
        rate_b = torch.from_numpy(rng.beta(*cfg.peak_rate_beta, size=B)).float()
    else:
        rate_b = torch.full((B,), float(cfg.peak_rate))
    U = _logit_rows(gen, B * G, V, rate_b.repeat_interleave(G), dev, dt).view(B, G, V)
    bonus = _logit_rows(gen, B, V, rate_b, dev, torch.float32)
    t = torch.empty((B, G + 1, V), dtype=dt, device=dev)
    for b0 in range(0, B, max(1, (1 << 24) // (G * V))):
        b1 = min(B, b0 + max(1, (1 << 24) // (G * V)))
        noise = torch.randn((b1 - b0, G + 1, V), generator=gen, device=dev) * cfg.target_noise
        base = torch.cat([U[b0:b1].float(), bonus[b0:b1, None, :]], dim=1)
        t[b0:b1] = (base + noise).to(dt)
    W1 = (torch.randn((V, r), generator=gen, device=dev) * 0.05).to(dt)
    W2 = (torch.randn((V, r), generator=gen, device=dev) * 0.05).to(dt)
    w = (torch.randn((H + r,), generator=gen, device=dev) * 0.05).to(dt)
    h = torch.randn((B, G, H), generator=gen, device=dev).to(dt)
    x0 = torch.randint(0, V, (B,), generator=gen, device=dev).to(torch.int32)
    N = torch.arange(B * (G + 1) + 1, dtype=torch.float64)
    sps = (N / (20.0 + 0.05 * N)).to(dev)
    return dict(U=U, t=t, W1=W1, W2=W2, w=w, bias=0.0, h=h, x0=x0, sps=sps,
                temperature=cfg.temperature, seed=cfg.seed)


def make_tv_inputs(cfg, device="cpu", rows=None):
    """(d, t) [rows, V] in the config's dtype: d like U, t = d + N(0, sigma_row^2)."""
    dev = torch.device(device)
    n = cfg.rows if rows is None else rows
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed)
    dt = _torch_dtype(cfg.dtype)
    d = _logit_rows(gen, n, cfg.V, torch.full((n,), 0.7), dev, dt)
    sigma = 0.1 + 1.9 * torch.rand((n,), generator=gen, device=dev)
    t = torch.empty_like(d)
    rows_per_chunk = max(1, (1 << 24) // cfg.V)
    for r0 in range(0, n, rows_per_chunk):
        r1 = min(n, r0 + rows_per_chunk)
        noise = torch.randn((r1 - r0, cfg.V), generator=gen, device=dev) * sigma[r0:r1, None]
        t[r0:r1] = (d[r0:r1].float() + noise).to(dt)
    return d, t


def make_round_pool(cfg, pool, device="cpu"):
    """A pool of `pool` synthetic rounds for multi-round decoding: slot 0 is
    make_draft_inputs(cfg); slot p > 0 draws U, h and t the same way from seed
    cfg.seed + 7919 p.  W1, W2, w, bias, x0 and the SPS table are slot 0's.
    Returns dict U [P, B, gamma, V], h [P, B, gamma, H], t [P, B, gamma+1, V] and
    the shared tensors."""
    base = make_draft_inputs(cfg, device=device)
    Us, hs, ts = [base["U"]], [base["h"]], [base["t"]]
    for p in range(1, pool):
        g = make_draft_inputs(replace(cfg, seed=cfg.seed + 7919 * p), device=device)
        Us.append(g["U"])
        hs.append(g["h"])
        ts.append(g["t"])
        del g
    out = dict(base)
    out["U"], out["h"], out["t"] = torch.stack(Us), torch.stack(hs), torch.stack(ts)
    return out


def make_head_weights(cfg, kind, device="cpu"):
    """Weights of a gated (kind 1) or recurrent (kind 2) sequential head in the
    config's dtype: Wg [r, H + r] (gated) or Wg, Wc [r, 2r + H] (recurrent), each
    entry ~ N(0, 1 / (row length)) so that a gate's pre-activation is O(1)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed + 31 * kind)
    dt = _torch_dtype(cfg.dtype)
    ld = cfg.H + cfg.r if kind == 1 else 2 * cfg.r + cfg.H
    Wg = (torch.randn((cfg.r, ld), generator=gen, device=dev) / ld ** 0.5).to(dt)
    Wc = (torch.randn((cfg.r, ld), generator=gen, device=dev) / ld ** 0.5).to(dt) if kind == 2 else None
    return Wg, Wc


LOSS_BLOCK = 16   # training block size: rows are (sequence, anchor, block position k)


def make_loss_inputs(cfg, device="cpu", rows=None):
    """The training loss's per-row inputs beside make_tv_inputs' (d, t):
    target [rows] int32 ~ uniform over the vocabulary, conf_logit [rows]
    float32 ~ N(0, 2^2) (the confidence head's logit), and the block position
    k [rows] int64 = row mod 16 + 1 (rows are sequence x anchor x position)."""
    dev = torch.device(device)
    n = cfg.rows if rows is None else rows
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed + 1000)
    target = torch.randint(0, cfg.V, (n,), generator=gen, device=dev).to(torch.int32)
    conf_logit = torch.randn((n,), generator=gen, device=dev) * 2.0
    k = torch.arange(n, device=dev) % LOSS_BLOCK + 1
    return target, conf_logit, k


def to_f64(x):
    """Exact float64 numpy copy of a float tensor (bf16 and f32 widen exactly)."""
    return x.detach().to("cpu").to(torch.float64).numpy()
