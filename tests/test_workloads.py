"""The seeded input generators follow the stated recipe: logits N(0, 2^2) with
a +8 peak on one token of a row at the configured rate, target rows = draft
rows + N(0, sigma^2), weights N(0, 0.05^2), the SPS table N / (20 + 0.05 N),
TV rows with sigma_row ~ U(0.1, 2.0), and the training rows' block positions."""
import numpy as np
import torch

from serving_draft_verify_gb300 import workloads as wl


def _small(**kw):
    base = dict(B=64, gamma=7, V=512, H=32, r=16, dtype="f32")
    base.update(kw)
    return wl.scaled(wl.TINY, **base)


def test_shapes_dtypes_and_tables():
    cfg = _small()
    g = wl.make_draft_inputs(cfg)
    B, G, V, H, r = cfg.B, cfg.gamma, cfg.V, cfg.H, cfg.r
    assert g["U"].shape == (B, G, V) and g["t"].shape == (B, G + 1, V)
    assert g["W1"].shape == (V, r) and g["W2"].shape == (V, r) and g["w"].shape == (H + r,)
    assert g["h"].shape == (B, G, H) and g["x0"].shape == (B,) and g["x0"].dtype == torch.int32
    assert int(g["x0"].min()) >= 0 and int(g["x0"].max()) < V
    N = np.arange(B * (G + 1) + 1, dtype=np.float64)
    assert np.array_equal(g["sps"].numpy(), N / (20.0 + 0.05 * N))
    gb = wl.make_draft_inputs(wl.scaled(cfg, dtype="bf16"))
    assert gb["U"].dtype == torch.bfloat16 and gb["t"].dtype == torch.bfloat16


def test_same_seed_same_inputs():
    a, b = wl.make_draft_inputs(_small()), wl.make_draft_inputs(_small())
    for k in ("U", "t", "W1", "W2", "w", "h", "x0"):
        assert torch.equal(a[k], b[k]), k
    c = wl.make_draft_inputs(_small(seed=5))
    assert not torch.equal(a["U"], c["U"])


def test_peak_is_plus_eight_on_one_token_at_the_rate():
    # the coin and the token are drawn whatever the rate: rate 1 minus rate 0 is the peak itself
    hi = wl.make_draft_inputs(_small(peak_rate=1.0))["U"].reshape(-1, 512)
    lo = wl.make_draft_inputs(_small(peak_rate=0.0))["U"].reshape(-1, 512)
    diff = (hi - lo).numpy()
    peak = np.abs(diff - 8.0) < 1e-5                           # (x + 8) - x: 8 up to float32 rounding
    assert np.all(peak | (diff == 0.0))
    assert np.all(peak.sum(axis=1) == 1)                       # exactly one token per row
    # the peaked token is uniform over the vocabulary (chi-square over 8 bins)
    bins = np.bincount(np.argmax(diff, axis=1) * 8 // 512, minlength=8)
    exp = diff.shape[0] / 8
    assert ((bins - exp) ** 2 / exp).sum() < 24.3             # chi2(7) 0.999 quantile
    # at rate 0.7 the peaked rows are a binomial fraction
    mid = wl.make_draft_inputs(_small(peak_rate=0.7, B=512))["U"].reshape(-1, 512)
    base = wl.make_draft_inputs(_small(peak_rate=0.0, B=512))["U"].reshape(-1, 512)
    frac = float(((mid - base - 8.0).abs() < 1e-5).any(dim=1).float().mean())
    n = mid.shape[0]
    assert abs(frac - 0.7) < 4 * (0.7 * 0.3 / n) ** 0.5
    # the rest is N(0, 2^2)
    x = lo.numpy().ravel()
    assert abs(x.mean()) < 4 * 2.0 / len(x) ** 0.5
    assert abs(x.std() - 2.0) < 0.02


def test_target_rows_are_draft_rows_plus_noise():
    for sigma in (0.5, 1.0):
        cfg = _small(target_noise=sigma)
        g = wl.make_draft_inputs(cfg)
        noise = (g["t"][:, :cfg.gamma] - g["U"]).numpy().ravel()   # float32: the noise up to one rounding
        assert abs(noise.mean()) < 4 * sigma / len(noise) ** 0.5
        assert abs(noise.std() / sigma - 1.0) < 0.01
        # the bonus row is a fresh U-like row plus noise: spread sqrt(4 + sigma^2), uncorrelated with U_gamma
        bonus = g["t"][:, cfg.gamma].numpy().ravel()
        assert abs(bonus.std() - (4.0 + sigma ** 2) ** 0.5) < 0.05
        last = g["U"][:, cfg.gamma - 1].numpy().ravel()
        assert abs(np.corrcoef(bonus, last)[0, 1]) < 0.02


def test_weights_and_hidden_states():
    g = wl.make_draft_inputs(_small(V=4096, r=64, H=512))
    for k, s in (("W1", 0.05), ("W2", 0.05), ("h", 1.0)):
        x = g[k].numpy().ravel()
        assert abs(x.std() / s - 1.0) < 0.02, k
    assert abs(g["w"].numpy().std() / 0.05 - 1.0) < 0.1


def test_per_request_beta_rates():
    cfg = wl.scaled(wl.HIGH_CONC, V=64, H=8, r=16, dtype="f32")
    hi = wl.make_draft_inputs(cfg)["U"]
    lo = wl.make_draft_inputs(wl.scaled(cfg, peak_rate_beta=None, peak_rate=0.0))["U"]
    peaked = ((hi - lo - 8.0).abs() < 1e-5).any(dim=2).float()   # [B, gamma]
    rate = peaked.mean(dim=1).numpy()                            # per request, gamma = 16 draws
    # Beta(5, 2): mean 5/7, variance 5*2/(7^2*8); the per-request fraction adds binomial noise
    assert abs(rate.mean() - 5 / 7) < 0.02
    var_beta = 10 / (49 * 8)
    var_expected = var_beta + (5 / 7 - (var_beta + (5 / 7) ** 2)) / 16
    assert 0.7 * var_expected < rate.var() < 1.3 * var_expected


def test_tv_and_loss_rows():
    cfg = wl.scaled(wl.TV_TRAIN, V=2048, dtype="f32")
    d, t = wl.make_tv_inputs(cfg, rows=400)
    sig = (t - d).std(dim=1).numpy()
    rel = 4 / (2 * cfg.V) ** 0.5                                 # four standard errors of a sample std
    assert sig.min() > 0.1 * (1 - rel) and sig.max() < 2.0 * (1 + rel)
    # sigma_row ~ U(0.1, 2.0): mean 1.05, spread 1.9 / sqrt(12)
    assert abs(sig.mean() - 1.05) < 4 * (1.9 / 12 ** 0.5) / 400 ** 0.5
    target, conf, k = wl.make_loss_inputs(cfg, rows=4096)
    assert target.dtype == torch.int32 and int(target.min()) >= 0 and int(target.max()) < cfg.V
    assert torch.equal(k, torch.arange(4096) % wl.LOSS_BLOCK + 1)
    assert abs(float(conf.std()) - 2.0) < 0.1
