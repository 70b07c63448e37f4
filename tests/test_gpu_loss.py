"""GPU parity of dspark_training_loss against the oracle (float64 loss and
gradient).

Tolerances (the parity bar: 2e-3 for bf16 inputs, 1e-5 for fp32), applied
relative to each quantity's scale: ce and the row totals relative to
max(1, |value|); c*, bce and grad_conf absolute; grad_d element-wise against
the element's own terms, omega (a_ce (p_d + [v = target]) + a_l1 p_d), with
bf16 outputs also allowed their rounding (2^-8 relative).

sign(p_d - p_t) decides a term of the gradient.  Where p_d and p_t agree to
within float32 error the kernel's sign may differ from float64's, and through
sum_u p_d(u) sgn_u the choice reaches the whole row: a row with such ties must
match the gradient of one valid assignment of signs to them."""
import itertools

import numpy as np
import pytest
import torch

import oracle
from oracle import loss as oloss
from serving_draft_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-3, torch.float32: 1e-5}
GRAD_REL = {torch.bfloat16: 2 ** -8 + 1e-4, torch.float32: 2e-5}


@pytest.fixture(scope="module")
def dsv():
    import serving_draft_verify_gb300 as m
    m.load()
    return m


def _omega(k):
    w = oloss.position_weights(np.asarray(k))
    return torch.from_numpy(w / w.sum()).float()


def _run(dsv, d, t, target, s, omega, grad=True, **kw):
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    out = dsv.dspark_training_loss(d.cuda(), t.cuda(), target.cuda(), s.cuda(), omega.cuda(), grad=grad,
                                   workspace=ws, **kw)
    assert dsv.workspace_status(ws) == 0
    return {k: v.cpu() for k, v in out.items()}


def _check_rows(got, want, dtype):
    tol = TOL[dtype]
    row = got["row"].double().numpy()
    ce, cs, bce, tot = row.T
    assert np.all(np.abs(ce - want["ce"]) <= tol * np.maximum(1.0, np.abs(want["ce"]))), \
        np.max(np.abs(ce - want["ce"]))
    assert np.max(np.abs(cs - want["c_star"])) <= tol
    assert np.max(np.abs(bce - want["bce"])) <= tol * np.maximum(1.0, np.abs(want["bce"])).max()
    assert np.all(np.abs(tot - want["row"]) <= tol * np.maximum(1.0, np.abs(want["row"])))
    L = float(got["loss"][0])
    assert abs(L - want["loss"]) <= tol * max(1.0, abs(want["loss"])), (L, want["loss"])


def _check_grad(got_gd, got_gc, d64, t64, target, s, omega, dtype, kw=None):
    kw = kw or {}
    a_ce = kw.get("alpha_ce", oloss.ALPHA_CE)
    a_l1 = kw.get("alpha_l1", oloss.ALPHA_L1)
    a_conf = kw.get("alpha_conf", oloss.ALPHA_CONF)
    want_gd, want_gc = oloss.dspark_loss_grad(d64, t64, target, s, omega, a_ce, a_l1, a_conf)
    assert np.max(np.abs(got_gc - want_gc)) <= TOL[dtype]
    p_d, p_t = oracle.tv.softmax(d64), oracle.tv.softmax(t64)
    R = d64.shape[0]
    onehot = np.zeros_like(d64)
    onehot[np.arange(R), target] = 1.0
    om = np.asarray(omega, dtype=np.float64)[:, None]
    scale = np.abs(om) * (abs(a_ce) * (p_d + onehot) + abs(a_l1) * p_d) + 1e-30
    err = np.abs(got_gd - want_gd)
    bad = err > GRAD_REL[dtype] * scale
    # near ties of p_d and p_t (|p_d - p_t| within float32 error of the kernel's
    # decision): the kernel may take any sign there, and through the row's
    # sum_u p_d(u) sgn_u that choice moves every element of the row.  The kernel
    # decides by d_v - t_v against L_d - L_t, so tied elements with the same
    # d_v - t_v share one decision (with bf16 inputs whole runs do: t rounds to
    # d's value where the noise is small).  A row with ties passes if some
    # assignment of signs to its groups of tied elements reproduces it: every
    # assignment for at most 4 groups, else one sign for all of them.
    tie = np.abs(p_d - p_t) <= 1e-5 * np.maximum(p_d, p_t)
    sgn = np.sign(p_d - p_t)
    tol = GRAD_REL[dtype] * scale
    for r in np.nonzero(bad.any(axis=1))[0]:
        T = np.nonzero(tie[r])[0]
        assert T.size > 0, ("row", r, np.nonzero(bad[r])[0][:5], err[r][bad[r]][:5], scale[r][bad[r]][:5])
        _, grp = np.unique(d64[r, T] - t64[r, T], return_inverse=True)
        ng = int(grp.max()) + 1
        if ng <= 4:
            choices = itertools.product((-1.0, 0.0, 1.0), repeat=ng)
        else:
            choices = [(c,) * ng for c in (-1.0, 0.0, 1.0)]
        ok = False
        for ch in choices:
            sg = sgn[r].copy()
            sg[T] = np.asarray(ch)[grp]
            sb = np.sum(p_d[r] * sg)
            g = om[r] * (a_ce * (p_d[r] - onehot[r]) + a_l1 * 0.5 * p_d[r] * (sg - sb))
            if np.all(np.abs(got_gd[r] - g) <= tol[r]):
                ok = True
                break
        assert ok, ("row", r, T[:8], np.nonzero(bad[r])[0][:5], err[r][bad[r]][:5], scale[r][bad[r]][:5])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V", [8, 1024, 5000, 151936, 262144])
def test_loss_parity_seeded_rows(dsv, dtype, V):
    cfg = wl.scaled(wl.TV_TRAIN, V=V)
    rows = 37
    d, t = wl.make_tv_inputs(cfg, rows=rows)
    target, s, k = wl.make_loss_inputs(cfg, rows=rows)
    d, t = d.to(dtype), t.to(dtype)
    omega = _omega(k)
    got = _run(dsv, d, t, target, s, omega)
    d64, t64 = wl.to_f64(d), wl.to_f64(t)
    tg, s64, om64 = target.numpy(), s.double().numpy(), omega.double().numpy()
    want = oloss.dspark_loss(d64, t64, tg, s64, om64)
    _check_rows(got, want, dtype)
    _check_grad(got["grad_d"].double().numpy(), got["grad_conf"].double().numpy(), d64, t64, tg, s64, om64,
                dtype)


def test_loss_weights_targets_at_slice_edges_and_no_grad(dsv):
    """Other alpha weights, negative omega, targets at every CTA slice boundary
    of V = 1024 (slices of 128), and the call without gradient outputs."""
    V, dtype = 1024, torch.float32
    cfg = wl.scaled(wl.TV_TRAIN, V=V)
    d, t = wl.make_tv_inputs(cfg, rows=20)
    d, t = d.to(dtype), t.to(dtype)
    target = torch.tensor([0, 127, 128, 255, 256, 511, 512, 767, 768, 895, 896, 1023] + [5] * 8, dtype=torch.int32)
    s = torch.linspace(-30, 30, 20)
    omega = torch.linspace(-1.0, 2.0, 20)
    kw = dict(alpha_ce=0.7, alpha_l1=-0.25, alpha_conf=2.5)
    got = _run(dsv, d, t, target, s, omega, **kw)
    d64, t64 = wl.to_f64(d), wl.to_f64(t)
    want = oloss.dspark_loss(d64, t64, target.numpy(), s.double().numpy(), omega.double().numpy(), **kw)
    _check_rows(got, want, dtype)
    _check_grad(got["grad_d"].double().numpy(), got["grad_conf"].double().numpy(), d64, t64, target.numpy(),
                s.double().numpy(), omega.double().numpy(), dtype, kw)
    nog = _run(dsv, d, t, target, s, omega, grad=False, **kw)
    assert set(nog) == {"row", "loss"}
    assert torch.equal(nog["row"], got["row"]) and torch.equal(nog["loss"], got["loss"])


def test_loss_degenerate_rows(dsv):
    """d = t (c* = 1, the L1 gradient vanishes), disjoint supports (c* = 0),
    a single finite logit per row (ce = 0 at that target)."""
    V = 4096
    rng = np.random.default_rng(5)
    d = torch.from_numpy(rng.normal(0, 2, (4, V))).float()
    t = d.clone()
    d[1] = -1e30
    d[1, : V // 2] = 0.0
    t[1] = -1e30
    t[1, V // 2:] = 0.0
    d[2] = float("-inf")
    d[2, 100] = 1.0
    t[2] = float("-inf")
    t[2, 100] = -4.0
    target = torch.tensor([9, 3, 100, 4000], dtype=torch.int32)
    s = torch.tensor([0.5, -2.0, 3.0, 0.0])
    omega = torch.ones(4)
    for dt in (torch.float32, torch.bfloat16):
        got = _run(dsv, d.to(dt), t.to(dt), target, s, omega)
        row = got["row"].double().numpy()
        assert abs(row[0, 1] - 1.0) < 1e-5 and row[1, 1] == 0.0 and abs(row[2, 1] - 1.0) < 1e-6
        assert abs(row[2, 0]) < 1e-6
        gd = got["grad_d"].double().numpy()
        p0 = oracle.tv.softmax(wl.to_f64(d.to(dt))[0:1])[0]
        g0 = oloss.ALPHA_CE * (p0 - np.eye(V)[9])            # row 0: the CE term alone
        assert np.max(np.abs(gd[0] - g0)) <= GRAD_REL[dt] * oloss.ALPHA_CE + 1e-7
        assert np.all(gd[2, np.arange(V) != 100] == 0.0)


def test_loss_empty_deterministic_and_bad_target(dsv):
    d = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(0, device="cuda")
    out = dsv.dspark_training_loss(d, d, torch.zeros(0, dtype=torch.int32, device="cuda"), z, z)
    assert float(out["loss"][0]) == 0.0
    cfg = wl.scaled(wl.TV_TRAIN, V=151936)
    d, t = wl.make_tv_inputs(cfg, rows=300, device="cuda")
    target, s, k = wl.make_loss_inputs(cfg, rows=300, device="cuda")
    omega = _omega(k.cpu()).cuda()
    a = dsv.dspark_training_loss(d, t, target, s, omega)
    b = dsv.dspark_training_loss(d, t, target, s, omega)
    assert torch.equal(a["loss"], b["loss"]) and torch.equal(a["grad_d"], b["grad_d"])
    assert abs(float(a["loss"][0]) - float(a["row"][:, 3].double().sum())) <= 1e-5 * abs(float(a["loss"][0]))
    bad = target.clone()
    bad[7] = cfg.V
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    dsv.dspark_training_loss(d, t, bad, s, omega, workspace=ws)
    assert dsv.workspace_status(ws) == 6          # DSPARK_ERR_DEVICE_CHECK


def test_loss_full_training_size_sampled_rows(dsv):
    """16384 x 151936 bf16 rows (the training workload, one launch as the
    benchmark times it): sampled rows against the oracle, and the loss against
    the float64 sum of the row totals."""
    cfg = wl.TV_TRAIN
    d, t = wl.make_tv_inputs(cfg, device="cuda")
    target, s, k = wl.make_loss_inputs(cfg, device="cuda")
    omega = _omega(k.cpu()).cuda()
    out = dsv.dspark_training_loss(d, t, target, s, omega)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 15, 16, 4097, 9999, cfg.rows - 2, cfg.rows - 1])
    idx = torch.from_numpy(rows).cuda()
    d64, t64 = wl.to_f64(d[idx]), wl.to_f64(t[idx])
    tg, s64, om64 = target[idx].cpu().numpy(), s[idx].double().cpu().numpy(), omega[idx].double().cpu().numpy()
    want = oloss.dspark_loss(d64, t64, tg, s64, om64)
    got = {"row": out["row"][idx].cpu(), "loss": torch.tensor([want["loss"]], dtype=torch.float32)}
    _check_rows(got, want, torch.bfloat16)
    _check_grad(out["grad_d"][idx].double().cpu().numpy(), out["grad_conf"][idx].double().cpu().numpy(),
                d64, t64, tg, s64, om64, torch.bfloat16)
    tot = out["row"][:, 3].double().sum().item()
    assert abs(float(out["loss"][0]) - tot) <= 1e-5 * max(1.0, abs(tot))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V", [1024, 151936])
def test_gradient_signs_exact_beyond_the_tie_band(dsv, dtype, V):
    """The tie band of _check_grad (|p_d - p_t| <= 1e-5 max(p_d, p_t)) is no wider than
    needed: rows whose decisive log ratios sit just outside it must get every sign of
    sign(p_d - p_t) exactly as float64 does, with no tie allowance at all.

    Row: d = 0 everywhere; t = +h on the first half of the vocabulary and -h on the
    second.  Then L_d - L_t = -ln cosh h, and every token's |ln(p_d / p_t)| is
    h -/+ ln cosh h, about h: margins from 1.2e-5 (just beyond the band) to 1e-3.
    A wrong sign on either half moves sum_u p_d(u) sgn_u by about 1, and with it
    every element of the row's gradient by about half its scale, far beyond the
    tolerance.  The kernel's own sums here are of exact terms (ones, and e^(+-h)
    whose total differs from V by less than float32 resolves), so its decision
    error is far below h and these rows must pass the exact check."""
    hs = [1.2e-5, 2e-5, 5e-5, 1e-4, 1e-3]
    rows = len(hs)
    d = np.zeros((rows, V), np.float64)
    t = np.zeros((rows, V), np.float64)
    for r, h in enumerate(hs):
        h = float(torch.tensor(h, dtype=dtype).double())   # representable in the input dtype
        t[r, :V // 2] = h
        t[r, V // 2:] = -h
    dt_, tt_ = torch.from_numpy(d).to(dtype), torch.from_numpy(t).to(dtype)
    target = torch.tensor([(r * 7919 + 13) % V for r in range(rows)], dtype=torch.int32)
    s = torch.linspace(-1.0, 1.0, rows)
    omega = torch.full((rows,), 1.0 / rows)
    got = _run(dsv, dt_, tt_, target, s, omega)
    d64, t64 = wl.to_f64(dt_), wl.to_f64(tt_)
    p_d, p_t = oracle.tv.softmax(d64), oracle.tv.softmax(t64)
    lr = np.abs(np.log(p_d / p_t))
    assert np.all(lr > 1.1e-5), lr.min()                  # every token beyond the band
    want_gd, _ = oloss.dspark_loss_grad(d64, t64, target.numpy(), s.double().numpy(), omega.double().numpy())
    onehot = np.zeros_like(d64)
    onehot[np.arange(rows), target.numpy()] = 1.0
    om = omega.double().numpy()[:, None]
    scale = np.abs(om) * (abs(oloss.ALPHA_CE) * (p_d + onehot) + abs(oloss.ALPHA_L1) * p_d) + 1e-30
    err = np.abs(got["grad_d"].double().numpy() - want_gd)
    assert np.all(err <= GRAD_REL[dtype] * scale), np.max(err / scale)
