"""Helpers shared by the GPU parity tests: run the library on seeded inputs
and the oracle on the same inputs (teacher-forced / stage-isolated)."""
import numpy as np
import torch

import oracle
from serving_draft_verify_gb300 import workloads as wl

MARGIN = 1e-4
FTOL = {"bf16": 2e-3, "f32": 1e-5}

# Exempt decisions (oracle margin below MARGIN) seen by the parity tests of this
# session: (test id, kind, exempt, decisions checked).  conftest prints them in
# the terminal summary.
EXEMPT = []


def report_exempt(kind, exempt, checked):
    import os
    EXEMPT.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], kind, int(exempt), int(checked)))


def npy(t):
    return t.detach().cpu().numpy()


def dev_inputs(inp):
    d = torch.device("cuda")
    return {k: (v.to(d) if torch.is_tensor(v) else v) for k, v in inp.items()}


def gpu_draft(dsv, inp, temperature=None, seed=None):
    g = dev_inputs(inp)
    T = inp["temperature"] if temperature is None else temperature
    s = inp["seed"] if seed is None else seed
    B, G, V = g["U"].shape
    ws = torch.empty(dsv.load().dspark_draft_block_workspace_size(B, G, V, g["W1"].shape[1]),
                     dtype=torch.uint8, device="cuda")
    out = dsv.dspark_draft_block(g["U"], g["h"], g["W1"], g["W2"], g["w"], inp["bias"], g["x0"], T, s,
                                 workspace=ws)
    assert dsv.workspace_status(ws) == 0
    return out


def gpu_verify(dsv, inp, draft_out, ell, temperature=None, seed=None):
    g = dev_inputs(inp)
    T = inp["temperature"] if temperature is None else temperature
    s = inp["seed"] if seed is None else seed
    B, G, V = g["U"].shape
    ws = torch.empty(dsv.load().dspark_verify_workspace_size(B, G, V, g["W1"].shape[1]),
                     dtype=torch.uint8, device="cuda")
    ell = torch.as_tensor(ell, dtype=torch.int32).cuda()
    out = dsv.dspark_verify(g["t"], g["U"], g["W1"], g["W2"], g["x0"], draft_out["x"], draft_out["lse_d"],
                            draft_out["logp_d"], ell, T, s, workspace=ws)
    assert dsv.workspace_status(ws) == 0
    return {k: npy(v) for k, v in out.items()}


def oracle_draft(inp, gpu_x, temperature=None, seed=None, rows=None):
    """Teacher-forced oracle for the listed requests, each keyed by its own index."""
    rows = np.arange(inp["U"].shape[0]) if rows is None else np.asarray(rows)
    T = inp["temperature"] if temperature is None else temperature
    s = inp["seed"] if seed is None else seed
    idx = torch.from_numpy(rows).to(inp["U"].device)
    return oracle.draft_block(wl.to_f64(inp["U"][idx]), wl.to_f64(inp["h"][idx]), wl.to_f64(inp["W1"]),
                              wl.to_f64(inp["W2"]), wl.to_f64(inp["w"]), inp["bias"], npy(inp["x0"])[rows], T, s,
                              forced_tokens=gpu_x[rows], requests=rows)


def oracle_verify(inp, draft_np, ell, temperature=None, seed=None, rows=None):
    """Oracle verify on the GPU draft's x, lse_d and logp_d (stage-isolated)."""
    rows = np.arange(inp["U"].shape[0]) if rows is None else np.asarray(rows)
    T = inp["temperature"] if temperature is None else temperature
    s = inp["seed"] if seed is None else seed
    idx = torch.from_numpy(rows).to(inp["U"].device)
    return oracle.verify_round(wl.to_f64(inp["t"][idx]), wl.to_f64(inp["U"][idx]), wl.to_f64(inp["W1"]),
                               wl.to_f64(inp["W2"]), npy(inp["x0"])[rows], draft_np["x"][rows],
                               draft_np["lse_d"][rows], draft_np["logp_d"][rows], np.asarray(ell)[rows], T, s,
                               requests=rows)


def compare_draft(gpu, ref, dtype, rows=None):
    rows = np.arange(gpu["x"].shape[0]) if rows is None else np.asarray(rows)
    gx = gpu["x"][rows]
    exempt = ref["margin"] < MARGIN
    mismatch = (gx != ref["x"]) & ~exempt
    assert not mismatch.any(), f"{mismatch.sum()} token mismatches at {np.argwhere(mismatch)[:5]}"
    same = gx == ref["x"]
    for k in ("c", "a"):
        err = np.abs(gpu[k][rows] - ref[k]).max()
        assert err <= FTOL[dtype], (k, err)
    for k in ("lse_d", "logp_d"):
        err = np.abs(gpu[k][rows] - ref[k])[same].max(initial=0.0)
        assert err <= FTOL["bf16"], (k, err)
    report_exempt("draft tokens", exempt.sum(), exempt.size)
    return int(exempt.sum())


def compare_verify(gpu, ref, rows=None, exact=False):
    """exact: no exemption at all.  Greedy verification compares the same bf16 / fp32
    target values on both sides and breaks ties by the lowest index on both, so its
    decisions agree even where the top-2 gap is zero (exact ties are common among
    bf16 logits); the near-tie count is still reported."""
    rows = np.arange(gpu["n_accept"].shape[0]) if rows is None else np.asarray(rows)
    near = ref["margin"] < MARGIN
    exempt = np.zeros_like(near) if exact else near
    bad = ((gpu["n_accept"][rows] != ref["n_accept"]) | (gpu["next_token"][rows] != ref["next_token"])) & ~exempt
    assert not bad.any(), (f"{bad.sum()} verify mismatches; first rows {rows[bad][:5]}: gpu "
                           f"{gpu['n_accept'][rows][bad][:5]}/{gpu['next_token'][rows][bad][:5]} oracle "
                           f"{ref['n_accept'][bad][:5]}/{ref['next_token'][bad][:5]}")
    report_exempt("verify requests" + (" (exact)" if exact else ""), near.sum(), near.size)
    return int(exempt.sum())
