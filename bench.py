"""Benchmark of the DSpark serving round on GB300: draft block -> prefix
scheduler -> verification, on the high-concurrency workload (B = 1024
requests, gamma = 16, V = 151936, H = 4096, r = 256, bf16, T = 1.0, per-request
peak rate ~ Beta(5, 2)), synthetic seeded inputs; the Qwen3-8B-shaped (B = 64,
gamma = 7, T = 0.7 and greedy) and 27B-draft-shaped (B = 256, gamma = 7)
serving rounds are reported under `extra`, each with its own roofline.

One step = one round through the library's C ABI (all kernels on one stream),
captured once in a CUDA graph and replayed (--no-graph launches the calls
directly every step).
The timed region holds exactly K steps; the L2 is flushed (a 512 MiB write)
between steps, outside each step's CUDA-event pair.  The JSON line also
reports the dominant kernel's roofline (the draft engine, one cooperative
launch per draft call: timed with CUDA events the library records around it,
against the measured copy bandwidth and, for its bias GEMM, the measured
sustained bf16 tensor rate), an end-to-end number through the same C-ABI
calls with inputs copied from pinned host memory each step, the oracle timed
on the host cores on a bounded sample, and the oracle's teacher-forced check
of a sample of the GPU's draws with the exempt decisions counted.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --gpus N > 1 (under torchrun) every rank runs an independent replica of
the round (the path has no cross-request exchange); value = rows of all ranks
over the slowest rank's time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft+verify rows/s over B·γ×V logits; achieved HBM GB/s vs GB300 peak"
WORKLOAD = ("high-concurrency serving round: B=1024 requests, gamma=16, V=151936, H=4096, r=256, bf16, "
            "T=1.0, per-request peak rate ~ Beta(5,2), seed 4")
FALLBACK_HBM_GBS = 6800.0


NOMINAL_HBM_GBS = 8000.0     # the pages' roofline figure for the part
FALLBACK_BF16_SUSTAINED_TFLOPS = 1700.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Sustained dense bf16 TFLOP/s (for a kernel timed inside a long step) and its source."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured (sustained)"
    return FALLBACK_BF16_SUSTAINED_TFLOPS, "fallback (sustained)"


def engine_source_hash():
    """Hash of the draft engine's sources: a recorded ncu traffic figure is only
    reported while the kernel it was measured on is unchanged."""
    import hashlib
    h = hashlib.sha256()
    for f in ("engine.cuh", "tc.cuh", "common.cuh"):   # the draft engine kernel's device code
        with open(os.path.join(ROOT, "serving_draft_verify_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_engine_traffic(l2_resident=False):
    """DRAM bytes of one draft launch (ncu), with or without W2 held in L2, while the
    engine's sources still hash to the captured version."""
    p = os.path.join(ROOT, "profiles", "draft_engine_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    key = "dram_bytes_per_launch_l2_resident" if l2_resident else "dram_bytes_per_launch"
    return d.get(key) if d.get("source_hash") == engine_source_hash() else None


def recorded_engine_issue():
    """Warp instructions per logit of the draft launch (an ncu count on a small case of
    the same kernel), while the engine's sources still hash to the captured version."""
    p = os.path.join(ROOT, "profiles", "draft_engine_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    iss = d.get("issue")
    if not iss or iss.get("source_hash") != engine_source_hash():
        return None
    return iss["warp_instructions"] / iss["logits"]


def issue_roof(logits, launch_us, sm_mhz, n_sm):
    """The issue roof of the draft launch: its warp instructions at one instruction a
    cycle on every scheduler (4 per SM) at the sampled SM clock, against the launch time."""
    wipl = recorded_engine_issue()
    if wipl is None or not sm_mhz or not launch_us:
        return None
    ideal_us = logits * wipl / (n_sm * 4 * sm_mhz)
    return {"warp_instructions_per_logit": round(wipl, 4), "sm_mhz": sm_mhz, "sms": n_sm,
            "ideal_us": round(ideal_us, 1), "frac": round(ideal_us / launch_us, 4),
            "source": "ncu instruction count of the same kernel on B = 1024, gamma = 2"}


def apply_l2_residency(dsv, args, default=False):
    """--l2-residency on|off|auto: the library keeps W2 (V x r bf16 of the Markov head, the
    same shape in every serving config here) in L2 for the draft and verify calls; `auto`
    takes `default` (on for the headline run, off for the one-kernel modes).  Returns the
    bytes set aside, 0 when off."""
    from serving_draft_verify_gb300 import workloads as wl
    mode = getattr(args, "l2_residency", "auto")
    if not (mode == "on" or (mode == "auto" and default)):
        return 0
    nbytes = wl.HIGH_CONC.V * wl.HIGH_CONC.r * 2
    dsv.dspark_set_l2_residency(nbytes)
    return nbytes


def smi_index(local):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local < len(ids) and ids[local].isdigit():
            return int(ids[local])
    return local


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(local_ms, local_rows, world, device):
    """Whole-job figures over `world` ranks: the slowest rank's time and the
    rows of all ranks (every rank calls this, after its own timed region)."""
    if world == 1:
        return float(local_ms), int(local_rows)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    n = torch.tensor([int(local_rows)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


# ------------------------------------------------------------ clocks ---
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "25"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- GPU arm ---
def draft_launch_bytes(B, G, V, H, r):
    """Algorithmic bytes of one draft engine launch (all positions): U, W2 once, h
    (the confidence head reads it in the same launch) and the W1 rows."""
    return B * G * V * 2 + V * r * 2 + B * G * H * 2 + B * G * r * 2


class Serving:
    """One serving config on the GPU: inputs, workspaces, outputs and the round."""

    def __init__(self, dsv, lib, cfg, dev, T=None):
        from serving_draft_verify_gb300 import workloads as wl
        import torch
        self.dsv, self.cfg, self.dev = dsv, cfg, dev
        self.inp = wl.make_draft_inputs(cfg, device=dev)
        self.T = cfg.temperature if T is None else T
        B, G, V, r = cfg.B, cfg.gamma, cfg.V, cfg.r
        self.ws_d = torch.empty(lib.dspark_draft_block_workspace_size(B, G, V, r), dtype=torch.uint8, device=dev)
        self.ws_s = torch.empty(lib.dspark_schedule_prefix_workspace_size(B, G), dtype=torch.uint8, device=dev)
        self.ws_v = torch.empty(lib.dspark_verify_workspace_size(B, G, V, r), dtype=torch.uint8, device=dev)
        self.outd = dict(x=torch.empty((B, G), dtype=torch.int32, device=dev),
                         **{k: torch.empty((B, G), dtype=torch.float32, device=dev)
                            for k in ("lse_d", "logp_d", "c", "a")})
        self.outs = dict(ell=torch.empty(B, dtype=torch.int32, device=dev),
                         n_sched=torch.empty(1, dtype=torch.int32, device=dev),
                         theta=torch.empty(1, dtype=torch.float64, device=dev))
        self.outv = dict(n_accept=torch.empty(B, dtype=torch.int32, device=dev),
                         next_token=torch.empty(B, dtype=torch.int32, device=dev))

    def draft(self, g=None, T=None):
        g = self.inp if g is None else g
        self.dsv.dspark_draft_block(g["U"], g["h"], g["W1"], g["W2"], g["w"], 0.0, g["x0"],
                                    self.T if T is None else T, self.cfg.seed, out=self.outd, workspace=self.ws_d)

    def schedule(self, g=None):
        g = self.inp if g is None else g
        self.dsv.dspark_schedule_prefix(self.outd["a"], g["sps"], out=self.outs, workspace=self.ws_s)

    def verify(self, g=None, T=None):
        g = self.inp if g is None else g
        o = self.outd
        self.dsv.dspark_verify(g["t"], g["U"], g["W1"], g["W2"], g["x0"], o["x"], o["lse_d"], o["logp_d"],
                               self.outs["ell"], self.T if T is None else T, self.cfg.seed, out=self.outv,
                               workspace=self.ws_v)

    def round(self, g=None, T=None):
        self.draft(g, T)
        self.schedule(g)
        self.verify(g, T)

    def status_ok(self):
        return self.dsv.workspace_status(self.ws_d) == 0 and self.dsv.workspace_status(self.ws_v) == 0


def run_gpu(args):
    import torch
    import serving_draft_verify_gb300 as dsv
    from serving_draft_verify_gb300 import workloads as wl

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dsv.load()
    l2_keep = apply_l2_residency(dsv, args, default=True)
    lib = dsv._binding.load()
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    peak, peak_kind = peaks()
    tpk, tpk_kind = tensor_peak()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            torch.cuda.synchronize()

    def timed(fn, steps, warmup, phase_times=False):
        for _ in range(warmup):
            fn()
        barrier()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        phases = []
        for s, e in evs:
            flush.zero_()
            s.record(stream)
            fn()
            e.record(stream)
            if phase_times:
                phases.extend(dsv._binding.phase_times())
        barrier()
        return [s.elapsed_time(e) for s, e in evs], phases

    def graphed(fn):
        """fn's launches captured once in a CUDA graph (the library's calls are plain
        stream work); returns the replay, or None if capture is not possible."""
        if args.no_graph:
            return None
        fn()                                              # one-time attribute setup outside capture
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(g):
                fn()
        except Exception:
            torch.cuda.synchronize()
            return None
        return g.replay

    def measure(sv, steps, warmup, clocks=None):
        """Round throughput of one serving config, the draft engine's roofline from the
        library's events, and per-call device times (directly launched calls)."""
        cfg = sv.cfg
        B, G, V, H, r = cfg.B, cfg.gamma, cfg.V, cfg.H, cfg.r
        dsv._binding.phase_timing(True)
        rnd = graphed(sv.round)
        use_graph = rnd is not None
        if not use_graph:
            rnd = sv.round
        if clocks is not None:
            clocks.start()
        times, phase_ms = timed(rnd, steps, warmup, phase_times=True)
        engine_timing = "events around the draft launch, captured with the replayed round"
        if not phase_ms:                                  # events in the graph not timeable here
            _, phase_ms = timed(sv.round, steps, warmup, phase_times=True)
            engine_timing = "events around the draft launch, in as many directly launched rounds"
        clk = clocks.stop() if clocks is not None else None
        dsv._binding.phase_timing(False)
        assert sv.status_ok()
        total_ms = sum(times)
        ell = sv.outs["ell"].cpu().numpy()
        nacc = sv.outv["n_accept"].cpu().numpy()
        n_rej = int((nacc < ell).sum())
        sched_rows = int((ell + 1).sum())
        round_bytes = draft_launch_bytes(B, G, V, H, r) + sched_rows * V * 2 + n_rej * 2 * V * 2
        per_call = max(len(phase_ms) // steps, 1) if steps else 1
        launch_bytes = draft_launch_bytes(B, G, V, H, r) / per_call
        phase_avg = sum(phase_ms) / len(phase_ms) if phase_ms else float("nan")
        achieved = launch_bytes / (phase_avg * 1e-3) / 1e9
        flops = 2.0 * B * G * V * r / per_call
        tflops = flops / (phase_avg * 1e-3) / 1e12
        roof = {"bound": "hbm", "kernel": "bias_engine_tc<kDraft> (draft block, all positions, one launch)",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": None, "peak_kind": f"{peak_kind} copy bandwidth",
                "bytes_per_launch": int(launch_bytes), "avg_launch_us": round(phase_avg * 1e3, 2),
                "launches_timed": len(phase_ms), "timing": engine_timing,
                "tensor": {"flops_per_launch": flops, "achieved_tflops": round(tflops, 1), "peak_tflops": tpk,
                           "frac": round(tflops / tpk, 4), "peak_kind": tpk_kind}}
        # per-call device times, launched directly (events between the calls, L2 flushed first)
        ev_ = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        call_us = [[], [], []]
        for it_ in range(min(max(10, steps), 40) + 3):
            flush.zero_()
            ev_[0].record(stream)
            sv.draft()
            ev_[1].record(stream)
            sv.schedule()
            ev_[2].record(stream)
            sv.verify()
            ev_[3].record(stream)
            torch.cuda.synchronize()
            if it_ >= 3:
                for i_ in range(3):
                    call_us[i_].append(ev_[i_].elapsed_time(ev_[i_ + 1]) * 1e3)
        med = [statistics.median(x) for x in call_us]
        ver_bytes = sched_rows * V * 2
        out = {"workload": cfg.name, "B": B, "gamma": G, "V": V, "H": H, "r": r, "temperature": sv.T,
               "rows_per_s": B * G * steps / (total_ms * 1e-3), "ms_per_step": total_ms / steps, "steps": steps,
               "cuda_graph": use_graph, "round_hbm_gbs": round_bytes * steps / (total_ms * 1e-3) / 1e9,
               "roofline": roof,
               "per_call": {"timing": "CUDA events between directly launched calls, median",
                            "draft_us": med[0], "schedule_us": med[1], "verify_us": med[2],
                            "verify_algorithmic_bytes": ver_bytes,
                            "verify_gbs": ver_bytes / (med[2] * 1e-6) / 1e9,
                            "verify_frac": ver_bytes / (med[2] * 1e-6) / 1e9 / peak},
               "scheduled_rows": sched_rows, "rejected_requests": n_rej,
               "accepted_per_request": float(nacc.mean())}
        return out, clk

    def parity_sample(sv, nreq):
        """The oracle, teacher-forced on the GPU's draft tokens and verifying the GPU's
        own draft outputs, on the first nreq requests: mismatches beyond the exempt
        decisions (oracle margin < 1e-4), and the exempt counts."""
        import numpy as np
        import oracle
        rows = np.arange(nreq)
        inp = sv.inp
        idx = torch.from_numpy(rows).to(inp["U"].device)
        f64 = wl.to_f64
        dn = {k: v.cpu().numpy() for k, v in sv.outd.items()}
        ell = sv.outs["ell"].cpu().numpy()
        ref = oracle.draft_block(f64(inp["U"][idx]), f64(inp["h"][idx]), f64(inp["W1"]), f64(inp["W2"]),
                                 f64(inp["w"]), 0.0, inp["x0"].cpu().numpy()[rows], sv.T, sv.cfg.seed,
                                 forced_tokens=dn["x"][rows], requests=rows)
        ex_d = ref["margin"] < 1e-4
        mis_d = int(((dn["x"][rows] != ref["x"]) & ~ex_d).sum())
        vr = oracle.verify_round(f64(inp["t"][idx]), f64(inp["U"][idx]), f64(inp["W1"]), f64(inp["W2"]),
                                 inp["x0"].cpu().numpy()[rows], dn["x"][rows], dn["lse_d"][rows],
                                 dn["logp_d"][rows], ell[rows], sv.T, sv.cfg.seed, requests=rows)
        ex_v = vr["margin"] < 1e-4
        na = sv.outv["n_accept"].cpu().numpy()[rows]
        nt = sv.outv["next_token"].cpu().numpy()[rows]
        mis_v = int((((na != vr["n_accept"]) | (nt != vr["next_token"])) & ~ex_v).sum())
        return {"requests": int(nreq), "draft_tokens": int(ex_d.size), "draft_exempt": int(ex_d.sum()),
                "draft_mismatches": mis_d, "verify_requests": int(ex_v.size), "verify_exempt": int(ex_v.sum()),
                "verify_mismatches": mis_v}

    # ------------------------------------------------ headline: high concurrency
    cfg = wl.HIGH_CONC
    sv = Serving(dsv, lib, cfg, dev)
    B, G, V, H, r = cfg.B, cfg.gamma, cfg.V, cfg.H, cfg.r
    clocks = ClockSampler(smi_index(local))
    head, clk = measure(sv, args.steps, args.warmup, clocks=clocks)
    total_ms, rows = aggregate(head["ms_per_step"] * args.steps, B * G * args.steps, world, dev)
    value = rows / (total_ms * 1e-3)
    ms_per_step = total_ms / args.steps
    roofline = dict(head["roofline"])
    roofline["traffic"] = (args.phase_traffic if args.phase_traffic is not None
                           else recorded_engine_traffic(l2_resident=bool(l2_keep)))
    roofline["issue"] = issue_roof(B * G * V, roofline["avg_launch_us"], (clk or {}).get("sm_mhz"),
                                   torch.cuda.get_device_properties(dev).multi_processor_count)

    # end to end: every step's per-call inputs (U, h, x0, the SPS table and the target
    # logits t) are in pinned host memory and go to the C-ABI calls as host buffers, all
    # inside the timed region: the draft call copies U and h to the device in one
    # copy-engine transfer each, and the kernels read the rest over the host link, each
    # byte they need once (t only in its scheduled rows; the weights W1, W2, w stay
    # resident on the device).  Each step's results (x, n_accept, next_token) are copied back to pinned
    # host memory.  Two host input sets alternate between steps; every step streams more
    # than 5 GB, so nothing of a step's inputs is still in L2 for the next.
    e2e = None
    if not args.skip_e2e:
        host_sets = [{k: sv.inp[k].cpu().pin_memory() for k in ("U", "h", "x0", "sps", "t")} for _ in range(2)]
        t_rows_bytes = head["scheduled_rows"] * V * 2
        h2d = sum(host_sets[0][k].numel() * host_sets[0][k].element_size() for k in ("U", "h", "x0", "sps")) \
            + t_rows_bytes
        res_host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                    for k, v in (("x", sv.outd["x"]), ("n_accept", sv.outv["n_accept"]),
                                 ("next_token", sv.outv["next_token"]))}
        d2h = sum(v.numel() * v.element_size() for v in res_host.values())

        def e2e_run(nsteps):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            t0.record(stream)
            for i in range(nsteps):
                g_ = dict(sv.inp)
                g_.update(host_sets[i % 2])
                sv.round(g_)
                for k in ("x", "n_accept", "next_token"):
                    res_host[k].copy_(sv.outd["x"] if k == "x" else sv.outv[k], non_blocking=True)
            t1.record(stream)
            barrier()
            return t0.elapsed_time(t1)

        e2e_steps = max(3, min(args.steps, args.e2e_steps))
        e2e_run(min(args.warmup, 3))
        staged0 = dsv._binding.staged_bytes()
        e_ms, e_rows = aggregate(e2e_run(e2e_steps), B * G * e2e_steps, world, dev)
        staged = (dsv._binding.staged_bytes() - staged0) // e2e_steps
        assert sv.status_ok()
        e2e = {"value": e_rows / (e_ms * 1e-3), "unit": "rows/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "staged_bytes_per_step": staged,
               "inputs": "pinned host buffers passed to the C-ABI calls; the draft call copies U and h to the device"
                         " (one copy-engine transfer each), the kernels read x0, the SPS table and t's scheduled rows"
                         " over the host link",
               "l2": "no flush: every step reads more than 5 GB of host inputs"}
        del host_sets
    parity = None if args.no_cpu_baseline or world > 1 else parity_sample(sv, args.parity_requests)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(sv.inp, sv.T, cfg.seed)
    del sv
    torch.cuda.empty_cache()

    # ------------------------------------------------ the other serving configs
    extra_cfgs = {}
    if not args.skip_extra_configs:
        for key, c_, T_ in (("qwen3_8b", wl.QWEN3_8B, None), ("qwen3_8b_greedy", wl.QWEN3_8B, 0.0),
                            ("draft_27b", wl.DRAFT_27B, None)):
            sv_ = Serving(dsv, lib, c_, dev, T=T_)
            res, _ = measure(sv_, max(10, min(args.steps, 200)), args.warmup)
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                res["parity_sample"] = parity_sample(sv_, min(c_.B, 16))
                res["cpu_baseline"] = cpu_baseline(sv_.inp, sv_.T, c_.seed, min_seconds=3.0, max_rounds=4,
                                                   nreq=min(c_.B, 16))
            extra_cfgs[key] = res
            del sv_
            torch.cuda.empty_cache()

    # accept-rate TV on the training workload (16384 x 151936 bf16 rows): its second pass
    # needs the whole L2, so W2's persisting lines (the residency) are released first
    tv = None
    if not args.skip_tv:
        if l2_keep:
            dsv.dspark_set_l2_residency(0)
        d_, t_ = wl.make_tv_inputs(wl.TV_TRAIN, device=dev)
        cst = torch.empty(d_.shape[0], dtype=torch.float32, device=dev)
        ws_t = torch.empty(256, dtype=torch.uint8, device=dev)
        tv_times, _ = timed(lambda: dsv.dspark_accept_rate_tv(d_, t_, c_star=cst, workspace=ws_t), 5, 3)
        tvb = 2 * d_.numel() * 2
        tv_ms = sum(tv_times) / len(tv_times)
        tv = {"rows": d_.shape[0], "ms": tv_ms, "rows_per_s": d_.shape[0] / (tv_ms * 1e-3),
              "achieved_gbs": tvb / (tv_ms * 1e-3) / 1e9, "frac_of_peak": tvb / (tv_ms * 1e-3) / 1e9 / peak}
        # the joint training loss with its gradient on the same rows: d, t read, dL/dd written
        tgt_, s_, k_ = wl.make_loss_inputs(wl.TV_TRAIN, device=dev)
        w_ = torch.exp(-(k_.double() - 1.0) / 4.0)      # position weights, normalised to a weighted mean
        om_ = (w_ / w_.sum()).float()
        lout = dict(row=torch.empty((d_.shape[0], 4), dtype=torch.float32, device=dev),
                    loss=torch.empty(1, dtype=torch.float32, device=dev),
                    grad_d=torch.empty_like(d_), grad_conf=torch.empty(d_.shape[0], dtype=torch.float32, device=dev))
        ws_l = torch.empty(1 << 16, dtype=torch.uint8, device=dev)
        l_times, _ = timed(lambda: dsv.dspark_training_loss(d_, t_, tgt_, s_, om_, out=lout, workspace=ws_l), 5, 3)
        lb = 3 * d_.numel() * 2
        l_ms = sum(l_times) / len(l_times)
        tv["training_loss"] = {"ms": l_ms, "rows_per_s": d_.shape[0] / (l_ms * 1e-3),
                               "bytes_per_row": 3 * d_.shape[1] * 2,
                               "achieved_gbs": lb / (l_ms * 1e-3) / 1e9,
                               "frac_of_peak": lb / (l_ms * 1e-3) / 1e9 / peak}
        del d_, t_, lout
        torch.cuda.empty_cache()
    # the draft block with the gated and recurrent heads (one launch per position plus a
    # head kernel between positions), on the Qwen3-8B-shaped workload
    if l2_keep and not args.skip_tv:
        apply_l2_residency(dsv, args, default=True)     # back on for the draft extras below
    heads_x = None
    if not args.skip_heads:
        heads_x = {}
        c8 = wl.QWEN3_8B
        sv8 = Serving(dsv, lib, c8, dev)
        for kind, name in ((1, "gated"), (2, "rnn")):
            Wg_, Wc_ = wl.make_head_weights(c8, kind, device=dev)
            head_ = dict(kind=kind, Wg=Wg_, Wc=Wc_, E=torch.empty((c8.B, c8.gamma, c8.r), dtype=torch.bfloat16,
                                                                  device=dev))
            ws_h = torch.empty(lib.dspark_draft_block_ex_workspace_size(c8.B, c8.gamma, c8.V, c8.r, kind),
                               dtype=torch.uint8, device=dev)
            g8 = sv8.inp

            def head_call():
                dsv.dspark_draft_block_ex(g8["U"], g8["h"], g8["W1"], g8["W2"], g8["w"], 0.0, g8["x0"], sv8.T,
                                          c8.seed, head_, out=sv8.outd, workspace=ws_h)
            h_fn = graphed(head_call)
            h_times, _ = timed(h_fn or head_call, 20, 3)
            heads_x[name] = {"workload": c8.name, "draft_ms": sum(h_times) / len(h_times),
                             "cuda_graph": h_fn is not None}
        del sv8
    # several rounds with the anchor carried (the last emitted token), one CUDA graph over
    # a pool of 8 synthetic rounds of the Qwen3-8B shape
    multi = None
    if not args.skip_rounds:
        c8 = wl.QWEN3_8B
        R, P = 32, 8
        pool_ = wl.make_round_pool(c8, P, device=dev)
        anchor_ = pool_["x0"].clone()
        ws_r = torch.empty(lib.dspark_decode_rounds_workspace_size(c8.B, c8.gamma, c8.V, c8.r), dtype=torch.uint8,
                           device=dev)
        rout = dict(tokens=torch.empty((R, c8.B, c8.gamma + 1), dtype=torch.int32, device=dev),
                    n_emitted=torch.empty((R, c8.B), dtype=torch.int32, device=dev),
                    stats=torch.empty((R, 2), dtype=torch.float64, device=dev))

        def rounds_call():
            anchor_.copy_(pool_["x0"])
            dsv.dspark_decode_rounds(pool_["U"], pool_["h"], pool_["t"], pool_["W1"], pool_["W2"], pool_["w"], 0.0,
                                     pool_["sps"], anchor_, R, c8.temperature, c8.seed, out=rout, workspace=ws_r)
        rounds_fn = graphed(rounds_call)
        r_times, _ = timed(rounds_fn or rounds_call, 10, 3)
        r_ms = sum(r_times) / len(r_times)
        st_ = rout["stats"].cpu()
        multi = {"workload": c8.name, "rounds": R, "pool": P, "cuda_graph": rounds_fn is not None,
                 "ms_per_round": r_ms / R,
                 "emitted_tokens_per_s": float(rout["n_emitted"].sum().item()) / (r_ms * 1e-3),
                 "E_tau": float(st_[:, 0].mean()), "realised_tau": float(st_[:, 1].mean())}
        del pool_
    # draft: the cooperative engine launch; schedule: chunks, rank, scan; verify: plan, rows, residual
    launches_per_step = 1 + 3 + 3

    line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; shapes of the pages' high-concurrency serving setting)",
            "config": dict(workload_config(world), cuda_graph=head["cuda_graph"],
                           l2_residency=(f"W2 held in L2 by a persisting access-policy window ({l2_keep} B set aside)"
                                         if l2_keep else "off")),
            "hbm_gbs": head["round_hbm_gbs"], "hbm_frac": head["round_hbm_gbs"] / peak, "roofline": roofline,
            "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "clocks": clk,
            "extra": {"per_call": head["per_call"], "scheduled_rows": head["scheduled_rows"],
                      "rejected_requests": head["rejected_requests"],
                      "accepted_per_request": head["accepted_per_request"],
                      "exempt": parity,
                      "serving_configs": extra_cfgs, "accept_rate_tv": tv, "multi_round": multi,
                      "heads": heads_x}}
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


# ------------------------------------------------------------ oracle ---
def workload_config(world):
    from serving_draft_verify_gb300 import workloads as wl
    c = wl.HIGH_CONC
    return {"workload": WORKLOAD, "B": c.B, "gamma": c.gamma, "V": c.V, "H": c.H, "r": c.r,
            "temperature": c.temperature, "l2": "flushed between steps (512 MiB write outside the timed step)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def oracle_inputs(inp, nreq=None):
    """The round's inputs (the first `nreq` requests) as float64 numpy arrays."""
    from serving_draft_verify_gb300 import workloads as wl
    n = inp["U"].shape[0] if nreq is None else nreq
    out = {k: wl.to_f64(inp[k][:n]) for k in ("U", "h", "t")}
    out.update({k: wl.to_f64(inp[k]) for k in ("W1", "W2", "w")})
    out["x0"] = inp["x0"][:n].cpu().numpy()
    return out


def oracle_round(f64, T, seed, nreq):
    """One round of the oracle (float64 numpy) over the first `nreq` requests:
    draft, schedule over the sample, verify.  Returns its wall time in s."""
    import numpy as np
    import oracle

    rows = np.arange(nreq)
    U, h, t, x0 = f64["U"][:nreq], f64["h"][:nreq], f64["t"][:nreq], f64["x0"][:nreq]
    W1, W2, w = f64["W1"], f64["W2"], f64["w"]
    G = U.shape[1]
    t0 = time.perf_counter()
    d = oracle.draft_block(U, h, W1, W2, w, 0.0, x0, T, seed, requests=rows)
    N = np.arange(nreq * (G + 1) + 1, dtype=np.float64)
    ell, _, _ = oracle.schedule_prefix(d["a"].astype(np.float32), N / (20.0 + 0.05 * N))
    oracle.verify_round(t, U, W1, W2, x0, d["x"], d["lse_d"], d["logp_d"], ell, T, seed, requests=rows)
    return time.perf_counter() - t0


def cpu_baseline(inp, T, seed, min_seconds=10.0, max_rounds=24, nreq=16):
    """The oracle on the host cores: rounds (draft, schedule over the sample, verify)
    of the first `nreq` requests of the same workload, repeated until at least
    `min_seconds` of work (at most `max_rounds`)."""
    f64 = oracle_inputs(inp, nreq)
    B, G = f64["U"].shape[0], f64["U"].shape[1]
    spent, n = 0.0, 0
    while n < max_rounds and (n == 0 or spent < min_seconds):
        spent += oracle_round(f64, T, seed, B)
        n += 1
    return {"value": n * B * G / spent, "unit": "rows/s", "cores": host_threads(), "kind": "oracle",
            "sample": f"{n} rounds (draft, schedule over the sample, verify) of the first {B} requests x {G} "
                      f"positions, float64 numpy (BLAS threads up to the core count); {spent:.1f} s"}


def run_reference(args):
    world, rank, local = dist_setup()
    if rank != 0:
        return
    from serving_draft_verify_gb300 import workloads as wl
    cfg = wl.HIGH_CONC
    # requests per step: one or two requests' full rounds (16 positions over the whole
    # vocabulary), so that even a long run stays within a few minutes.  The sample is an
    # instance of the same workload with B = nreq (every per-request shape and value
    # distribution of the config; W1, W2, w of the same shapes), so that the 10 GB of
    # the full batch are not drawn on the host for two of its requests.
    nreq = 2 if args.steps <= 100 else 1
    inp = wl.make_draft_inputs(wl.scaled(cfg, B=nreq), device="cpu")
    for _ in range(args.warmup):
        pass                                              # the oracle has nothing to warm
    times = []
    f64 = oracle_inputs(inp, nreq)
    for _ in range(args.steps):
        times.append(oracle_round(f64, cfg.temperature, cfg.seed, nreq))
    total = sum(times)
    value = nreq * cfg.gamma * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": workload_config(1),
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": host_threads(), "kind": "oracle",
                             "sample": f"{nreq} request(s) x {cfg.gamma} positions per step of the same "
                                       f"workload (a B = {nreq} instance), one round each (draft, schedule over "
                                       f"the sample, verify)"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_tv_only(args):
    """The accept-rate TV and training-loss kernels alone on `args.tv_rows` rows of
    the training workload (a small case for profiling); prints one JSON line."""
    import torch
    import serving_draft_verify_gb300 as dsv
    from serving_draft_verify_gb300 import workloads as wl

    dev = torch.device("cuda", 0)
    dsv.load()
    cfg = wl.scaled(wl.TV_TRAIN, rows=args.tv_rows)
    d, t = wl.make_tv_inputs(cfg, device=dev)
    tgt, s, k = wl.make_loss_inputs(cfg, device=dev)
    w = torch.exp(-(k.double() - 1.0) / 4.0)
    om = (w / w.sum()).float()
    cst = torch.empty(cfg.rows, dtype=torch.float32, device=dev)
    lout = dict(row=torch.empty((cfg.rows, 4), dtype=torch.float32, device=dev),
                loss=torch.empty(1, dtype=torch.float32, device=dev),
                grad_d=torch.empty_like(d), grad_conf=torch.empty(cfg.rows, dtype=torch.float32, device=dev))
    ws = torch.empty(1 << 16, dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    res = {"workload": f"{cfg.name}: {cfg.rows} x {cfg.V} {cfg.dtype}"}
    kernels = (("accept_rate_tv", lambda: dsv.dspark_accept_rate_tv(d, t, c_star=cst, workspace=ws), 2),
               ("training_loss", lambda: dsv.dspark_training_loss(d, t, tgt, s, om, out=lout, workspace=ws), 3))
    for name, fn, nb in kernels:
        for _ in range(args.warmup):
            fn()
        ms = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        m = sum(ms) / len(ms)
        res[name] = {"ms": m, "gbs": nb * d.numel() * d.element_size() / (m * 1e-3) / 1e9}
    print(json.dumps(res))


def run_round_case(args):
    """One draft -> schedule -> verify round on a high-concurrency-shaped case (B x gamma
    of the full vocabulary), for profiling the round's kernels on a small case; prints
    one JSON line with the per-call times (CUDA events, L2 flushed before each round)."""
    import torch
    import serving_draft_verify_gb300 as dsv
    from serving_draft_verify_gb300 import workloads as wl

    dev = torch.device("cuda", 0)
    dsv.load()
    l2_keep = apply_l2_residency(dsv, args)
    lib = dsv._binding.load()
    B, G = (int(x) for x in args.round_case.split(":"))
    sv = Serving(dsv, lib, wl.scaled(wl.HIGH_CONC, B=B, gamma=G), dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    us = [[], [], []]
    for it in range(args.warmup + args.steps):
        flush.zero_()
        ev[0].record()
        sv.draft()
        ev[1].record()
        sv.schedule()
        ev[2].record()
        sv.verify()
        ev[3].record()
        torch.cuda.synchronize()
        if it >= args.warmup:
            for i in range(3):
                us[i].append(ev[i].elapsed_time(ev[i + 1]) * 1e3)
    assert sv.status_ok()
    ell = sv.outs["ell"].cpu()
    print(json.dumps({"workload": f"round, B={B} gamma={G} V={sv.cfg.V} r={sv.cfg.r} T={sv.T}",
                      "l2_residency": l2_keep,
                      "draft_us": statistics.median(us[0]), "schedule_us": statistics.median(us[1]),
                      "verify_us": statistics.median(us[2]), "scheduled_rows": int((ell + 1).sum()),
                      "rejected": int((sv.outv["n_accept"].cpu() < ell).sum())}))


DRAFT_PATHS = {"auto": 0, "tcgen05": 1, "gemv": 2}


def run_draft_only(args):
    """dspark_draft_block alone on a high-concurrency-shaped case (B x gamma of the
    full vocabulary), for profiling one kernel on a small case; prints one JSON line
    with the per-call time (CUDA events, L2 flushed between calls)."""
    import torch
    import serving_draft_verify_gb300 as dsv
    from serving_draft_verify_gb300 import workloads as wl

    dev = torch.device("cuda", 0)
    dsv.load()
    l2_keep = apply_l2_residency(dsv, args)
    lib = dsv._binding.load()
    B, G = (int(x) for x in args.draft_case.split(":"))
    dsv._binding.set_draft_path(DRAFT_PATHS[args.draft_path])
    T = wl.HIGH_CONC.temperature if args.draft_temperature is None else args.draft_temperature
    sv = Serving(dsv, lib, wl.scaled(wl.HIGH_CONC, B=B, gamma=G), dev, T=T)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        sv.draft()
    ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        sv.draft()
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    assert dsv.workspace_status(sv.ws_d) == 0
    m = statistics.median(ms)
    cfg = sv.cfg
    nb = draft_launch_bytes(cfg.B, cfg.gamma, cfg.V, cfg.H, cfg.r)
    print(json.dumps({"workload": f"draft block, B={B} gamma={G} V={cfg.V} r={cfg.r} T={T}",
                      "path": args.draft_path, "l2_residency": l2_keep, "median_ms": m,
                      "gbs": nb / (m * 1e-3) / 1e9, "logits_per_ms": B * G * cfg.V / m}))


def arg_parser():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--skip-tv", action="store_true")
    ap.add_argument("--skip-rounds", action="store_true", help="skip the multi-round extra")
    ap.add_argument("--skip-heads", action="store_true", help="skip the gated / recurrent head extra")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the round's calls directly, without a CUDA graph")
    ap.add_argument("--skip-e2e", action="store_true", help="skip the end-to-end (host memory) measurement")
    ap.add_argument("--e2e-steps", type=int, default=40, help="steps of the end-to-end measurement (at most --steps)")
    ap.add_argument("--skip-extra-configs", action="store_true",
                    help="skip the Qwen3-8B-shaped and 27B-draft-shaped serving rounds")
    ap.add_argument("--parity-requests", type=int, default=8,
                    help="requests of the headline round the oracle re-checks (exempt decisions reported)")
    ap.add_argument("--phase-traffic", type=float, default=None,
                    help="dram bytes per draft phase launch from an ncu capture (reported as roofline.traffic)")
    ap.add_argument("--draft-case", default=None,
                    help="B:gamma -- time only dspark_draft_block on that high-concurrency-shaped case")
    ap.add_argument("--draft-temperature", type=float, default=None, help="temperature of --draft-case")
    ap.add_argument("--draft-path", default="auto", choices=sorted(DRAFT_PATHS),
                    help="draft path of --draft-case: by batch size, the tcgen05 engine, or the CUDA-core GEMV")
    ap.add_argument("--l2-residency", nargs="?", const="on", default="auto", choices=["auto", "on", "off"],
                    help="keep W2 in L2 with the library's opt-in persisting window (dspark_set_l2_residency) for "
                         "the draft and verify calls: on for the headline run and off for --draft-case and "
                         "--round-case unless given (the flag alone means on)")
    ap.add_argument("--round-case", default=None,
                    help="B:gamma -- time only the round's three calls on that high-concurrency-shaped case")
    ap.add_argument("--tv-rows", type=int, default=None,
                    help="time only the TV and training-loss kernels on this many training rows")
    return ap


def main():
    args = arg_parser().parse_args()
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3
    if args.tv_rows is not None:
        run_tv_only(args)
    elif args.draft_case is not None:
        run_draft_only(args)
    elif args.round_case is not None:
        run_round_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
