"""Benchmark of the DSpark serving round on GB300: draft block -> prefix
scheduler -> verification, on the Qwen3-8B-shaped serving workload
(B = 64 requests, gamma = 7, V = 151936, H = 4096, r = 256, bf16, T = 0.7),
synthetic seeded inputs.

One step = one round through the library's C ABI (all kernels on one stream),
captured once in a CUDA graph and replayed (--no-graph launches the calls
directly every step).
The timed region holds exactly K steps; the L2 is flushed (a 512 MiB write)
between steps, outside each step's CUDA-event pair.  The JSON line also
reports the dominant kernel's roofline (the draft engine, one cooperative
launch per draft call: timed with CUDA events the library records around it), an
end-to-end number through the same C-ABI calls with inputs copied from pinned
host memory each step, the oracle timed on the host cores on a bounded sample,
and extra lines for greedy decoding and the accept-rate TV kernel.

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
WORKLOAD = ("Qwen3-8B-shaped serving round: B=64, gamma=7 (verify width 8), V=151936, H=4096, r=256, "
            "bf16, T=0.7, seed 1")
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


def recorded_engine_traffic():
    p = os.path.join(ROOT, "profiles", "draft_engine_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    return d.get("dram_bytes_per_launch") if d.get("source_hash") == engine_source_hash() else None


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
    lib = dsv._binding.load()
    cfg = wl.QWEN3_8B
    inp = wl.make_draft_inputs(cfg, device=dev)
    B, G, V, H, r = cfg.B, cfg.gamma, cfg.V, cfg.H, cfg.r
    T, seed = cfg.temperature, cfg.seed
    stream = torch.cuda.current_stream()

    ws_d = torch.empty(lib.dspark_draft_block_workspace_size(B, G, V, r), dtype=torch.uint8, device=dev)
    ws_s = torch.empty(lib.dspark_schedule_prefix_workspace_size(B, G), dtype=torch.uint8, device=dev)
    ws_v = torch.empty(lib.dspark_verify_workspace_size(B, G, V, r), dtype=torch.uint8, device=dev)
    outd = dict(x=torch.empty((B, G), dtype=torch.int32, device=dev),
                **{k: torch.empty((B, G), dtype=torch.float32, device=dev) for k in ("lse_d", "logp_d", "c", "a")})
    outs = dict(ell=torch.empty(B, dtype=torch.int32, device=dev), n_sched=torch.empty(1, dtype=torch.int32, device=dev),
                theta=torch.empty(1, dtype=torch.float64, device=dev))
    outv = dict(n_accept=torch.empty(B, dtype=torch.int32, device=dev),
                next_token=torch.empty(B, dtype=torch.int32, device=dev))

    def round_(g, temperature):
        dsv.dspark_draft_block(g["U"], g["h"], g["W1"], g["W2"], g["w"], 0.0, g["x0"], temperature, seed,
                               out=outd, workspace=ws_d)
        dsv.dspark_schedule_prefix(outd["a"], g["sps"], out=outs, workspace=ws_s)
        dsv.dspark_verify(g["t"], g["U"], g["W1"], g["W2"], g["x0"], outd["x"], outd["lse_d"], outd["logp_d"],
                          outs["ell"], temperature, seed, out=outv, workspace=ws_v)

    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

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

    # main arm, T = 0.7, the round replayed from a CUDA graph; the library's events
    # around the draft launch are captured with it and time that launch every step
    clocks = ClockSampler(smi_index(local))
    dsv._binding.phase_timing(True)
    main_round = graphed(lambda: round_(inp, T))
    use_graph = main_round is not None
    if not use_graph:
        main_round = lambda: round_(inp, T)
    stream = torch.cuda.current_stream()
    clocks.start()
    times, phase_ms = timed(main_round, args.steps, args.warmup, phase_times=True)
    engine_timing = "events around the draft launch, captured with the replayed round"
    if not phase_ms:                                      # events in the graph not timeable here
        _, phase_ms = timed(lambda: round_(inp, T), args.steps, args.warmup, phase_times=True)
        engine_timing = "events around the draft launch, in as many directly launched rounds"
    clk = clocks.stop()
    dsv._binding.phase_timing(False)
    assert dsv.workspace_status(ws_d) == 0 and dsv.workspace_status(ws_v) == 0
    total_ms, rows = aggregate(sum(times), B * G * args.steps, world, dev)
    value = rows / (total_ms * 1e-3)
    ms_per_step = total_ms / args.steps

    # algorithmic bytes of one round: U and h once, W2 once per draft call, W1 rows,
    # the scheduled target rows, and the residual rows (U and t) of rejected requests
    ell = outs["ell"].cpu().numpy()
    nacc = outv["n_accept"].cpu().numpy()
    n_rej = int((nacc < ell).sum())
    round_bytes = (B * G * V * 2 + V * r * 2 + B * G * H * 2 + B * G * r * 2 + int((ell + 1).sum()) * V * 2
                   + n_rej * 2 * V * 2)
    hbm_gbs = round_bytes * args.steps / (total_ms * 1e-3) / 1e9
    peak, peak_kind = peaks()

    # dominant kernel: the draft engine, one cooperative launch per draft call that
    # covers all gamma positions (the library records CUDA events around it on the
    # launching stream).  Algorithmic bytes of one launch: U, W2 once, W1 rows.
    launch_bytes = B * G * V * 2 + V * r * 2 + B * G * r * 2
    per_call = len(phase_ms) // args.steps if args.steps else 0
    launch_bytes /= max(per_call, 1)
    ph = sorted(phase_ms)
    phase_avg = sum(ph) / len(ph) if ph else float("nan")
    achieved = launch_bytes / (phase_avg * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": "bias_engine_tc<kDraft> (draft block, all positions)",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": args.phase_traffic if args.phase_traffic is not None else recorded_engine_traffic(),
                "peak_kind": f"{peak_kind} (copy bandwidth)", "bytes_per_launch": int(launch_bytes),
                "avg_launch_us": round(phase_avg * 1e3, 2), "launches_timed": len(ph), "timing": engine_timing}

    # per-call device times of the round, launched directly (events between the calls,
    # L2 flushed before each round): draft, schedule (latency) and verify with its
    # algorithmic bytes (the scheduled target rows, plus U and t rows of rejected
    # requests are not counted)
    ev_ = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    call_us = [[], [], []]
    for it_ in range(max(10, min(args.steps, 100)) + 3):
        flush.zero_()
        ev_[0].record(stream)
        dsv.dspark_draft_block(inp["U"], inp["h"], inp["W1"], inp["W2"], inp["w"], 0.0, inp["x0"], T, seed,
                               out=outd, workspace=ws_d)
        ev_[1].record(stream)
        dsv.dspark_schedule_prefix(outd["a"], inp["sps"], out=outs, workspace=ws_s)
        ev_[2].record(stream)
        dsv.dspark_verify(inp["t"], inp["U"], inp["W1"], inp["W2"], inp["x0"], outd["x"], outd["lse_d"],
                          outd["logp_d"], outs["ell"], T, seed, out=outv, workspace=ws_v)
        ev_[3].record(stream)
        torch.cuda.synchronize()
        if it_ >= 3:
            for i_ in range(3):
                call_us[i_].append(ev_[i_].elapsed_time(ev_[i_ + 1]) * 1e3)
    med_ = [statistics.median(x) for x in call_us]
    ver_bytes = int((outs["ell"].cpu().long() + 1).sum()) * V * 2
    bias_flops = 2.0 * B * G * V * r
    tpk, tpk_kind = tensor_peak()
    breakdown = {"timing": "CUDA events between directly launched calls, median",
                 "draft_us": med_[0], "schedule_us": med_[1], "verify_us": med_[2],
                 "verify_algorithmic_bytes": ver_bytes, "verify_gbs": ver_bytes / (med_[2] * 1e-6) / 1e9,
                 "draft_bias_tflops": bias_flops / (phase_avg * 1e-3) / 1e12,
                 "draft_bias_frac_of_tensor_peak": bias_flops / (phase_avg * 1e-3) / 1e12 / tpk,
                 "tensor_peak_tflops": tpk, "tensor_peak_kind": tpk_kind,
                 "draft_frac_of_nominal_8tbs": launch_bytes / (phase_avg * 1e-3) / 1e9 / NOMINAL_HBM_GBS}

    # greedy round (same workload, T = 0)
    greedy_round = graphed(lambda: round_(inp, 0.0)) or (lambda: round_(inp, 0.0))
    g_times, _ = timed(greedy_round, max(3, args.steps // 2), args.warmup)
    greedy = {"value": B * G * len(g_times) / (sum(g_times) * 1e-3), "unit": "rows/s",
              "ms_per_step": sum(g_times) / len(g_times)}

    # end to end: every step takes its inputs from pinned host memory and reads its results
    # (x, n_accept, next_token) back.  U, h, x0 and SPS are uploaded (the draft reads all of
    # them); the target logits stay in host memory and verification reads, over the host
    # link, only the rows it needs (the scheduled prefix and its stop row: 135 of 512 rows
    # here).  The link (~200 GB/s) dominates, so the steps are pipelined: step i+1's upload
    # runs on a copy stream into the other of two device input sets while step i's round
    # computes.  Four host copies of t are cycled so that no step can find another step's
    # target rows in L2.  Timed over all K steps (events before the first upload and after
    # the last read-back): whole-job throughput.
    host = {k: inp[k].cpu().pin_memory() for k in ("U", "h", "x0", "sps")}
    host_t = [inp["t"].cpu().pin_memory() for _ in range(4)]
    dev_sets = [{k: torch.empty_like(inp[k]) for k in host} for _ in range(2)]
    t_rows_bytes = int((outs["ell"].cpu().long() + 1).sum()) * V * 2
    h2d = sum(v.numel() * v.element_size() for v in host.values()) + t_rows_bytes
    res_host = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                 for k, v in (("x", outd["x"]), ("n_accept", outv["n_accept"]), ("next_token", outv["next_token"]))}
                for _ in range(2)]
    d2h = sum(v.numel() * v.element_size() for v in res_host[0].values())
    copy_stream = torch.cuda.Stream(device=dev)

    def e2e_run(nsteps):
        """nsteps pipelined end-to-end steps; returns the elapsed ms (device events)."""
        copied = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]
        for f in freed:
            f.record(stream)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        t0.record(stream)
        copy_stream.wait_event(t0)

        def upload(i):
            sl = i % 2
            copy_stream.wait_event(freed[sl])            # the round that read this set is done
            with torch.cuda.stream(copy_stream):
                for k in host:
                    dev_sets[sl][k].copy_(host[k], non_blocking=True)
            copied[sl].record(copy_stream)

        upload(0)
        for i in range(nsteps):
            sl = i % 2
            if i + 1 < nsteps:
                upload(i + 1)
            stream.wait_event(copied[sl])
            g_ = dict(inp)
            g_.update(dev_sets[sl])
            g_["t"] = host_t[i % len(host_t)]
            round_(g_, T)
            freed[sl].record(stream)
            for k in ("x", "n_accept", "next_token"):
                src_ = outd["x"] if k == "x" else outv[k]
                res_host[sl][k].copy_(src_, non_blocking=True)
        t1.record(stream)
        barrier()
        return t0.elapsed_time(t1)

    e2e_run(args.warmup)
    e_ms, e_rows = aggregate(e2e_run(args.steps), B * G * args.steps, world, dev)   # slowest rank, all rows
    e2e = {"value": e_rows / (e_ms * 1e-3), "unit": "rows/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "pipelined": "step i+1's upload overlaps step i's round (two device input sets)",
           "target_rows": "read by verification from pinned host memory (the scheduled rows only)",
           "l2": "no flush: every step uploads 140 MB of fresh inputs and reads its target rows from "
                 "one of four host copies (623 MB together, more than L2)"}

    # accept-rate TV on the training workload (16384 x 151936 bf16 rows)
    tv = None
    if not args.skip_tv:
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
    # the draft block with the gated and recurrent heads (one launch per position plus a
    # head kernel between positions), same workload
    heads_x = None
    if not args.skip_heads:
        heads_x = {}
        for kind, name in ((1, "gated"), (2, "rnn")):
            Wg_, Wc_ = wl.make_head_weights(cfg, kind, device=dev)
            head_ = dict(kind=kind, Wg=Wg_, Wc=Wc_, E=torch.empty((B, G, r), dtype=inp["U"].dtype, device=dev))
            ws_h = torch.empty(lib.dspark_draft_block_ex_workspace_size(B, G, V, r, kind), dtype=torch.uint8,
                               device=dev)

            def head_call():
                dsv.dspark_draft_block_ex(inp["U"], inp["h"], inp["W1"], inp["W2"], inp["w"], 0.0, inp["x0"], T,
                                          seed, head_, out=outd, workspace=ws_h)
            h_fn = graphed(head_call)
            h_times, _ = timed(h_fn or head_call, 20, 3)
            heads_x[name] = {"draft_ms": sum(h_times) / len(h_times), "cuda_graph": h_fn is not None}
    # several rounds with the anchor carried (the last emitted token), one CUDA graph over
    # a pool of 8 synthetic rounds of the same shape
    multi = None
    if not args.skip_rounds:
        R, P = 32, 8
        pool_ = wl.make_round_pool(cfg, P, device=dev)
        anchor_ = pool_["x0"].clone()
        ws_r = torch.empty(lib.dspark_decode_rounds_workspace_size(B, G, V, r), dtype=torch.uint8, device=dev)
        rout = dict(tokens=torch.empty((R, B, G + 1), dtype=torch.int32, device=dev),
                    n_emitted=torch.empty((R, B), dtype=torch.int32, device=dev),
                    stats=torch.empty((R, 2), dtype=torch.float64, device=dev))

        def rounds_call():
            anchor_.copy_(pool_["x0"])
            dsv.dspark_decode_rounds(pool_["U"], pool_["h"], pool_["t"], pool_["W1"], pool_["W2"], pool_["w"], 0.0,
                                     pool_["sps"], anchor_, R, T, seed, out=rout, workspace=ws_r)
        rounds_fn = graphed(rounds_call)
        r_times, _ = timed(rounds_fn or rounds_call, 10, 3)
        r_ms = sum(r_times) / len(r_times)
        st_ = rout["stats"].cpu()
        multi = {"rounds": R, "pool": P, "cuda_graph": rounds_fn is not None, "ms_per_round": r_ms / R,
                 "emitted_tokens_per_s": float(rout["n_emitted"].sum().item()) / (r_ms * 1e-3),
                 "E_tau": float(st_[:, 0].mean()), "realised_tau": float(st_[:, 1].mean())}
        del pool_
    # draft: the cooperative engine launch; schedule: 1; verify: plan, rows, residual (+ final token)
    launches_per_step = 1 + 1 + 3

    line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; shapes of the Qwen3-8B draft setting)",
            "config": dict(workload_config(world), cuda_graph=use_graph),
            "hbm_gbs": hbm_gbs, "hbm_frac": hbm_gbs / peak, "roofline": roofline, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "clocks": clk,
            "extra": {"greedy_round": greedy, "per_call": breakdown, "accept_rate_tv": tv, "multi_round": multi,
                      "heads": heads_x,
                      "accepted_per_request": float(nacc.mean()), "scheduled_rows": int((ell + 1).sum())}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, T, seed)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


# ------------------------------------------------------------ oracle ---
def workload_config(world):
    from serving_draft_verify_gb300 import workloads as wl
    c = wl.QWEN3_8B
    return {"workload": WORKLOAD, "B": c.B, "gamma": c.gamma, "V": c.V, "H": c.H, "r": c.r,
            "temperature": c.temperature, "l2": "flushed between steps (512 MiB write outside the timed step)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def oracle_inputs(inp):
    """The round's inputs as float64 numpy arrays (converted once)."""
    from serving_draft_verify_gb300 import workloads as wl
    out = {k: wl.to_f64(inp[k]) for k in ("U", "h", "t", "W1", "W2", "w")}
    out["x0"] = inp["x0"].cpu().numpy()
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


def cpu_baseline(inp, T, seed, min_seconds=10.0, max_rounds=24):
    """The oracle on the host cores: whole 64-request rounds of the same workload,
    repeated until at least `min_seconds` of work (at most `max_rounds`)."""
    f64 = oracle_inputs(inp)
    B, G = f64["U"].shape[0], f64["U"].shape[1]
    spent, n = 0.0, 0
    while n < max_rounds and (n == 0 or spent < min_seconds):
        spent += oracle_round(f64, T, seed, B)
        n += 1
    return {"value": n * B * G / spent, "unit": "rows/s", "cores": host_threads(), "kind": "oracle",
            "sample": f"{n} full rounds (draft, schedule, verify) of all {B} requests x {G} positions, "
                      f"float64 numpy (BLAS threads up to the core count); {spent:.1f} s"}


def run_reference(args):
    world, rank, local = dist_setup()
    if rank != 0:
        return
    import torch
    from serving_draft_verify_gb300 import workloads as wl
    cfg = wl.QWEN3_8B
    inp = wl.make_draft_inputs(cfg, device="cpu")
    for _ in range(args.warmup):
        pass                                              # the oracle has nothing to warm
    times = []
    # requests per step: about 0.06 s of oracle work each, so that even a long run
    # (--steps 500) stays near a minute of host time
    nreq = 4 if args.steps <= 200 else (2 if args.steps <= 400 else 1)
    f64 = oracle_inputs(inp)
    for _ in range(args.steps):
        times.append(oracle_round(f64, cfg.temperature, cfg.seed, nreq))
    total = sum(times)
    value = nreq * cfg.gamma * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": workload_config(1),
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": host_threads(), "kind": "oracle",
                             "sample": f"{nreq} of {cfg.B} requests x {cfg.gamma} positions per step, one "
                                       f"round each (draft, schedule over the sample, verify)"},
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--skip-tv", action="store_true")
    ap.add_argument("--skip-rounds", action="store_true", help="skip the multi-round extra")
    ap.add_argument("--skip-heads", action="store_true", help="skip the gated / recurrent head extra")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the round's calls directly, without a CUDA graph")
    ap.add_argument("--phase-traffic", type=float, default=None,
                    help="dram bytes per draft phase launch from an ncu capture (reported as roofline.traffic)")
    ap.add_argument("--tv-rows", type=int, default=None,
                    help="time only the TV and training-loss kernels on this many training rows")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3
    if args.tv_rows is not None:
        run_tv_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
