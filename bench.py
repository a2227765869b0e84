"""Benchmark of the SDM forward step (addressing + scan) on GB300.

One step = one sdm_forward over one batch of the workload (default
``gdn_matched``: B=8, H=8, T=4096, N=65536 slots, W=R=64, d_v=128, bf16
inputs, fp32 table of 2 GiB).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--variant forward|fig2|logged|decode] [--workload NAME]

--impl reference times the CPU oracle (the plain C++ restatement of the
method) on this machine's host cores, on a bounded sample of the same workload.
Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import WORKLOADS, generate  # noqa: E402

METRIC = "SDM forward tokens/s on 1 GB300; scan-kernel GB/s as % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0


def scan_bytes_per_token_head(w) -> int:
    """Algorithmic bytes the scan must move per token-head: W rows read and
    written, R rows read (d_v fp32 each), v and the two gates (input dtype),
    slot indices and weights (8 B per slot), and y (d_v fp32)."""
    ib = 2 if w.bf16 else 4
    return (2 * w.W + w.R) * w.d_v * 4 + w.d_v * ib + 2 * ib + (w.W + w.R) * 8 + w.d_v * 4


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


L2_BYTES = 129 * 10**6            # GB300 L2 capacity (nominal)


def l2_copy_gbs(dev) -> float:
    """Live L2 reference: an in-place elementwise pass (read + write) over
    one 64 MiB buffer, which stays resident in L2; 20 passes per CUDA-graph
    replay so launch gaps do not count; best of 5 replays, CUDA events."""
    n = 64 * 2**20 // 4
    a = torch.ones(n, dtype=torch.float32, device=dev)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(3):
            a.mul_(1.0)
        with torch.cuda.graph(graph, stream=side):
            for _ in range(20):
                a.mul_(1.0)
    torch.cuda.synchronize(dev)
    for _ in range(3):
        graph.replay()
    best = float("inf")
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        best = min(best, e0.elapsed_time(e1) / 20)
    return 2 * n * 4 / (best / 1e3) / 1e9


def row_ceiling_gbs(sdm, w, dev, M) -> tuple[float, dict]:
    """Live ceiling for the scan's memory traffic: sdm_measure_row_traffic
    moves the scan's row pieces (W + R fetched, W stored per step of every
    (chain, column slice) unit, rows uniform over the chain's table, the
    scan's slice width) with no arithmetic.  Best of 3 CUDA-event-timed
    calls after one warm-up, on a scratch table the size of the state."""
    chains = w.B * w.H
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cw = 32 if (w.d_v % 32 == 0 and chains * (w.d_v // 32) >= sms) else 16
    steps = min(w.T, 8192)
    src = M.view(chains, w.N, w.d_v)
    dst = torch.empty_like(src)
    stream = torch.cuda.current_stream(dev)
    run = lambda: sdm.sdm_measure_row_traffic(src, dst, cw, steps, w.W + w.R, w.W, seed=7,
                                              stream=stream)
    nbytes = run()
    best = float("inf")
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        torch.cuda.synchronize(dev)
        best = min(best, a.elapsed_time(b))
    del dst
    desc = {"col_slice": cw, "units": chains * (w.d_v // cw), "steps": steps,
            "loads_per_step": w.W + w.R, "stores_per_step": w.W, "bytes": nbytes}
    return nbytes / (best / 1e3) / 1e9, desc


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed work runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, pw = [], [], []
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        # Samples under load: power within 40% of the highest seen.
        hi = max(pw) if pw else 0.0
        load = [s for s, p in zip(sm, pw) if p >= 0.6 * hi] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(load)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_workload(w, rank: int):
    """Each rank runs its own batch of the same shape (weak scaling)."""
    return w.with_(seed=w.seed + 1000 * rank) if rank else w


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time: the job's time."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank_step: int, world: int, steps: int, ms: float) -> float:
    """Whole-job throughput: tokens of all ranks over the max-over-ranks time."""
    return tokens_per_rank_step * world * steps / (ms / 1e3)


def traffic_for(kernel_srcs):
    """DRAM bytes per sdm_scan call recorded by an ncu capture of these exact
    kernel sources (profiles/traffic.json keyed by the sha256 of the files'
    concatenated bytes); None if a kernel changed since."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        hs = hashlib.sha256()
        for src in kernel_srcs:
            with open(src, "rb") as f:
                hs.update(f.read())
        h = hs.hexdigest()
        ent = rec.get(h)
        return None if ent is None else float(ent["bytes_per_launch"])
    except Exception:
        return None


def oracle_sample_rate(w, budget_s: float, seed_offset: int = 0):
    """Time the CPU oracle (single thread) on chain (0, 0) of the workload,
    growing the token count until about `budget_s` seconds of work.  Returns
    (equivalent tokens/s of the whole workload, description)."""
    import oracle as O
    T = min(64, w.T)
    spent = 0.0
    last = None
    while True:
        ws = w.with_(B=1, H=1, T=T, seed=w.seed + seed_offset)
        x = generate(ws)
        sh = O.Shape(1, 1, T, w.n_sub, w.d_h, w.d_v, w.W, w.R, k_w=w.k_w, k_r=w.k_r,
                     score_kind=w.score_kind, idw_eps=w.idw_eps, update_form=w.update_form)
        args = [x[k].float().numpy() for k in ("q_w", "q_r", "K", "alpha", "beta", "v")]
        t0 = time.perf_counter()
        O.forward(sh, *args, x["M0"].numpy())
        dt = time.perf_counter() - t0
        spent += dt
        last = (T, dt)
        if spent >= budget_s or T >= w.T or dt * 2 > budget_s - spent:
            break
        T = min(w.T, T * 2)
    T, dt = last
    # One token of the workload is H token-heads (all heads of the token).
    tok_per_s = (T / dt) / w.H
    desc = (f"oracle forward (subscores, selection, scan) of chain (b=0,h=0), first {T} of "
            f"{w.T} tokens, {dt:.2f} s on 1 thread; rate scaled to tokens of all {w.H} heads")
    return tok_per_s, desc, T, dt


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() in ("Model name", "Model"):
                name = ln.split(":", 1)[1].strip()
                if name and not name.isdigit():
                    return name
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def oracle_all_cores_rate(w, T: int, threads: int):
    """The same single-threaded oracle routine on `threads` independent
    (b, h) chains at once, one chain per host thread (the C++ oracle runs
    outside the interpreter lock), each on the first T tokens of its chain.
    Returns (equivalent tokens/s of the whole workload, description)."""
    import concurrent.futures as cf

    import oracle as O
    O.build()
    chains = [(i % w.B, (i // w.B) % w.H) for i in range(threads)]
    jobs = []
    for i, (b, h) in enumerate(chains):
        # Chain i of the sample: its own seeded draw of the workload's shape
        # (chains are independent; a fresh seed per thread stands in for (b, h)).
        ws = w.with_(B=1, H=1, T=T, seed=w.seed + 7919 * (i + 1))
        x = generate(ws)
        sh = O.Shape(1, 1, T, w.n_sub, w.d_h, w.d_v, w.W, w.R, k_w=w.k_w, k_r=w.k_r,
                     score_kind=w.score_kind, idw_eps=w.idw_eps, update_form=w.update_form)
        args = [x[k].float().numpy() for k in ("q_w", "q_r", "K", "alpha", "beta", "v")]
        jobs.append((sh, args, x["M0"].numpy()))
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        list(ex.map(lambda j: O.forward(j[0], *j[1], j[2]), jobs))
        dt = time.perf_counter() - t0
    tok_per_s = threads * T / dt / w.H
    desc = (f"the same oracle forward on {threads} independent chains at once, one per host "
            f"thread, first {T} tokens each, {dt:.2f} s wall; rate scaled to tokens of all "
            f"{w.H} heads")
    return tok_per_s, desc


def cpu_baseline_entry(w, budget_s: float):
    """cpu_baseline of the bench line: the oracle on one thread (the plain
    routine as it stands) and the same routine on every host core over
    independent chains, with the core count and the CPU model."""
    rate, desc, T, dt = oracle_sample_rate(w, budget_s)
    nproc = os.cpu_count() or 1
    # One chain's table in fp32 and in the oracle's double copy; keep the
    # threads' tables within 8 GB of host memory.
    per_chain = w.N * w.d_v * 12
    threads = max(1, min(nproc, (8 << 30) // per_chain))
    # Each thread's sample as long as the single-thread one (about the same wall time).
    rate_all, desc_all = oracle_all_cores_rate(w, T, threads)
    return {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc,
            "all_cores": {"value": rate_all, "unit": "tokens/s", "cores": threads,
                          "sample": desc_all},
            "nproc": nproc, "cpu_model": cpu_model()}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle as O
    O.build()
    steps, warm = args.steps, args.warmup
    # Per-step sample sized so the whole run stays within ~2 minutes.
    calib_rate, _, _, _ = oracle_sample_rate(w, 2.0)
    per_step_s = max(0.05, 120.0 / max(1, steps + warm))
    T = max(8, min(w.T, int(calib_rate * w.H * per_step_s)))
    sample = w.with_(B=1, H=1, T=T)
    x = generate(sample)
    sh = O.Shape(1, 1, T, w.n_sub, w.d_h, w.d_v, w.W, w.R, k_w=w.k_w, k_r=w.k_r,
                 score_kind=w.score_kind, idw_eps=w.idw_eps, update_form=w.update_form)
    arrays = [x[k].float().numpy() for k in ("q_w", "q_r", "K", "alpha", "beta", "v")]
    for _ in range(warm):
        O.forward(sh, *arrays, x["M0"].numpy())
    t0 = time.perf_counter()
    for _ in range(steps):
        O.forward(sh, *arrays, x["M0"].numpy())
    el = time.perf_counter() - t0
    tok_per_s = (steps * T / w.H) / el
    desc = (f"per step: oracle forward of one chain, {T} tokens ({T} token-heads) of the "
            f"{w.name} workload on 1 thread; rate scaled to tokens of all {w.H} heads")
    line = {
        "impl": "reference", "metric": METRIC, "value": tok_per_s, "unit": "tokens/s",
        "n_gpus": ws, "steps": steps, "warmup": warm,
        "ms_per_step": el / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": line_config(w, args, ws),
        "cpu_baseline": {"value": tok_per_s, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": desc, "nproc": os.cpu_count() or 1,
                         "cpu_model": cpu_model()},
        "e2e": {"value": tok_per_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def line_config(w, args, ws: int):
    """`config` of a bench line (the same keys for both arms)."""
    return dict(config_of(w), variant=args.variant,
                parallelism=f"dp{ws}" if ws > 1 else "single")


def config_of(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "N": w.N, "n_sub": w.n_sub,
            "d_h": w.d_h, "d_v": w.d_v, "W": w.W, "R": w.R,
            "inputs": "bf16" if w.bf16 else "f32", "state": "f32",
            "score": "dot" if w.score_kind == 0 else "inverse-distance",
            "global_batch": w.B, "seq_len": w.T, "l2": l2_note(w)}


def l2_note(w) -> str:
    """How the timed steps stand to L2 (no flush between steps either way)."""
    table = w.B * w.H * w.N * w.d_v * 4
    if table > 2 * L2_BYTES:
        return f"inputs larger than L2 (fp32 table {table / 2**30:.2f} GiB)"
    return (f"fp32 table of {table / 2**20:.1f} MiB fits or nearly fits in L2 ({L2_BYTES / 1e6:.0f} MB): "
            "no flush between steps, each step reads the state the previous one left, as "
            "the recurrence does; the line adds l2_roofline against a live L2 reference")


def variant_workload(args):
    """The workload a --variant runs on (forward: --workload as given)."""
    w = WORKLOADS[args.workload]
    if args.variant == "fig2":
        w = w.with_(update_form=1)
    if args.variant == "decode" and w.T != 1:
        w = WORKLOADS["decode_l08"]
    return w


def run_ours(args, w):
    import sparse_state_linear_gb300 as sdm
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    sdm.lib()
    rw = rank_workload(w, rank)
    big = rw.B * rw.H * rw.N * rw.d_v * 4 > (8 << 30)
    x = generate(rw, device=dev if big else None)
    g = {k: t.to(dev) for k, t in x.items() if k != "M0"}
    M = x["M0"].to(dev)
    del x
    sh = sdm.make_shape(w.B, w.H, w.T, w.n_sub, w.d_h, w.d_v, w.W, w.R, k_w=w.k_w, k_r=w.k_r,
                        in_dtype=sdm.SDM_BF16 if w.bf16 else sdm.SDM_F32, score=w.score_kind,
                        idw_eps=w.idw_eps, update=w.update_form)
    BHT = (w.B, w.H, w.T)
    y = torch.empty(BHT + (w.d_v,), dtype=torch.float32, device=dev)
    idx_w = torch.empty(BHT + (w.W,), dtype=torch.int32, device=dev)
    idx_r = torch.empty(BHT + (w.R,), dtype=torch.int32, device=dev)
    wt_w = torch.empty(BHT + (w.W,), dtype=torch.float32, device=dev)
    wt_r = torch.empty(BHT + (w.R,), dtype=torch.float32, device=dev)
    wsp = torch.empty(max(16, sdm.sdm_workspace_size(sh)), dtype=torch.uint8, device=dev)
    undo = uws = None
    if args.variant == "logged":
        undo = torch.empty(BHT + (w.W, w.d_v), dtype=torch.float32, device=dev)
        uws = torch.empty(max(16, sdm.sdm_undo_workspace_size(sh)), dtype=torch.uint8,
                          device=dev)
    stream = torch.cuda.current_stream(dev)

    def address():
        sdm.sdm_address(sh, g["q_w"], g["q_r"], g["K"], idx_w, wt_w, idx_r, wt_r, stream=stream)

    def scan():
        if undo is not None:
            sdm.sdm_scan_logged(sh, idx_w, wt_w, idx_r, wt_r, g["alpha"], g["beta"], g["v"], M, y,
                                undo=undo, workspace=wsp, stream=stream)
        else:
            sdm.sdm_scan(sh, idx_w, wt_w, idx_r, wt_r, g["alpha"], g["beta"], g["v"], M, y,
                         workspace=wsp, stream=stream)

    def forward():
        if args.variant == "decode":
            sdm.sdm_decode(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"], M, y,
                           idx_w, wt_w, idx_r, wt_r, stream=stream)
        elif undo is not None:
            address()
            scan()
        else:
            sdm.sdm_forward(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"], M, y,
                            idx_w, wt_w, idx_r, wt_r, workspace=wsp, stream=stream)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        forward()
    torch.cuda.synchronize(dev)
    if sdm.sdm_get_device_status(stream) != 0:
        raise RuntimeError("device reported a failure during warm-up")

    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(dev.index)).split(",")[dev.index]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else dev.index
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    with ClockSampler(gpu_index) as clk:
        # ---- the timed region: K full forward steps.
        barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = ev(), ev()
        e0.record(stream)
        for _ in range(args.steps):
            forward()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        ms = max_over_ranks(e0.elapsed_time(e1), dev)
        status = sdm.sdm_get_device_status(stream)

        # ---- per-kernel durations (same stream, events around each call).
        def per_call(fn, n):
            evs = [(ev(), ev()) for _ in range(n)]
            for a, b in evs:
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize(dev)
            return sum(a.elapsed_time(b) for a, b in evs) / n

        nk = max(3, min(args.steps, 20))
        kernels = {}
        if args.variant == "decode":
            t_main = per_call(forward, nk)
            kernels["sdm_decode"] = t_main
        else:
            kernels["sdm_address"] = per_call(address, nk)
            t_main = per_call(scan, nk)
            kernels["sdm_scan_logged" if undo is not None else "sdm_scan"] = t_main
            if undo is not None:
                kernels["sdm_scan_undo"] = per_call(
                    lambda: sdm.sdm_scan_undo(sh, idx_w, undo, M, workspace=uws, stream=stream), nk)

        # ---- end to end through the public API with host buffers: every
        # step copies its inputs from pinned host memory and its y back.  The
        # copies run on two more streams (uploads, read-backs), double-
        # buffered, so step i's compute overlaps step i+1's upload and step
        # i-1's read-back (the table is carried in place, in order, on the
        # compute stream).
        names = ("q_w", "q_r", "alpha", "beta", "v")
        host = {k: g[k].cpu().pin_memory() for k in names}
        bufs = [{k: torch.empty_like(g[k]) for k in names} for _ in range(2)]
        y_dev = [torch.empty_like(y) for _ in range(2)]
        y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = y_host[0].numel() * y_host[0].element_size()
        ne = max(4, min(args.steps, 20))
        # Uploads and read-backs on streams of their own: the two directions
        # overlap each other as well as the compute.
        copy = torch.cuda.Stream(dev)
        copy_back = torch.cuda.Stream(dev)
        g_keep = dict(g)

        def run_e2e(n):
            up = [torch.cuda.Event() for _ in range(n)]
            done = [torch.cuda.Event() for _ in range(n)]
            down = [torch.cuda.Event() for _ in range(n)]

            def upload(i):
                with torch.cuda.stream(copy):
                    if i >= 2:
                        copy.wait_event(done[i - 2])         # buffer i%2 is free again
                    for k in names:
                        bufs[i % 2][k].copy_(host[k], non_blocking=True)
                    up[i].record(copy)

            def read_back(j):
                with torch.cuda.stream(copy_back):
                    copy_back.wait_event(done[j])
                    y_host[j % 2].copy_(y_dev[j % 2], non_blocking=True)
                    down[j].record(copy_back)

            # Step i+1's upload and step i-1's read-back are enqueued before
            # step i's compute: a forward of many launches can fill the launch
            # queue and block the host inside it, and the copies must not wait
            # behind that.
            upload(0)
            for i in range(n):
                if i + 1 < n:
                    upload(i + 1)
                if i >= 1:
                    read_back(i - 1)
                stream.wait_event(up[i])
                if i >= 2:
                    stream.wait_event(down[i - 2])         # y buffer i%2 was read back
                for k in names:
                    g[k] = bufs[i % 2][k]
                forward_to(y_dev[i % 2])
                done[i].record(stream)
            read_back(n - 1)
            return down[n - 1]

        def forward_to(ydst):
            if args.variant == "decode":
                sdm.sdm_decode(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"], M,
                               ydst, idx_w, wt_w, idx_r, wt_r, stream=stream)
            elif undo is not None:
                sdm.sdm_address(sh, g["q_w"], g["q_r"], g["K"], idx_w, wt_w, idx_r, wt_r,
                                stream=stream)
                sdm.sdm_scan_logged(sh, idx_w, wt_w, idx_r, wt_r, g["alpha"], g["beta"], g["v"],
                                    M, ydst, undo=undo, workspace=wsp, stream=stream)
            else:
                sdm.sdm_forward(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"],
                                M, ydst, idx_w, wt_w, idx_r, wt_r, workspace=wsp, stream=stream)

        if args.variant == "decode":
            # A decode step is tens of microseconds: one end-to-end step
            # (upload of the step's inputs, the decode, read-back of y) is
            # captured in a CUDA graph and replayed, so host launch overhead
            # does not stand in for the path.
            for k in names:
                g[k] = bufs[0][k]
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                def one_step():
                    for k in names:
                        bufs[0][k].copy_(host[k], non_blocking=True)
                    sdm.sdm_decode(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"],
                                   g["v"], M, y_dev[0], idx_w, wt_w, idx_r, wt_r, stream=side)
                    y_host[0].copy_(y_dev[0], non_blocking=True)
                one_step()
                torch.cuda.synchronize(dev)
                with torch.cuda.graph(graph, stream=side):
                    one_step()
            graph.replay()                         # replays run on the current stream
            torch.cuda.synchronize(dev)
            barrier()
            a, b = ev(), ev()
            a.record(stream)
            for _ in range(ne):
                graph.replay()
            b.record(stream)
            torch.cuda.synchronize(dev)
            e2e_ms = a.elapsed_time(b) / ne
        else:
            run_e2e(2)
            torch.cuda.synchronize(dev)
            barrier()
            a, b = ev(), ev()
            a.record(stream)
            copy.wait_event(a)                     # no upload starts before the timed region
            copy_back.wait_event(a)
            last = run_e2e(ne)
            stream.wait_event(last)
            b.record(stream)
            torch.cuda.synchronize(dev)
            e2e_ms = a.elapsed_time(b) / ne
        g.update(g_keep)
    if status != 0:
        raise RuntimeError(f"device reported status {status} in the timed region")

    tokens = w.B * w.T
    value = job_tokens_per_s(tokens, ws, args.steps, ms)
    peak, peak_kind = measured_peaks()
    bytes_launch = scan_bytes_per_token_head(w) * w.B * w.H * w.T
    if undo is not None:
        bytes_launch += w.B * w.H * w.T * w.W * w.d_v * 4      # the log rows
    achieved = bytes_launch / (t_main / 1e3) / 1e9
    kname = {"decode": "sdm_decode (fused addressing + write + read)",
             "logged": "sdm_scan_logged (plan + scan kernels, undo log)"}.get(
                 args.variant, "sdm_scan (plan + scan kernels)")
    traffic = None
    if args.variant in ("forward", "fig2") and w.name == "gdn_matched" and w.update_form == 0:
        csrc = os.path.join(ROOT, "sparse_state_linear_gb300", "csrc")
        traffic = traffic_for([os.path.join(csrc, "plan.cu"), os.path.join(csrc, "scan.cu")])
    launches = {"decode": 1, "logged": 3}.get(args.variant, 3 * sdm.sdm_forward_windows(sh))
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; bf16 inputs, fp32 table)" if w.bf16 else "synthetic (seeded, fp32)",
        "config": line_config(w, args, ws),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": kname,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": bytes_launch},
        "kernels_ms": kernels,
        "e2e": {"value": tokens * ws / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
    }
    table_bytes = w.B * w.H * w.N * w.d_v * 4
    if args.variant != "decode" and table_bytes <= 2 * L2_BYTES:
        # Tables that fit (tiny) or nearly fit (mid: 128 MiB) in L2: the scan
        # against the L2 copy rate as well.
        l2 = l2_copy_gbs(dev)
        line["l2_roofline"] = {"achieved": achieved, "peak": l2, "unit": "GB/s",
                               "frac": achieved / l2, "table_bytes": table_bytes,
                               "peak_source": "live: in-place elementwise pass over a "
                                              "64 MiB L2-resident buffer (read + write)"}
    if args.variant != "decode":
        # The scan's access pattern (random row pieces of W + R rows per step)
        # does not reach the sequential copy peak on HBM; the same pieces moved
        # with no arithmetic give the ceiling for that pattern.
        ceil, desc = row_ceiling_gbs(sdm, w, dev, M)
        line["row_ceiling"] = {"achieved": achieved, "peak": ceil, "unit": "GB/s",
                               "frac": achieved / ceil,
                               "peak_source": "live: sdm_measure_row_traffic (the scan's row "
                                              "pieces, no arithmetic), best of 3",
                               **desc}
    if ws == 1 and rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_entry(w, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gdn_matched", choices=sorted(WORKLOADS))
    ap.add_argument("--variant", default="forward", choices=["forward", "fig2", "logged", "decode"],
                    help="forward: sdm_forward (the headline); fig2: the same with the Fig. 2 "
                         "update form; logged: addressing + scan with the undo log (undo timed "
                         "apart); decode: sdm_decode on a one-token-per-sequence workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = variant_workload(args)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
