#!/usr/bin/env python
"""Benchmark: exact attention forward + backward on GB300, one JSON line on rank 0.

A step is one pass of the whole path on one batch: fa_fwd (O, LSE), fa_bwd_preprocess
(D = rowsum(dO*O)) and fa_bwd (dQ, dK, dV), on the headline workload B=2, H=16,
N=8192, d=128, bf16, causal, unless --workload names another. FLOPs follow the
convention 4*B*H*N^2*d for the forward (halved when causal) and 2.5x that for the
backward. The inputs and outputs (8 tensors of 67 MB) exceed the 129 MB L2, so no
flush runs between steps.

--impl reference times the fp64 CPU oracle instead (a deliberately slow baseline),
one head of the workload per step, on the host cores.

Multi-GPU (torchrun): each rank runs its own copy of the workload (attention heads are
independent; no collective on the data path); value = all ranks' FLOPs / max time.
"""
import os
import platform

os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

import argparse  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOP/s (bf16, N=8192 d=128 causal), % of dense tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, c in zip(names, r[5:9]):
                if c.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def oracle_head_step(w, x, b, h):
    from oracle import attention as ora
    import numpy as np
    args = [x[n][b, h].astype(np.float64) for n in ("q", "k", "v", "do")]
    return ora.head_backward(*args, w.scale, w.causal)


def cpu_model():
    """The host CPU's model name as lscpu reports it (/proc/cpuinfo as a fallback)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine() or "unknown"


def cpu_baseline(w, x, budget_s=12.0, keep=None, keep_max=32):
    """The oracle, as it stands, on whole heads of the workload until ~budget_s have passed
    (every head at most once; batches taken in turn). With ``keep`` (a list), the outputs of
    the first ``keep_max`` heads are appended to it as ((b, h), outputs)."""
    flop_head = (w.fwd_flop() + w.bwd_flop()) / (w.B * w.H)
    t0 = time.perf_counter()
    n = 0
    while n < w.B * w.H and (n == 0 or (time.perf_counter() - t0) < budget_s):
        b, h = n % w.B, n // w.B
        r = oracle_head_step(w, x, b, h)
        if keep is not None and len(keep) < keep_max:
            keep.append(((b, h), r))
        n += 1
    dt = time.perf_counter() - t0
    return {"value": flop_head * n / dt / 1e12, "unit": "TFLOP/s",
            "cores": int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1)), "cpu": cpu_model(),
            "kind": "oracle",
            "sample": f"{n} whole head(s) of the workload (fwd+bwd, fp64 numpy), {dt:.1f} s; "
                      f"FLOPs counted by the same convention as the GPU line"}


def oracle_parity(w, ref_heads, got):
    """Errors of the timed run's outputs against the oracle, on the heads the CPU baseline
    computed, in the metrics and bounds of the parity tests: bf16 O and LSE max-abs (2e-2,
    1e-3) and dQ, dK, dV relative Frobenius (2e-2); fp32 max-abs 1e-4 on all five."""
    import numpy as np
    bf16 = w.dtype == "bf16"
    err = {"o": 0.0, "lse": 0.0, "dq": 0.0, "dk": 0.0, "dv": 0.0}
    for (b, h), r in ref_heads:
        for n in err:
            g = got[n][b, h].float().cpu().numpy().astype(np.float64)
            if bf16 and n in ("dq", "dk", "dv"):
                e = float(np.linalg.norm(g - r[n]) / max(float(np.linalg.norm(r[n])), 1e-300))
            else:
                e = float(np.abs(g - r[n]).max())
            err[n] = max(err[n], e)
    bound = ({"o": 2e-2, "lse": 1e-3, "dq": 2e-2, "dk": 2e-2, "dv": 2e-2} if bf16
             else dict.fromkeys(err, 1e-4))
    kind = {n: ("rel_fro" if bf16 and n in ("dq", "dk", "dv") else "max_abs") for n in err}
    return {"heads": [list(bh) for bh, _ in ref_heads], "error": err, "metric": kind, "bound": bound,
            "pass": bool(ref_heads) and all(err[n] <= bound[n] for n in err)}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from exact_attention_02_gb300.workloads import make_inputs
    x = make_inputs(w)
    flop_head = (w.fwd_flop() + w.bwd_flop()) / (w.B * w.H)
    for i in range(args.warmup):
        oracle_head_step(w, x, 0, i % w.H)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_head_step(w, x, (i // w.H) % w.B, i % w.H)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = flop_head / dt / 1e12
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "step": "one whole head (fwd+bwd) of the workload per step, fp64 numpy oracle on the host"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "cpu": cpu_model(), "kind": "oracle",
                         "sample": "one head of the workload per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def count_launches(step):
    """Kernels one step launches, counted with the CUDA activity profiler (CUPTI)."""
    import torch
    try:
        from torch.profiler import ProfilerActivity, profile
        with profile(activities=[ProfilerActivity.CPU, ProfilerActivity.CUDA]) as prof:
            step()
            torch.cuda.synchronize()
        evs = list(prof.events())
        kern = [e.name for e in evs if "CUDA" in str(getattr(e, "device_type", "")).upper()]
        ours = [n for n in kern if "fa::" in n or "_ZN2fa" in n or "fa_" in n]
        if not ours:
            seen = sorted({f"{getattr(e, 'device_type', '?')}:{e.name[:60]}" for e in evs})[:12]
            return None, ["no library kernels seen by the profiler"] + seen
        return len(ours), sorted(set(n.split("(")[0][:120] for n in ours))
    except Exception as e:  # profiler unavailable: report nothing rather than guess
        return None, [f"profiler unavailable: {e}"]


class _Named:
    """A workload known only by name (the split-KV and FP8 lines)."""
    def __init__(self, name):
        self.name = name


L2_BYTES = 129e6  # GB300 L2 (nominal)


def l2_plan(working_bytes):
    """Whether timed steps flush L2 first: only when the step's data could stay resident
    between steps (less than twice the L2); returns (flush, note for the config)."""
    if working_bytes >= 2 * L2_BYTES:
        return False, f"no flush: the step's tensors ({working_bytes / 1e6:.0f} MB) exceed twice the 129 MB L2"
    return True, (f"L2 flushed before every timed step (a 256 MB write, outside the events): the step's "
                  f"tensors ({working_bytes / 1e6:.0f} MB) are under twice the 129 MB L2")


def clocked_loop(step, steps, soak_s, flush=None):
    """Runs `step` for soak_s seconds untimed while the clock sampler starts, then `steps`
    timed steps on the current stream; returns (ms per step, clock record). With `flush`, it
    runs before every timed step and the time is the sum of the steps' own events."""
    import torch
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    torch.cuda.synchronize()
    clocks.start()
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < soak_s:
        for _ in range(8):
            step()
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for e0, e1 in ev:
        if flush is not None:
            flush()
        e0.record(stream)
        step()
        e1.record(stream)
    b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if flush is not None:
        ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
    else:
        ms = a.elapsed_time(b) / steps
    return ms, dict(clk, window=f"{soak_s:.1f} s of untimed steps, then the timed region")


def recorded_traffic(kernel, w):
    """DRAM bytes per launch from profiles/traffic.json, if recorded for this workload and the
    kernel's sources are unchanged since the capture; else None."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            recs = json.load(f)
        rec = recs.get(f"{kernel}@{w.name}") or recs.get(kernel)  # a record for this workload first
        if not rec or rec["workload"] != w.name:
            return None
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["source_sha256"]:
            return None
        return rec["captured_bytes"] * rec["scale"]
    except (OSError, KeyError, ValueError):
        return None


def run_ours(args, w):
    import numpy as np
    import torch
    import torch.distributed as dist

    import exact_attention_02_gb300 as fa
    from exact_attention_02_gb300.build import build
    from exact_attention_02_gb300.parallel import max_over_ranks
    from exact_attention_02_gb300.workloads import make_inputs

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
    fa.lib()
    fa.fa_set_bwd_dq_mode({"auto": fa.FA_BWD_DQ_AUTO, "atomic": fa.FA_BWD_DQ_ATOMIC,
                           "separate": fa.FA_BWD_DQ_SEPARATE}[args.dq_mode])
    dev = torch.device("cuda", local)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    x = make_inputs(w)
    host = {n: torch.from_numpy(x[n]).to(tdt).pin_memory() for n in ("q", "k", "v", "do")}
    q, k, v, do = (host[n].to(dev) for n in ("q", "k", "v", "do"))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    D = torch.empty_like(lse)
    ws_bytes = fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d, tdt)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    esz = 2 if w.dtype == "bf16" else 4
    # Q, K, V, O, dO, dQ, dK, dV, the fp32 dQ accumulator, LSE and D
    working = 8 * w.B * w.H * w.N * w.d * esz + w.B * w.H * w.N * w.d * 4 + 2 * w.B * w.H * w.N * 4
    flush_l2, l2_note = l2_plan(working)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush_l2 else None

    def fwd():
        fa.fa_fwd(q, k, v, w.causal, w.scale, o=o, lse=lse)

    def pre():
        fa.fa_bwd_preprocess(o, do, D=D)

    def bwd():
        fa.fa_bwd(q, k, v, o, do, lse, w.causal, w.scale, D=D, dq=dq, dk=dk, dv=dv, workspace=ws)

    def step():
        fwd()
        pre()
        bwd()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    launches, kernel_names = (None, ["not counted (--no-count)"]) if args.no_count else count_launches(step)
    launch_source = "CUDA activity profiler"
    if launches is None and not args.no_count:
        # the profiler saw nothing: count by the library's launch sequence instead
        seq = dict(fa.BF16_KERNELS) if w.dtype == "bf16" else fa.FP32_KERNELS
        if w.dtype == "bf16" and args.dq_mode == "separate":
            seq["fa_bwd"] = ["fa_bwd_wide_kernel", "fa_bwd_dq_kernel"]
        kernel_names = [k for e in ("fa_fwd", "fa_bwd_preprocess", "fa_bwd") for k in seq[e]]
        launches = len(kernel_names)
        launch_source = "library launch sequence (profiler saw no kernels); ncu launch list in profiles/ agrees"

    peaks, peak_src = load_peaks()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    # keep the GPU under the same load for a moment so the sampler sees it before the
    # timed region starts (the timed region itself may be shorter than one sample period)
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:
        for _ in range(8):
            step()
        torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        e = ev[i]
        if flush_l2:
            flush_buf.zero_()
        e[0].record(stream)
        fwd()
        e[1].record(stream)
        pre()
        e[2].record(stream)
        bwd()
        e[3].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    if flush_l2:  # the steps' own time, without the flushes between them
        ms = statistics.mean(e[0].elapsed_time(e[3]) for e in ev)
    else:
        ms = t_start.elapsed_time(t_end) / args.steps
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    pre_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    bwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    ms, fwd_ms, pre_ms, bwd_ms = max_over_ranks([ms, fwd_ms, pre_ms, bwd_ms], device=dev)
    status = fa.fa_get_last_device_status()
    if status != fa.FA_OK:
        raise RuntimeError(f"device status {fa.error_string(status)}")

    flop = w.fwd_flop() + w.bwd_flop()
    value = world * flop / (ms * 1e-3) / 1e12

    # end to end: pinned host inputs in, results (O, LSE, dQ, dK, dV) back to pinned host memory
    e2e = None
    e2e_out = None
    if not args.no_e2e:
        out_host = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                    for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in out_host.values())

        if w.dtype == "bf16":
            # the library's host-tensor entry point: copies of one head group overlap the
            # kernels of another (fa_fwd_bwd_host, default schedule: five head groups in
            # the ratio 1:2:2:2:1)
            e2e_path = "fa_fwd_bwd_host (C ABI on pinned host tensors; copies overlapped with kernels)"
            hws = torch.empty(fa.fa_fwd_bwd_host_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                              device=dev)
            outs = tuple(out_host[n] for n in ("o", "lse", "dq", "dk", "dv"))

            def e2e_step():
                fa.fa_fwd_bwd_host(host["q"], host["k"], host["v"], host["do"], w.causal, w.scale, out=outs,
                                   workspace=hws, stream=stream)
        else:
            e2e_path = "copies and device entry points in sequence on one stream"

            def e2e_step():
                for n, dst in (("q", q), ("k", k), ("v", v), ("do", do)):
                    dst.copy_(host[n], non_blocking=True)
                step()
                for n, src in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items():
                    out_host[n].copy_(src, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(3, args.steps // 2)
        a.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a.elapsed_time(b) / n_e2e
        e2e_ms = max_over_ranks([e2e_ms], device=dev)[0]
        e2e = {"value": world * flop / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "path": e2e_path}
        e2e_out = out_host

    rows = w.B * w.H * w.N
    pre_bytes = 2 * rows * w.d * esz + rows * 4
    kern = {"fa_fwd": fwd_ms, "fa_bwd": bwd_ms, "fa_bwd_preprocess": pre_ms}
    dominant = max(kern, key=kern.get)
    bound = fa.BF16_KERNEL_BOUND[dominant] if w.dtype == "bf16" else ("hbm" if dominant == "fa_bwd_preprocess" else "alu")
    dom_flop = {"fa_fwd": w.fwd_flop(), "fa_bwd": w.bwd_flop()}.get(dominant)
    if bound == "tensor":
        # The burst figure: the kernel runs in a timed region of well under a second at the
        # maximum SM clock, while the sustained figure was taken over seconds under the
        # power cap at a lower clock. The sustained fraction is reported beside it.
        peak = peaks["bf16_tflops"]
        peak_desc = f"bf16 dense, burst ({peak_src})"
        unit = "TFLOP/s"
        achieved = dom_flop / (kern[dominant] * 1e-3) / 1e12
    elif bound == "alu":
        # FFMA path: 152 SMs x 128 FMA/clk x 2 FLOP x max SM clock
        peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        peak_desc = "fp32 FFMA: 152 SMs x 128 FMA/clk x 2 x max SM clock (derived)"
        unit = "TFLOP/s"
        achieved = dom_flop / (kern[dominant] * 1e-3) / 1e12
    else:
        achieved = pre_bytes / (pre_ms * 1e-3) / 1e9
        peak, unit, peak_desc = peaks["hbm_gbs"], "GB/s", f"HBM copy ({peak_src})"
    # the records describe the default kernels; another dQ mode runs other kernels
    traffic = recorded_traffic(dominant, w) if args.dq_mode == "auto" or dominant != "fa_bwd" else None
    roofline = {"kernel": dominant, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "peak_source": peak_desc, "traffic": traffic,
                "traffic_note": "DRAM bytes per launch from profiles/traffic.json (ncu, scaled by heads)"
                if traffic else "no capture recorded for this kernel build and workload"}
    if bound == "tensor":
        sus = peaks.get("bf16_tflops_sustained")
        roofline["frac_burst"] = achieved / peaks["bf16_tflops"]
        roofline["frac_sustained"] = achieved / sus if sus else None

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "scale": w.scale, "parallelism": f"replicas x{world} (heads independent, no collective)",
                   "dq_mode": args.dq_mode, "l2": l2_note},
        "fwd": {"ms": fwd_ms, "tflops": w.fwd_flop() / (fwd_ms * 1e-3) / 1e12},
        "bwd": {"ms": pre_ms + bwd_ms, "tflops": w.bwd_flop() / ((pre_ms + bwd_ms) * 1e-3) / 1e12,
                "note": "preprocess + fa_bwd"},
        "preprocess": {"ms": pre_ms, "gbs": pre_bytes / (pre_ms * 1e-3) / 1e9,
                       "frac_hbm": pre_bytes / (pre_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        "roofline": roofline,
        "gpu_launches": None if launches is None else launches * args.steps,
        "kernels_per_step": kernel_names,
        "launch_count_source": launch_source,
        "clocks": dict(clk, window=f"{args.soak_s:.1f} s of untimed steps, then the timed region"),
        "e2e": e2e,
    }
    # fractions of the dense bf16 tensor peak: burst (the headline) and sustained
    tpeak, spk = peaks["bf16_tflops"], peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    for key, tf in (("fwd", line["fwd"]["tflops"]), ("bwd", line["bwd"]["tflops"])):
        line[key]["frac_tensor_peak"] = tf / tpeak if w.dtype == "bf16" else None
        line[key]["frac_tensor_peak_sustained"] = tf / spk if w.dtype == "bf16" else None
    line["frac_tensor_peak"] = value / world / tpeak if w.dtype == "bf16" else None
    line["frac_tensor_peak_sustained"] = value / world / spk if w.dtype == "bf16" else None
    line["tensor_peak"] = {"burst": tpeak, "sustained": spk, "source": peak_src,
                           "headline": "burst: the timed region lasts well under a second"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ref_heads = []
        line["cpu_baseline"] = cpu_baseline(w, x, keep=ref_heads)
        try:  # the oracle's heads double as a full-size parity check of the timed outputs
            line["oracle_parity"] = oracle_parity(w, ref_heads, dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv))
        except Exception as e:  # a failed check is reported, never fatal to the bench line
            line["oracle_parity"] = {"error": f"{type(e).__name__}: {e}"}
        if e2e_out is not None:  # and of what the end-to-end leg copied back to the host
            try:
                line["e2e"]["oracle_parity"] = oracle_parity(w, ref_heads, e2e_out)
            except Exception as e:
                line["e2e"]["oracle_parity"] = {"error": f"{type(e).__name__}: {e}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_splitkv(args):
    """Few-query forward (fa_fwd_splitkv) on [B,H,Nq,d] queries against [B,H,Nk,d] keys/values.

    HBM-bound: the algorithmic bytes are one read of K and V plus Q, O and LSE; the line
    reports them per second against the measured HBM copy bandwidth."""
    import numpy as np
    import torch

    import exact_attention_02_gb300 as fa
    from exact_attention_02_gb300.build import build
    from exact_attention_02_gb300.workloads import round_to_bf16

    B, H, Nq, Nk, d, c = (int(v) for v in args.splitkv.split(","))
    build()
    fa.lib()
    rng = np.random.default_rng(0)
    q, k, v = (torch.from_numpy(round_to_bf16(rng.standard_normal(shape, dtype=np.float32))).cuda().to(torch.bfloat16)
               for shape in ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d)))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(16, fa.lib().fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, 0)), dtype=torch.uint8,
                     device="cuda")

    def step():
        fa.fa_fwd_splitkv(q, k, v, bool(c), o=o, lse=lse, workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    nbytes = 2 * B * H * Nk * d * 2 + 2 * B * H * Nq * d * 2 + B * H * Nq * 4
    flush_l2, l2_note = l2_plan(nbytes)
    fbuf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if flush_l2 else None
    ms, clk = clocked_loop(step, args.steps, args.soak_s, flush=fbuf.zero_ if flush_l2 else None)
    peaks, src = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    flop = 4.0 * B * H * Nq * Nk * d
    workload = f"splitkv_b{B}h{H}_q{Nq}_k{Nk}_d{d}" + ("_causal" if c else "")
    # one traffic record per head dimension of the tensor-core partial kernel
    kernel = "fa_fwd_splitkv_tc" if d == 128 else "fa_fwd_splitkv_tc_d64"
    print(json.dumps({
        "metric": "split-KV forward HBM GB/s (few queries against a long key/value sequence)",
        "value": gbs, "unit": "GB/s", "ms_per_step": ms, "steps": args.steps, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload,
                   "B": B, "H": H, "Nq": Nq, "Nk": Nk, "d": d, "causal": bool(c),
                   "l2": l2_note},
        "tflops": flop / (ms * 1e-3) / 1e12,
        "clocks": clk,
        "roofline": {"kernel": kernel, "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "peak_source": f"HBM copy ({src})",
                     "traffic": recorded_traffic(kernel, _Named(workload))},
        "gpu_launches": 2 * args.steps, "kernels_per_step": fa.SPLITKV_KERNELS,
    }), flush=True)
    return 0


def run_fp8(args):
    """Forward on e4m3 inputs (fa_fwd_fp8) for a B,H,N,d,causal shape (d = 128).

    Tensor-bound like the bf16 forward and counted with the same FLOP convention; the
    peak is the measured dense bf16 burst rate times 2, the nominal fp8/bf16 ratio of the
    part (4.5 / 2.25 PFLOP/s); the fraction of 2 x the sustained rate is reported beside it."""
    import torch

    import exact_attention_02_gb300 as fa
    from exact_attention_02_gb300.build import build
    from exact_attention_02_gb300.workloads import make_fp8_inputs

    B, H, N, d, c = (int(v) for v in args.fp8.split(","))
    build()
    fa.lib()
    (q8, k8, v8), desc = make_fp8_inputs(B, H, N, d, seed=0)
    q, k, v = (torch.from_numpy(x).cuda() for x in (q8, k8, v8))
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")

    def step():
        fa.fa_fwd_fp8(q, k, v, desc, bool(c), o=o, lse=lse)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    in_bytes = 3 * B * H * N * d
    flush_l2, l2_note = l2_plan(in_bytes + B * H * N * d * 2 + B * H * N * 4)
    fbuf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if flush_l2 else None
    ms, clk = clocked_loop(step, args.steps, args.soak_s, flush=fbuf.zero_ if flush_l2 else None)
    peaks, src = load_peaks()
    flop = 4.0 * B * H * N * N * d / (2 if c else 1)
    tf = flop / (ms * 1e-3) / 1e12
    peak = 2 * peaks["bf16_tflops"]
    peak_sus = 2 * peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    workload = f"fp8_b{B}h{H}_n{N}_d{d}" + ("_causal" if c else "")
    print(json.dumps({
        "metric": "attention fwd TFLOP/s on e4m3 inputs (fa_fwd_fp8)", "value": tf, "unit": "TFLOP/s",
        "ms_per_step": ms, "steps": args.steps, "higher_is_better": True, "dtype": "e4m3 (fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": workload, "B": B, "H": H, "N": N,
                   "d": d, "causal": bool(c),
                   "l2": l2_note},
        "roofline": {"kernel": "fa_fwd_tc_kernel<128, e4m3>", "bound": "tensor", "achieved": tf, "peak": peak,
                     "unit": "TFLOP/s", "frac": tf / peak, "frac_sustained": tf / peak_sus,
                     "peak_source": f"2 x dense bf16 burst ({src}); nominal fp8/bf16 ratio",
                     "traffic": recorded_traffic("fa_fwd_fp8", _Named(workload))},
        "clocks": clk,
        "gpu_launches": args.steps, "kernels_per_step": fa.FP8_KERNELS,
    }), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--shape", default=None,
                    help="ad-hoc bf16 workload B,H,N,d,causal (e.g. for a small profiler capture)")
    ap.add_argument("--splitkv", default=None,
                    help="measure fa_fwd_splitkv instead: B,H,Nq,Nk,d,causal (prints its own JSON line)")
    ap.add_argument("--fp8", default=None,
                    help="measure fa_fwd_fp8 instead: B,H,N,d,causal (prints its own JSON line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-count", action="store_true", help="skip the profiler launch count")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="extra untimed steps (seconds) run under the clock sampler before the timed region")
    ap.add_argument("--dq-mode", choices=["auto", "atomic", "separate"], default="auto",
                    help="how fa_bwd computes dQ (fa_set_bwd_dq_mode): by default the library's choice")
    args = ap.parse_args()
    from exact_attention_02_gb300.workloads import HEADLINE, WORKLOADS, Workload
    if args.shape:
        B, H, N, d, c = (int(v) for v in args.shape.split(","))
        w = Workload(f"b{B}h{H}_n{N}_d{d}_bf16" + ("_causal" if c else ""), B, H, N, d, "bf16", bool(c))
    else:
        w = WORKLOADS[args.workload or HEADLINE]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.splitkv:
        return run_splitkv(args)
    if args.fp8:
        return run_fp8(args)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
