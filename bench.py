"""Benchmark of the fused norm hot path on GB300.

One step = one pass of the whole path over one batch: the LayerNorm forward
(bf16 in/out, fp32 gamma/beta, mu/rsigma saved) followed by the backward
(dx, then dgamma/dbeta reduced over all rows), on 16384 rows x 4096.
Inputs are resident in HBM when the timed region starts.  Timed steps run
back to back without an L2 flush: the inputs of one step (x and dz, 268 MB)
are larger than the 129 MB L2, so a step finds little of them there, and
every step pays for the dirty lines its predecessor left (the steady state
of a training loop).  The same step with a 512 MiB write between steps is
reported beside it (``l2_flushed``).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (test infrastructure, single-threaded C++) on the same workload.
Also reported, in ``detail``: every workload of the target table (forward and
backward separately, back to back and with L2 flushed, GB/s against the HBM
roofline).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

MAIN = "ln_bf16_16384x4096"
METRIC = "norm fwd/bwd rows/s and achieved HBM GB/s (% of 8 TB/s) at bf16 h=4096-12288"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000
NOMINAL_HBM_GBS = 8000.0
ESZ = {"f32": 4, "bf16": 2, "f16": 2}


# ---------------------------------------------------------------- algorithmic bytes

def fwd_bytes(w) -> int:
    """Each input read once, each output written once, weights counted once."""
    N, H, e, we = w.rows, w.hidden, ESZ[w.in_dtype], ESZ[w.w_dtype]
    b = N * H * e + H * we * (2 if w.norm == "layernorm" else 1)
    b += N * 4 * (2 if w.norm == "layernorm" else 1)          # mu, rsigma
    rowwise = w.scaling == "none" or w.layout != "colwise"
    colwise = w.scaling != "none" and w.layout != "rowwise"
    if w.scaling == "none":
        b += N * H * e
    else:
        b += N * H * (int(rowwise) + int(colwise))
        if w.scaling == "delayed":
            b += 4 + 4 + 4 * (int(rowwise) + int(colwise))   # scale, amax, scale_inv(s)
        else:
            b += (N * H // 32) * (int(rowwise) + int(colwise))
    return b


def bwd_bytes(w) -> int:
    N, H, e, we = w.rows, w.hidden, ESZ[w.in_dtype], ESZ[w.w_dtype]
    streams = 3 + (1 if w.dresidual else 0)                     # dz, x, (dres), dx
    b = streams * N * H * e + N * 4 * (2 if w.norm == "layernorm" else 1)
    b += H * we + H * we * (2 if w.norm == "layernorm" else 1)  # gamma; dgamma (+dbeta)
    return b


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi every 50 ms
    while started.  The benchmark samples over the same back-to-back steps
    just before and just after the timed steps, not during them: nvidia-smi
    polling during the timed steps was measured to slow them (about 8 % per
    step in three of four runs)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, args=(self.proc,), daemon=True).start()
            n0, t0 = len(self.lines), time.monotonic()
            while len(self.lines) == n0 and time.monotonic() - t0 < 10.0:
                time.sleep(0.01)
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self, proc):
        for line in proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.proc = None

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "0.5 s of the same back-to-back steps just before and just after "
                          "the timed steps"}


def run_for(calls, seconds):
    """Runs `calls` back to back for about `seconds` (untimed load)."""
    t0 = time.monotonic()
    while time.monotonic() - t0 < seconds:
        for _ in range(20):
            for c in calls:
                c()
        torch.cuda.synchronize()


# ---------------------------------------------------------------- helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "hbm_GBs", "hbm"):
            if k in d:
                v = d[k]
                if isinstance(v, dict):
                    v = v.get("burst", v.get("value"))
                return float(v), "measured"
    except (OSError, ValueError, TypeError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """Hash of the sources the norm kernels are built from (the softmax
    translation unit is separate and not part of them)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rmsnorm_fp8_quantization_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f == "softmax.cu":
            continue
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or
    None if the kernel sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return e["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        return None


class L2Flush:
    def __init__(self, dev):
        self.buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.buf.fill_(1)


# ---------------------------------------------------------------- GPU arm

def make_step(ops, w, inp):
    """Closures for the forward call, the backward call and their buffers."""
    dev = inp["x"].device
    outs = ops.fwd_outputs(w.rows, w.hidden, inp["x"].dtype, w.norm, w.scaling, w.layout, dev)
    ws = ops.bwd_workspace(w.rows, w.hidden, inp["x"].dtype, inp["gamma"].dtype, w.norm,
                           w.zero_centered_gamma, 0, dev)
    dx = torch.empty_like(inp["x"])
    dg = torch.empty_like(inp["gamma"])
    db = torch.empty_like(inp["gamma"]) if w.norm == "layernorm" else None
    rs = torch.rand(w.rows, device=dev) + 0.5
    mu = torch.randn(w.rows, device=dev) * 0.1

    def fwd():
        ops.norm_fwd(inp["x"], inp["gamma"], inp["beta"], norm=w.norm, eps=w.eps,
                     zero_centered_gamma=w.zero_centered_gamma, scaling=w.scaling,
                     layout=w.layout, scale=inp["scale"], amax=inp["amax"], outputs=outs)

    def bwd():
        m = outs["mu"] if "fwd" in w.passes else mu
        r = outs["rsigma"] if "fwd" in w.passes else rs
        ops.norm_bwd(inp["dz"], inp["x"], m if w.norm == "layernorm" else None, r,
                     inp["gamma"], inp["dresidual"], norm=w.norm,
                     zero_centered_gamma=w.zero_centered_gamma, workspace=ws, dx=dx,
                     dgamma=dg, dbeta=db)

    return fwd, bwd, outs, (dx, dg, db)


def time_calls(calls, steps, warmup, flush=None, barrier=None):
    """Times `steps` steps of `calls` with events on the current stream
    around every call.  With `flush`, it runs before each step, outside the
    events; without, steps run back to back.  Returns (per-step ms of each
    call, total ms from the first call to the last)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for c in calls:
            c()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    per = [[] for _ in calls]
    tot = 0.0
    if flush is None:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
              for _ in range(steps)]
        for k in range(steps):
            ev[k][0].record(stream)
            for i, c in enumerate(calls):
                c()
                ev[k][i + 1].record(stream)
        torch.cuda.synchronize()
        for k in range(steps):
            for i in range(len(calls)):
                per[i].append(ev[k][i].elapsed_time(ev[k][i + 1]))
        tot = ev[0][0].elapsed_time(ev[-1][-1])
    else:
        for _ in range(steps):
            flush()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
            ev[0].record(stream)
            for i, c in enumerate(calls):
                c()
                ev[i + 1].record(stream)
            ev[-1].synchronize()
            for i in range(len(calls)):
                per[i].append(ev[i].elapsed_time(ev[i + 1]))
            tot += ev[0].elapsed_time(ev[-1])
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    return per, tot


def run_gpu(args):
    from rmsnorm_fp8_quantization_gb300 import _build
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if rank == 0:
        _build.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        dist.barrier()
        _build.build()  # no-op once rank 0 has built
    else:
        torch.cuda.set_device(0)
    from rmsnorm_fp8_quantization_gb300 import ops
    from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs

    dev = torch.device("cuda", torch.cuda.current_device())
    barrier = (lambda: dist.barrier()) if dist else None
    flush = L2Flush(dev)
    peak, peak_kind = measured_peak()

    # ---- main workload: LayerNorm fwd + bwd, steps back to back
    w = WORKLOADS[MAIN]
    inp = make_inputs(w, seed=rank, device=str(dev))
    fwd, bwd, outs, grads = make_step(ops, w, inp)
    sampler = ClockSampler(dev.index)
    sampler.start()
    run_for([fwd, bwd], 0.5)
    sampler.stop()
    per, tot = time_calls([fwd, bwd], args.steps, args.warmup, None, barrier)
    sampler.start()
    run_for([fwd, bwd], 0.5)
    sampler.stop()
    clocks = sampler.summary()
    ms_step = tot / args.steps
    if dist:
        t = torch.tensor([tot], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        tot = float(t.item())
    rows_total = w.rows * args.steps * world
    value = rows_total / (tot / 1e3)
    fwd_ms = statistics.mean(per[0])
    bwd_ms = statistics.mean(per[1])
    bb = bwd_bytes(w)
    achieved = bb / (bwd_ms / 1e3) / 1e9

    # ---- the same step with L2 flushed (512 MiB write) before every step
    fper, ftot = time_calls([fwd, bwd], args.steps, args.warmup, flush, barrier)
    flushed = {"fwd_ms": statistics.mean(fper[0]), "bwd_ms": statistics.mean(fper[1]),
               "ms_per_step": ftot / args.steps, "value": rows_total / (ftot / 1e3)}

    # ---- end to end through the C ABI with pinned host buffers
    e2e = run_e2e(ops, w, inp, args, barrier, world, dev)

    calib = copy_calibration(dev) if rank == 0 else None
    detail = {}
    if rank == 0 and not args.no_detail:
        del inp, outs, grads
        torch.cuda.empty_cache()
        detail = run_detail(ops, WORKLOADS, make_inputs, args, flush, dev, peak)
        detail.update(run_softmax_detail(ops, args, flush, dev, peak))

    result = {
        "metric": METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": tot / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": MAIN, "rows": w.rows, "hidden": w.hidden, "norm": w.norm,
                   "io_dtype": w.in_dtype, "w_dtype": w.w_dtype, "step": "fwd+bwd",
                   "l2": "not flushed: steps back to back; the inputs of a step (x, dz: "
                         "268 MB) are larger than the 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "hbm_gbs": (fwd_bytes(w) + bb) / (ms_step / 1e3) / 1e9,
        "fwd_ms": fwd_ms,
        "bwd_ms": bwd_ms,
        "l2_flushed": flushed,
        "roofline": {"bound": "hbm", "kernel": "norm_bwd (row pass + finalize)",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": bb,
                     "traffic": recorded_traffic("norm_bwd"),
                     "same_box_elementwise_gbs": calib},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "detail": detail,
    }
    if rank == 0:
        result["cpu_baseline"] = cpu_baseline(args)
        result["cpu_baseline_all_cores"] = cpu_baseline_all_cores()
        print(json.dumps(result))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def copy_calibration(dev):
    """GB/s of torch's own elementwise kernels on this GPU, timed like the
    main step (back to back, CUDA events, median): a bf16 copy (one read,
    one write stream) at the workload's size (16384 x 4096: 2 x 134 MB) and
    at 1 Gi elements (2 x 2 GiB, the size of the measured HBM peak), and a
    bf16 multiply (two reads, one write) at the workload's size.  Context for
    the roofline fraction -- what a plain streaming kernel reaches at each
    size -- not its denominator."""
    def gbs(fn, nbytes, steps):
        per, _ = time_calls([fn], steps, 5)
        return nbytes / (statistics.median(per[0]) / 1e3) / 1e9

    out = {}
    a = torch.zeros(16384, 4096, dtype=torch.bfloat16, device=dev)
    b = torch.zeros_like(a)
    o = torch.empty_like(a)
    nb = a.numel() * a.element_size()
    out["copy_workload_size"] = gbs(lambda: o.copy_(a), 2 * nb, 20)
    out["mul_workload_size"] = gbs(lambda: torch.mul(a, b, out=o), 3 * nb, 20)
    del a, b, o
    torch.cuda.empty_cache()
    try:
        a = torch.zeros(1 << 30, dtype=torch.bfloat16, device=dev)
        o = torch.empty_like(a)
        out["copy_2gib"] = gbs(lambda: o.copy_(a), 2 * a.numel() * a.element_size(), 10)
        del a, o
    except torch.cuda.OutOfMemoryError:
        out["copy_2gib"] = None
    torch.cuda.empty_cache()
    out["sizes"] = {"workload": "2 x 134,217,728 bytes (copy), 3 x (mul)",
                    "2gib": "2 x 2,147,483,648 bytes"}
    return out


def run_e2e(ops, w, inp, args, barrier, world, dev):
    """Same step through the C ABI with host buffers: every step copies x,
    dz, gamma, beta host -> device from pinned memory, runs the forward and
    the backward, and copies out, mu, rsigma, dx, dgamma, dbeta device ->
    host, all inside the timed region.

    Headline: two buffer sets and three streams (copies in, compute, copies
    out), so step i's device -> host copies overlap step i+1's host -> device
    copies and kernels, as a pipeline feeding the GPU would run.  `serial`
    is the same work on one stream, nothing overlapped."""
    keys = ("x", "dz", "gamma", "beta")
    host_in = {k: inp[k].cpu().pin_memory() for k in keys}
    sets = []
    for _ in range(2):
        dev_in = {k: torch.empty_like(inp[k]) for k in keys}
        dinp = dict(inp)
        dinp.update(dev_in)
        fwd, bwd, outs, (dx, dg, db) = make_step(ops, w, dinp)
        res = [outs["out"], outs["mu"], outs["rsigma"], dx, dg, db]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in res]
        sets.append((dev_in, fwd, bwd, res, host_out))
    h2d_bytes = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h_bytes = sum(t.numel() * t.element_size() for t in sets[0][4])
    steps = max(3, args.steps)

    def h2d(b):
        for k in keys:
            sets[b][0][k].copy_(host_in[k], non_blocking=True)

    def d2h(b):
        for h, d in zip(sets[b][4], sets[b][3]):
            h.copy_(d, non_blocking=True)

    # serial: one stream, one buffer set
    _, tot_serial = time_calls([lambda: h2d(0), sets[0][1], sets[0][2], lambda: d2h(0)], steps,
                               args.warmup, None, barrier)

    # pipelined
    cur = torch.cuda.current_stream()
    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, in_free, out_ready, out_free = ([ev(), ev()] for _ in range(4))
    for e in in_free + out_free:
        e.record(cur)

    def step(i):
        b = i % 2
        s_in.wait_event(in_free[b])
        with torch.cuda.stream(s_in):
            h2d(b)
        in_ready[b].record(s_in)
        s_c.wait_event(in_ready[b])
        s_c.wait_event(out_free[b])
        with torch.cuda.stream(s_c):
            sets[b][1]()
            sets[b][2]()
        in_free[b].record(s_c)
        out_ready[b].record(s_c)
        s_out.wait_event(out_ready[b])
        with torch.cuda.stream(s_out):
            d2h(b)
        out_free[b].record(s_out)

    def run(n):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(cur)
        s_in.wait_event(start)
        for i in range(n):
            step(i)
        cur.wait_stream(s_out)
        end.record(cur)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    run(max(args.warmup, 2))
    if barrier:
        barrier()
    torch.cuda.synchronize()
    tot = run(steps)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([tot, tot_serial], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        tot, tot_serial = float(t[0].item()), float(t[1].item())
    return {"value": w.rows * steps * world / (tot / 1e3), "unit": "rows/s",
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
            "ms_per_step": tot / steps,
            "pipeline": "2 buffer sets; host->device copies, kernels and device->host copies "
                        "on three streams (step i's copies out overlap step i+1's copies in)",
            "serial": {"value": w.rows * steps * world / (tot_serial / 1e3),
                       "ms_per_step": tot_serial / steps}}


def run_detail(ops, WORKLOADS, make_inputs, args, flush, dev, peak):
    out = {}
    steps = max(5, args.steps // 2)
    for name, w in WORKLOADS.items():
        inp = make_inputs(w, seed=0, device=str(dev))
        fwd, bwd, outs, grads = make_step(ops, w, inp)
        calls, labels = [], []
        if "fwd" in w.passes:
            calls.append(fwd)
            labels.append("fwd")
        if "bwd" in w.passes:
            calls.append(bwd)
            labels.append("bwd")
        per, _ = time_calls(calls, steps, 3)
        fper, _ = time_calls(calls, steps, 3, flush)
        d = {}
        for lab, ts, fts in zip(labels, per, fper):
            ms = statistics.median(ts)
            nb = fwd_bytes(w) if lab == "fwd" else bwd_bytes(w)
            gbs = nb / (ms / 1e3) / 1e9
            d[lab] = {"us": ms * 1e3, "us_l2_flushed": statistics.median(fts) * 1e3,
                      "rows_per_s": w.rows / (ms / 1e3), "bytes": nb,
                      "gbs": gbs, "frac_of_peak": gbs / peak,
                      "frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
                      "fits_in_l2": nb < L2_BYTES}
            if nb < L2_BYTES:
                # far below a microsecond of HBM time: the per-call latency
                # (launch and one pass of the kernel) is the figure, and the
                # workload is outside the bandwidth target
                d[lab]["launch_bound"] = True
                d[lab]["latency_us"] = ms * 1e3
        out[name] = d
        del inp, outs, grads, fwd, bwd
        torch.cuda.empty_cache()
    return out


def softmax_bytes(w, pass_):
    """Forward: the kept logits read (causal rows need none past their last
    kept key), the mask read once, y written; backward: y, dy read, dx
    written."""
    e = ESZ[w.dtype]
    n = w.batches * w.heads * w.sq * w.sk
    if pass_ == "bwd":
        return 3 * n * e
    kept = n
    if w.mask == "causal":
        kept = w.batches * w.heads * w.sq * (w.sq + 1) // 2
    elif w.mask == "causal_aligned":
        per = sum(min(max(i + 1 + w.sk - w.sq, 0), w.sk) for i in range(w.sq))
        kept = w.batches * w.heads * per
    b = kept * e + n * e
    if w.mask == "padding":
        b += w.mask_batches * w.sq * w.sk
    return b


def run_softmax_detail(ops, args, flush, dev, peak):
    from rmsnorm_fp8_quantization_gb300.workloads import SOFTMAX_WORKLOADS, make_softmax_inputs
    out = {}
    steps = max(5, args.steps // 2)
    for name, w in SOFTMAX_WORKLOADS.items():
        inp = make_softmax_inputs(w, seed=0, device=str(dev))
        y = torch.empty_like(inp["x"])
        dx = torch.empty_like(inp["x"])

        def fwd():
            ops.softmax_fwd(inp["x"], w.scale, w.mask, inp["mask"], out=y)

        def bwd():
            ops.softmax_bwd(inp["dy"], y, w.scale, out=dx)

        per, _ = time_calls([fwd, bwd], steps, 3)
        fper, _ = time_calls([fwd, bwd], steps, 3, flush)
        d = {}
        for lab, ts, fts in zip(("fwd", "bwd"), per, fper):
            ms = statistics.median(ts)
            nb = softmax_bytes(w, lab)
            gbs = nb / (ms / 1e3) / 1e9
            d[lab] = {"us": ms * 1e3, "us_l2_flushed": statistics.median(fts) * 1e3,
                      "bytes": nb, "gbs": gbs, "frac_of_peak": gbs / peak,
                      "frac_of_8tbs": gbs / NOMINAL_HBM_GBS}
        out[name] = d
        del inp, y, dx
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- CPU oracle arm

def cpu_baseline(args, min_seconds=10.0):
    """The oracle (single-threaded C++, double) on the main workload: full
    forward + backward over all 16384 rows, repeated until >= 10 s of CPU
    time; rows/s over all repetitions."""
    import numpy as np

    import oracle
    from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS[MAIN]
    inp = make_inputs(w, seed=0)
    oracle.build()
    reps = 0
    t0 = time.perf_counter()
    while True:
        z, mu, rs = oracle.norm_fwd(inp["x"], inp["gamma"], inp["beta"], 0, False, w.eps)
        oracle.round_to(z, "bf16")
        del z
        dx, dg, db = oracle.norm_bwd(inp["dz"], inp["x"], mu.astype(np.float32),
                                     rs.astype(np.float32), inp["gamma"], None, 0, False)
        oracle.round_to(dx, "bf16")
        del dx
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= 20:
            break
    return {"value": w.rows * reps / el, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": f"full {w.rows}x{w.hidden} LayerNorm fwd+bwd, {reps} repetitions, "
                      f"{el:.1f} s, single-threaded C++ (double)",
            "host": host_description()}


def cpu_baseline_all_cores(min_seconds=10.0):
    """The same oracle with the rows split over every host core: one thread
    per core runs the oracle's C functions on a contiguous slice of the rows
    (the foreign calls release the interpreter lock), and the slices'
    dgamma / dbeta are added afterwards.  Labelled apart from the
    single-threaded baseline; the oracle itself is unchanged."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS[MAIN]
    inp = make_inputs(w, seed=0)
    oracle.build()
    n = max(1, os.cpu_count() or 1)
    bounds = np.linspace(0, w.rows, n + 1).astype(int)

    def part(i):
        sl = slice(int(bounds[i]), int(bounds[i + 1]))
        z, mu, rs = oracle.norm_fwd(inp["x"][sl], inp["gamma"], inp["beta"], 0, False, w.eps)
        oracle.round_to(z, "bf16")
        del z
        dx, dg, db = oracle.norm_bwd(inp["dz"][sl], inp["x"][sl], mu.astype(np.float32),
                                     rs.astype(np.float32), inp["gamma"], None, 0, False)
        oracle.round_to(dx, "bf16")
        return dg, db

    part(0)  # loads the oracle library before the threads start
    reps = 0
    with ThreadPoolExecutor(max_workers=n) as ex:
        t0 = time.perf_counter()
        while True:
            parts = list(ex.map(part, range(n)))
            dg = sum(p[0] for p in parts)
            db = sum(p[1] for p in parts)
            oracle.round_to(dg, "f32")
            oracle.round_to(db, "f32")
            reps += 1
            el = time.perf_counter() - t0
            if el >= min_seconds or reps >= 50:
                break
    return {"value": w.rows * reps / el, "unit": "rows/s", "cores": n,
            "kind": "oracle, rows split over all host cores",
            "sample": f"full {w.rows}x{w.hidden} LayerNorm fwd+bwd, {reps} repetitions, "
                      f"{el:.1f} s, {n} threads",
            "host": host_description()}


def host_description():
    """The host the CPU legs ran on: logical CPUs and the CPU model string."""
    model = platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu": model, "arch": platform.machine()}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from rmsnorm_fp8_quantization_gb300.workloads import WORKLOADS
    w = WORKLOADS[MAIN]
    import numpy as np

    import oracle
    from rmsnorm_fp8_quantization_gb300.workloads import make_inputs
    oracle.build()
    # Each step: the oracle on a 1024-row sample of the workload (fwd + bwd).
    sample = w.with_shape(1024)
    inp = make_inputs(sample, seed=0)

    def step():
        z, mu, rs = oracle.norm_fwd(inp["x"], inp["gamma"], inp["beta"], 0, False, w.eps)
        oracle.round_to(z, "bf16")
        dx, _, _ = oracle.norm_bwd(inp["dz"], inp["x"], mu.astype(np.float32),
                                   rs.astype(np.float32), inp["gamma"], None, 0, False)
        oracle.round_to(dx, "bf16")

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    v = sample.rows * args.steps / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "rows/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": MAIN, "rows": w.rows, "hidden": w.hidden,
                   "sample_rows_per_step": sample.rows},
        "cpu_baseline": {"value": v, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{sample.rows} rows of {MAIN} per step (fwd+bwd)",
                         "host": host_description()},
        "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_only(args):
    """A short run of one workload's passes (the command profiled by ncu).
    Softmax workloads: --rows overrides the batch count."""
    from rmsnorm_fp8_quantization_gb300 import _build
    _build.build()
    from rmsnorm_fp8_quantization_gb300 import ops
    from rmsnorm_fp8_quantization_gb300.workloads import (SOFTMAX_WORKLOADS, WORKLOADS,
                                                          make_inputs, make_softmax_inputs)
    torch.cuda.set_device(0)
    if args.only in SOFTMAX_WORKLOADS:
        w = SOFTMAX_WORKLOADS[args.only]
        if args.rows:
            w = w.with_shape(args.rows, w.heads, w.sq, w.sk)
        inp = make_softmax_inputs(w, seed=0, device="cuda")
        y = torch.empty_like(inp["x"])
        dx = torch.empty_like(inp["x"])
        calls = [lambda: ops.softmax_fwd(inp["x"], w.scale, w.mask, inp["mask"], out=y),
                 lambda: ops.softmax_bwd(inp["dy"], y, w.scale, out=dx)]
        per, _ = time_calls(calls, args.steps, args.warmup)
        print(json.dumps({"workload": w.name, "batches": w.batches,
                          "us": [statistics.median(t) * 1e3 for t in per]}))
        return
    w = WORKLOADS[args.only]
    if args.rows:
        w = w.with_shape(args.rows)
    inp = make_inputs(w, seed=0, device="cuda")
    fwd, bwd, _, _ = make_step(ops, w, inp)
    calls = [c for p, c in (("fwd", fwd), ("bwd", bwd)) if p in w.passes]
    per, _ = time_calls(calls, args.steps, args.warmup)
    print(json.dumps({"workload": w.name, "rows": w.rows, "hidden": w.hidden,
                      "us": [statistics.median(t) * 1e3 for t in per]}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gbnorm", choices=["gbnorm", "reference"])
    ap.add_argument("--no-detail", action="store_true")
    ap.add_argument("--only", default=None, help="time one workload's passes only")
    ap.add_argument("--rows", type=int, default=0, help="with --only: override the row count")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
