"""Attention-backward benchmark on GB300.

One step = one whole backward pass of the causal GQA workload
(B=2, H=32, H_kv=8, N=4096, d=128, tau=1/sqrt(d)) through the C ABI:
attn_bwd_preprocess -> attn_bwd -> attn_bwd_finalize, inputs resident in HBM.
The metric is backward TFLOPS (5 GEMMs of 2 N^2 d per head, halved for
causal) and its fraction of the measured dense bf16 peak; ms per call is
reported alongside. The per-step working set (about 450 MiB) is larger than
L2, so no explicit flush is done between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on the host
  python bench.py --kernel-only attn_fwd --workload causal_gqa --steps 3 --warmup 3
      # W + K launches of one kernel alone (for ncu captures); prints its
      # median time

Under torchrun every rank runs its own copy of the workload on its own GPU
(weak scaling, no data-path collective); rank 0 prints one JSON line with the
max-over-ranks time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import torch  # noqa: E402

METRIC = "attention-backward TFLOPS and % of GB300 bf16 tensor peak; ms per bwd call"
UNIT = "TFLOPS"
PEAK_FALLBACK = {"bf16_tflops": 1890.0, "hbm_gbs": 6800.0, "source": "fallback"}
KERNEL_SOURCES = ["flashattention_attention_backward_gb300/csrc/attn_bwd.cu",
                  "flashattention_attention_backward_gb300/csrc/sm103_ptx.cuh"]
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "attn_bwd_causal_gqa_traffic.json")


# ---------------------------------------------------------------- helpers
def dist_env():
    """(rank, local_rank, world_size) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world, device=None):
    """Max of a float over all ranks (plain host value when world == 1)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base, rank):
    """Each rank draws its own synthetic batch of the same shape."""
    return base + 7919 * rank


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(PEAK_FALLBACK)


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu counters of the timed
    kernel, if they were taken on the current kernel source (else None)."""
    try:
        with open(TRAFFIC_PROFILE) as f:
            rec = json.load(f)
        sha, nbytes = rec["kernel_source_sha256"], float(rec["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None
    return nbytes if sha == kernel_source_hash() else None


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- our arm
def hbm_bytes_preprocess(B, H, N, d):
    """Algorithmic DRAM bytes of attn_bwd_preprocess: O and dO read (bf16),
    D written (fp32), dQaccum zeroed (fp32)."""
    return B * H * N * (2 * d * 2 + 4 + d * 4)


def hbm_bytes_finalize(B, H, N, d):
    """Algorithmic DRAM bytes of attn_bwd_finalize: dQaccum read (fp32), dQ
    written (bf16)."""
    return B * H * N * d * (4 + 2)


def step_kernels(w, pre_ms, bwd_ms, fin_ms, peaks):
    """Mean time per launch of each kernel of the step (CUDA events between
    the launches of up to 200 steps run right after the timed region); the
    two HBM-bound kernels against the measured copy bandwidth."""
    mean = lambda xs: sum(xs) / len(xs)  # noqa: E731
    out = {"attn_bwd": {"ms": mean(bwd_ms), "bound": "tensor"}}
    for name, xs, nbytes in (
            ("attn_bwd_preprocess", pre_ms, hbm_bytes_preprocess(w.B, w.H, w.N, w.d)),
            ("attn_bwd_finalize", fin_ms, hbm_bytes_finalize(w.B, w.H, w.N, w.d))):
        ms = mean(xs)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "bound": "hbm", "bytes": nbytes, "GB/s": gbs,
                     "peak_GB/s": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"]}
    return out


def run_ours(args, w):
    import flashattention_attention_backward_gb300 as attn
    from flashattention_attention_backward_gb300 import runner
    from flashattention_attention_backward_gb300.inputs import make_inputs

    rank, local_rank, world = dist_env()
    dist_init(world, "nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    attn.library()

    w = w.with_(seed_base=rank_seed(w.seed_base, rank))
    x = make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap)
    bufs = runner.BackwardBuffers(q, k)
    stream = torch.cuda.current_stream(dev)
    B, H, H_kv, N, d = w.B, w.H, w.H_kv, w.N, w.d

    def step(before_pre=None, before_bwd=None, after_bwd=None, after_fin=None):
        # optional CUDA events recorded between the three launches
        def mark(e):
            if e is not None:
                e.record(stream)

        mark(before_pre)
        attn.check(attn.attn_bwd_preprocess(o, do, bufs.dpsum, bufs.dq_accum, B, H, N, d, stream))
        mark(before_bwd)
        attn.check(attn.attn_bwd(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, B, H, H_kv,
                                 N, d, w.scale, w.causal, w.softcap, bufs.dpsum, stream))
        mark(after_bwd)
        attn.check(attn.attn_bwd_finalize(bufs.dq_accum, bufs.dq, w.scale, B, H, N, d, stream))
        mark(after_fin)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    rc, status = attn.attn_device_status(clear=True, stream=stream)
    if rc != 0 or status != 0:
        raise RuntimeError("device status %d after warm-up" % status)

    kev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2))
           for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.start()
        time.sleep(0.25)
    t0.record(stream)
    for i in range(args.steps):
        step(before_bwd=kev[i][0], after_bwd=kev[i][1])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clock_info = clocks.stop() if clocks else None
    ms_total = t0.elapsed_time(t1)
    bwd_ms = [e[0].elapsed_time(e[1]) for e in kev]
    # each launch of the step on its own: the same steps again, with events
    # between all three launches (kept out of the headline loop, whose only
    # events are the two around attn_bwd)
    kev4 = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4))
            for _ in range(min(args.steps, 200))]
    for e in kev4:
        step(*e)
    torch.cuda.synchronize(dev)
    pre_ms = [e[0].elapsed_time(e[1]) for e in kev4]
    bwd4_ms = [e[1].elapsed_time(e[2]) for e in kev4]
    fin_ms = [e[2].elapsed_time(e[3]) for e in kev4]
    rc, status = attn.attn_device_status(clear=True, stream=stream)
    if rc != 0 or status != 0:
        raise RuntimeError("device status %d after the timed region" % status)
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / args.steps
    flops = w.flops()
    value = world * flops * args.steps / (ms_total * 1e-3) / 1e12

    # end to end: pinned host inputs -> device, backward, results -> host,
    # every step. Steps are streamed as a user would: two device copies of
    # the inputs and outputs, so that the host->device copy of step i+1 and
    # the device->host copy of step i-1 run on their own streams while step i
    # computes. Events order each buffer's reuse.
    pin = {n: x[n].pin_memory() for n in ("q", "k", "v", "do")}
    pin["o"], pin["lse"] = o.cpu().pin_memory(), lse.cpu().pin_memory()
    h_out = {n: torch.empty_like(t, device="cpu").pin_memory()
             for n, t in (("dq", bufs.dq), ("dk", bufs.dk), ("dv", bufs.dv))}
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    e2e_steps = max(4, min(args.steps, 20))
    dins = [{"q": q, "k": k, "v": v, "do": do, "o": o, "lse": lse},
            {n: torch.empty_like(t) for n, t in (("q", q), ("k", k), ("v", v), ("do", do),
                                                   ("o", o), ("lse", lse))}]
    dbufs = [bufs, runner.BackwardBuffers(q, k)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run_e2e(n_steps):
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_ready, computed, out_done = {}, {}, {}
        for i in range(n_steps):
            j = i & 1
            a = dins[j]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(computed[i - 2])  # step i-2 has read these inputs
                for n in pin:
                    a[n].copy_(pin[n], non_blocking=True)
                in_ready[i] = ev()
                in_ready[i].record(s_in)
            stream.wait_event(in_ready[i])
            if i >= 2:
                stream.wait_event(out_done[i - 2])  # step i-2's results are on the host
            bb = dbufs[j]
            attn.check(attn.attn_bwd_preprocess(a["o"], a["do"], bb.dpsum, bb.dq_accum, B, H, N, d,
                                                stream))
            attn.check(attn.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"],
                                     bb.dq_accum, bb.dk, bb.dv, B, H, H_kv, N, d, w.scale,
                                     w.causal, w.softcap, bb.dpsum, stream))
            attn.check(attn.attn_bwd_finalize(bb.dq_accum, bb.dq, w.scale, B, H, N, d, stream))
            computed[i] = ev()
            computed[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[i])
                h_out["dq"].copy_(bb.dq, non_blocking=True)
                h_out["dk"].copy_(bb.dk, non_blocking=True)
                h_out["dv"].copy_(bb.dv, non_blocking=True)
                out_done[i] = ev()
                out_done[i].record(s_out)

    run_e2e(2)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_in.wait_stream(stream)
    run_e2e(e2e_steps)
    s_out.wait_stream(s_in)
    s_out.wait_stream(stream)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(world)
    rc, status = attn.attn_device_status(clear=True, stream=stream)
    if rc != 0 or status != 0:
        raise RuntimeError("device status %d after the end-to-end steps" % status)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / e2e_steps
    e2e_value = world * flops / (e2e_ms * 1e-3) / 1e12

    if rank != 0:
        return None
    peaks = measured_peaks()
    bwd_avg = sum(bwd_ms) / len(bwd_ms)
    achieved = flops / (bwd_avg * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded i.i.d. normal bf16 Q/K/V/dO; O and LSE from attn_fwd)",
        "config": {
            "workload": "%s B=%d H=%d H_kv=%d N=%d d=%d %s%s" % (
                w.name, w.B, w.H, w.H_kv, w.N, w.d, "causal" if w.causal else "non-causal",
                (" softcap=%g" % w.softcap) if w.softcap > 0 else ""),
            "B": w.B, "H": w.H, "H_kv": w.H_kv, "N": w.N, "d": w.d, "causal": w.causal,
            "softcap": w.softcap, "scale": w.scale,
            "step": "attn_bwd_preprocess + attn_bwd + attn_bwd_finalize",
            "flops_per_step_per_gpu": flops,
            "l2": "inputs larger than L2 (about %d MiB touched per step), no flush" % (
                (4 * B * H * N * d * 2 + 4 * B * H_kv * N * d * 2 + B * H * N * d * 4
                 + 2 * B * H * N * 4) >> 20),
        },
        "bwd_ms": bwd_avg,
        "bwd_tflops": achieved,
        "pct_of_bf16_peak": 100.0 * achieved / peaks["bf16_tflops"],
        "roofline": {
            "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
            "traffic": profiled_traffic(),
            "kernel": "attn_bwd_kernel<128, causal>",
            "peak_source": "%s burst dense bf16 (MEASURED_PEAKS.json)" % peaks["source"],
        },
        "kernels": step_kernels(w, pre_ms, bwd4_ms, fin_ms, peaks),
        "clocks": clock_info,
        "gpu_launches": 3 * args.steps,
        "e2e": {"value": e2e_value, "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "streaming": "two device buffer sets; step i+1's host->device copy and step "
                             "i-1's device->host copy overlap step i's kernels"},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if world == 1 and not args.no_all_configs:
        del q, k, v, do, o, lse, bufs, pin, h_out, dins, dbufs
        torch.cuda.empty_cache()
        line["all_configs"] = all_configs(dev, peaks["bf16_tflops"])
    return line


def all_configs(dev, peak, iters=20, warmup=3):
    """attn_bwd alone on each named workload (CUDA events around each launch,
    median of `iters`): ms, TFLOP/s and the fraction of the bf16 peak; the
    same for the tensor-core forward attn_fwd."""
    import flashattention_attention_backward_gb300 as attn
    from flashattention_attention_backward_gb300 import runner
    from flashattention_attention_backward_gb300.inputs import WORKLOADS, make_inputs

    out = {}
    stream = torch.cuda.current_stream(dev)
    for name, w in WORKLOADS.items():
        x = make_inputs(w)
        q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
        o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap)
        bufs = runner.BackwardBuffers(q, k)
        times = []
        for i in range(warmup + iters):
            attn.check(attn.attn_bwd_preprocess(o, do, bufs.dpsum, bufs.dq_accum, w.B, w.H, w.N,
                                                w.d, stream))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            attn.check(attn.attn_bwd(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, w.B,
                                     w.H, w.H_kv, w.N, w.d, w.scale, w.causal, w.softcap,
                                     bufs.dpsum, stream))
            e1.record(stream)
            if i >= warmup:
                times.append((e0, e1))
        torch.cuda.synchronize(dev)
        rc, status = attn.attn_device_status(clear=True, stream=stream)
        if rc != 0 or status != 0:
            raise RuntimeError("device status %d on %s" % (status, name))
        ms = sorted(a.elapsed_time(b) for a, b in times)[len(times) // 2]
        tf = w.flops() / (ms * 1e-3) / 1e12
        # the tensor-core forward on the same inputs (2 GEMMs of 2 N^2 d per
        # head, halved for causal)
        fts = []
        for i in range(warmup + iters):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            attn.check(attn.attn_fwd(q, k, v, o, lse, w.B, w.H, w.H_kv, w.N, w.d, w.scale,
                                     w.causal, w.softcap, stream))
            e1.record(stream)
            if i >= warmup:
                fts.append((e0, e1))
        torch.cuda.synchronize(dev)
        fms = sorted(a.elapsed_time(b) for a, b in fts)[len(fts) // 2]
        ftf = w.flops() * 2 / 5 / (fms * 1e-3) / 1e12
        out[name] = {"B": w.B, "H": w.H, "H_kv": w.H_kv, "N": w.N, "d": w.d,
                     "causal": w.causal, "softcap": w.softcap, "bwd_ms": ms,
                     "tflops": tf, "frac_of_peak": tf / peak,
                     "fwd_ms": fms, "fwd_tflops": ftf, "fwd_frac_of_peak": ftf / peak}
        del x, q, k, v, do, o, lse, bufs
        torch.cuda.empty_cache()
    out["causal_gqa_window1024"] = local_window_timing(dev, peak, iters, warmup)
    out["causal_gqa_variants"] = variant_timing(dev, peak, iters, warmup)
    out["causal_gqa_d256"] = d256_timing(dev, peak, iters, warmup)
    out["causal_gqa_d256_variants"] = variant_timing(dev, peak, iters, warmup, w=d256_workload())
    return out


def d256_workload():
    from flashattention_attention_backward_gb300.inputs import Workload
    return Workload("causal_gqa_d256", 2, 16, 4, 4096, 256, True, seed_base=20261202 + 6000)


def d256_timing(dev, peak, iters, warmup):
    """attn_bwd with head dimension 256 (its own kernel) on a causal GQA shape
    of the same token count as the causal GQA workload: B=2, H=16, H_kv=4,
    N=4096, d=256; FLOPs as for the plain backward (5 GEMMs of 2 N^2 d per
    head, halved for causal)."""
    import flashattention_attention_backward_gb300 as attn
    from flashattention_attention_backward_gb300 import runner
    from flashattention_attention_backward_gb300.inputs import make_inputs

    w = d256_workload()
    stream = torch.cuda.current_stream(dev)
    x = make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, True)
    torch.cuda.synchronize(dev)
    rc, status = attn.attn_device_status(clear=True, stream=stream)
    if rc != 0 or status != 0:
        raise RuntimeError("device status %d after the d = 256 forward" % status)
    bufs = runner.BackwardBuffers(q, k)
    ts = []
    for i in range(warmup + iters):
        attn.check(attn.attn_bwd_preprocess(o, do, bufs.dpsum, bufs.dq_accum, w.B, w.H, w.N, w.d,
                                            stream))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        attn.check(attn.attn_bwd(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, w.B, w.H,
                                 w.H_kv, w.N, w.d, w.scale, True, 0.0, bufs.dpsum, stream))
        e1.record(stream)
        if i >= warmup:
            ts.append((e0, e1))
    torch.cuda.synchronize(dev)
    rc, status = attn.attn_device_status(clear=True, stream=stream)
    if rc != 0 or status != 0:
        raise RuntimeError("device status %d on the d = 256 timing" % status)
    ms = sorted(a.elapsed_time(b) for a, b in ts)[len(ts) // 2]
    tf = w.flops() / (ms * 1e-3) / 1e12
    # the tensor-core forward at d = 256 (one query tile per CTA): 2 GEMMs of
    # 2 N^2 d per head, halved for causal
    fts = []
    for i in range(warmup + iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        attn.check(attn.attn_fwd(q, k, v, o, lse, w.B, w.H, w.H_kv, w.N, w.d, w.scale, True, 0.0,
                                 stream))
        e1.record(stream)
        if i >= warmup:
            fts.append((e0, e1))
    torch.cuda.synchronize(dev)
    rc, status = attn.attn_device_status(clear=True, stream=stream)
    if rc != 0 or status != 0:
        raise RuntimeError("device status %d on the d = 256 forward timing" % status)
    fms = sorted(a.elapsed_time(b) for a, b in fts)[len(fts) // 2]
    ftf = w.flops() * 2 / 5 / (fms * 1e-3) / 1e12
    del x, q, k, v, do, o, lse, bufs
    torch.cuda.empty_cache()
    return {"B": w.B, "H": w.H, "H_kv": w.H_kv, "N": w.N, "d": w.d, "causal": True,
            "bwd_ms": ms, "tflops": tf, "frac_of_peak": tf / peak,
            "fwd_ms": fms, "fwd_tflops": ftf, "fwd_frac_of_peak": ftf / peak}


def variant_timing(dev, peak, iters, warmup, p_drop=0.1, seed=1234, w=None):
    """The deterministic-dQ step (preprocess + attn_bwd_deterministic +
    attn_bwd_finalize_partials), attn_bwd_dropout and attn_fwd_dropout on the
    causal GQA workload (or `w`, a causal workload), against the plain step
    and attn_fwd; FLOPs as for the plain kernels."""
    import flashattention_attention_backward_gb300 as attn
    from flashattention_attention_backward_gb300 import runner
    from flashattention_attention_backward_gb300.inputs import WORKLOADS, make_inputs

    if w is None:
        w = WORKLOADS["causal_gqa"]
    B, H, H_kv, N, d = w.B, w.H, w.H_kv, w.N, w.d
    stream = torch.cuda.current_stream(dev)
    x = make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, True)
    bufs = runner.BackwardBuffers(q, k)
    nbytes = attn.attn_bwd_dq_partials_bytes(B, H, N, d, True)
    attn.check(int(nbytes) if nbytes < 0 else 0)
    partials = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)

    def timed(fn):
        ts = []
        for i in range(warmup + iters):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= warmup:
                ts.append((e0, e1))
        torch.cuda.synchronize(dev)
        rc, status = attn.attn_device_status(clear=True, stream=stream)
        if rc != 0 or status != 0:
            raise RuntimeError("device status %d on the variant timing" % status)
        return sorted(a.elapsed_time(b) for a, b in ts)[len(ts) // 2]

    def plain_step():
        attn.check(attn.attn_bwd_preprocess(o, do, bufs.dpsum, bufs.dq_accum, B, H, N, d, stream))
        attn.check(attn.attn_bwd(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, B, H,
                                 H_kv, N, d, w.scale, True, 0.0, bufs.dpsum, stream))
        attn.check(attn.attn_bwd_finalize(bufs.dq_accum, bufs.dq, w.scale, B, H, N, d, stream))

    def det_step():
        attn.check(attn.attn_bwd_preprocess(o, do, bufs.dpsum, None, B, H, N, d, stream))
        attn.check(attn.attn_bwd_deterministic(q, k, v, o, do, lse, partials, bufs.dk, bufs.dv,
                                               B, H, H_kv, N, d, w.scale, True, 0.0, bufs.dpsum,
                                               stream))
        attn.check(attn.attn_bwd_finalize_partials(partials, bufs.dq, w.scale, B, H, N, d, True,
                                                   stream))

    def drop_bwd():
        attn.check(attn.attn_bwd_dropout(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, B,
                                         H, H_kv, N, d, w.scale, True, 0.0, bufs.dpsum, p_drop,
                                         seed, stream))

    res = {"plain_step_ms": timed(plain_step), "deterministic_step_ms": timed(det_step),
           "dq_partials_bytes": int(nbytes)}
    attn.check(attn.attn_bwd_preprocess(o, do, bufs.dpsum, bufs.dq_accum, B, H, N, d, stream))
    res["dropout_bwd_ms"] = timed(drop_bwd)
    res["dropout_p"] = p_drop
    res["dropout_fwd_ms"] = timed(lambda: attn.check(attn.attn_fwd_dropout(
        q, k, v, o, lse, B, H, H_kv, N, d, w.scale, True, 0.0, p_drop, seed, stream)))
    res["plain_fwd_ms"] = timed(lambda: attn.check(attn.attn_fwd(
        q, k, v, o, lse, B, H, H_kv, N, d, w.scale, True, 0.0, stream)))
    f = w.flops()
    for key in ("plain_step_ms", "deterministic_step_ms", "dropout_bwd_ms"):
        res[key.replace("_ms", "_tflops")] = f / (res[key] * 1e-3) / 1e12
    res["dropout_bwd_frac_of_peak"] = res["dropout_bwd_tflops"] / peak
    for key in ("dropout_fwd_ms", "plain_fwd_ms"):
        res[key.replace("_ms", "_tflops")] = f * 2 / 5 / (res[key] * 1e-3) / 1e12
    del x, q, k, v, do, o, lse, bufs, partials
    torch.cuda.empty_cache()
    return res


def visible_pairs(N, causal, left, right):
    """(query, key) pairs of one head inside the band i - left <= j <= i + right
    (negative = unbounded) and, if causal, j <= i."""
    total = 0
    for i in range(N):
        lo = 0 if left < 0 else max(0, i - left)
        hi = N - 1 if right < 0 else min(N - 1, i + right)
        if causal:
            hi = min(hi, i)
        total += max(0, hi - lo + 1)
    return total


def local_window_timing(dev, peak, iters, warmup, left=1023):
    """attn_bwd_local and attn_fwd_local on the causal GQA shape under a
    causal sliding window of left + 1 keys; FLOPs counted over the visible
    pairs (5 GEMMs of 2 d per pair backward, 2 forward)."""
    import flashattention_attention_backward_gb300 as attn
    from flashattention_attention_backward_gb300 import runner
    from flashattention_attention_backward_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS["causal_gqa"]
    win = (left, -1)
    stream = torch.cuda.current_stream(dev)
    x = make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = runner.forward(q, k, v, w.scale, True, window=win)
    bufs = runner.BackwardBuffers(q, k)
    bt, ft = [], []
    for i in range(warmup + iters):
        attn.check(attn.attn_bwd_preprocess(o, do, bufs.dpsum, bufs.dq_accum, w.B, w.H, w.N, w.d,
                                            stream))
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        attn.check(attn.attn_bwd_local(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, w.B,
                                       w.H, w.H_kv, w.N, w.d, w.scale, True, 0.0, bufs.dpsum,
                                       win[0], win[1], stream))
        e[1].record(stream)
        e[2].record(stream)
        attn.check(attn.attn_fwd_local(q, k, v, o, lse, w.B, w.H, w.H_kv, w.N, w.d, w.scale,
                                       True, 0.0, win[0], win[1], stream))
        e[3].record(stream)
        if i >= warmup:
            bt.append((e[0], e[1]))
            ft.append((e[2], e[3]))
    torch.cuda.synchronize(dev)
    rc, status = attn.attn_device_status(clear=True, stream=stream)
    if rc != 0 or status != 0:
        raise RuntimeError("device status %d on the local-window timing" % status)
    pairs = w.B * w.H * visible_pairs(w.N, True, left, -1)
    bms = sorted(a.elapsed_time(b) for a, b in bt)[len(bt) // 2]
    fms = sorted(a.elapsed_time(b) for a, b in ft)[len(ft) // 2]
    btf = 10.0 * w.d * pairs / (bms * 1e-3) / 1e12
    ftf = 4.0 * w.d * pairs / (fms * 1e-3) / 1e12
    del x, q, k, v, do, o, lse, bufs
    torch.cuda.empty_cache()
    return {"B": w.B, "H": w.H, "H_kv": w.H_kv, "N": w.N, "d": w.d, "causal": True,
            "window": list(win), "visible_pairs": pairs, "bwd_ms": bms, "tflops": btf,
            "frac_of_peak": btf / peak, "fwd_ms": fms, "fwd_tflops": ftf,
            "fwd_frac_of_peak": ftf / peak}


# ---------------------------------------------------------------- the oracle on the host
def _oracle_unit(x, w, b, h, M):
    """fp64 oracle backward of query head h (batch b) on its first M rows/keys."""
    from oracle import attention_backward

    g = h // w.G
    q = x["q"][b:b + 1, h:h + 1, :M].double().numpy()
    do = x["do"][b:b + 1, h:h + 1, :M].double().numpy()
    k = x["k"][b:b + 1, g:g + 1, :M].double().numpy()
    v = x["v"][b:b + 1, g:g + 1, :M].double().numpy()
    attention_backward(q, k, v, do, w.scale, w.causal, w.softcap)
    f = 5.0 * 2.0 * M * M * w.d
    return f / 2.0 if w.causal else f


def cpu_baseline(w, budget_s=15.0):
    """The oracle timed on the host cores on a bounded sample: whole query
    heads of one batch of the workload (full N), as many as fit in
    `budget_s` seconds."""
    from flashattention_attention_backward_gb300.inputs import make_inputs

    wb = w.with_(B=1)
    x = make_inputs(wb)
    flops, heads = 0.0, 0
    t0 = time.perf_counter()
    while heads < wb.H and (heads == 0 or time.perf_counter() - t0 < budget_s):
        flops += _oracle_unit(x, wb, 0, heads, w.N)
        heads += 1
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": _CORES, "kind": "oracle",
            "sample": "%d query head(s) x N=%d of batch 0 of %s, fp64 numpy, %.1f s"
                      % (heads, w.N, w.name, dt)}


def run_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return None
    from flashattention_attention_backward_gb300.inputs import make_inputs

    x = make_inputs(w.with_(B=1, H=w.G, H_kv=1))
    wx = w.with_(B=1, H=w.G, H_kv=1)
    # size the per-step sample so warm-up + timed steps stay within the budget
    t0 = time.perf_counter()
    _oracle_unit(x, wx, 0, 0, 512)
    t512 = max(time.perf_counter() - t0, 1e-3)
    n_units = args.steps + args.warmup
    M = w.N
    while M > 256 and n_units * t512 * (M / 512.0) ** 2 > args.ref_budget:
        M //= 2
    for i in range(args.warmup):
        _oracle_unit(x, wx, 0, i % w.G, M)
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops += _oracle_unit(x, wx, 0, i % w.G, M)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = ("per step: one query head of %s, first %d queries and keys (%s), fp64 numpy"
              % (w.name, M, "causal" if w.causal else "non-causal"))
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": "%s B=%d H=%d H_kv=%d N=%d d=%d %s" % (
            w.name, w.B, w.H, w.H_kv, w.N, w.d, "causal" if w.causal else "non-causal"),
            "sample_rows": M},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _CORES, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def kernel_only(args, w):
    """W + K launches of one kernel of the path on workload `w`, nothing else
    between them (inputs prepared first); returns a short JSON-able record."""
    import flashattention_attention_backward_gb300 as attn
    from flashattention_attention_backward_gb300 import runner
    from flashattention_attention_backward_gb300.inputs import make_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    if args.kernel_only in ("attn_bwd_d256", "attn_fwd_d256"):  # the d = 256 shape of all_configs
        w = d256_workload()
    x = make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    win = (args.window_left, -1) if args.kernel_only.endswith("_local") else None
    o, lse = runner.forward(q, k, v, w.scale, w.causal, w.softcap, window=win)
    bufs = runner.BackwardBuffers(q, k)
    B, H, H_kv, N, d = w.B, w.H, w.H_kv, w.N, w.d
    attn.check(attn.attn_bwd_preprocess(o, do, bufs.dpsum, bufs.dq_accum, B, H, N, d, stream))

    def launch():
        name = args.kernel_only
        if name in ("attn_fwd", "attn_fwd_d256"):
            return attn.attn_fwd(q, k, v, o, lse, B, H, H_kv, N, d, w.scale, w.causal, w.softcap,
                                 stream)
        if name == "attn_fwd_local":
            return attn.attn_fwd_local(q, k, v, o, lse, B, H, H_kv, N, d, w.scale, w.causal,
                                       w.softcap, win[0], win[1], stream)
        if name == "attn_fwd_dropout":
            return attn.attn_fwd_dropout(q, k, v, o, lse, B, H, H_kv, N, d, w.scale, w.causal,
                                         w.softcap, args.p_drop, 1234, stream)
        if name == "attn_bwd_dropout":
            return attn.attn_bwd_dropout(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, B,
                                         H, H_kv, N, d, w.scale, w.causal, w.softcap, bufs.dpsum,
                                         args.p_drop, 1234, stream)
        if name == "attn_bwd_local":
            return attn.attn_bwd_local(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, B, H,
                                       H_kv, N, d, w.scale, w.causal, w.softcap, bufs.dpsum,
                                       win[0], win[1], stream)
        return attn.attn_bwd(q, k, v, o, do, lse, bufs.dq_accum, bufs.dk, bufs.dv, B, H, H_kv, N,
                             d, w.scale, w.causal, w.softcap, bufs.dpsum, stream)

    times = []
    for i in range(args.warmup + args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        attn.check(launch())
        e1.record(stream)
        if i >= args.warmup:
            times.append((e0, e1))
    torch.cuda.synchronize(dev)
    rc, status = attn.attn_device_status(clear=True, stream=stream)
    if rc != 0 or status != 0:
        raise RuntimeError("device status %d" % status)
    ms = sorted(a.elapsed_time(b) for a, b in times)[len(times) // 2]
    return {"kernel": args.kernel_only, "workload": w.name, "window": win,
            "launches": args.warmup + args.steps, "median_ms": ms}


def main(argv=None):
    from flashattention_attention_backward_gb300.inputs import WORKLOADS

    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="causal_gqa", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-all-configs", action="store_true",
                    help="skip the per-workload attn_bwd timings added to the line")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=120.0)
    ap.add_argument("--kernel-only", default=None,
                    choices=["attn_bwd", "attn_fwd", "attn_bwd_local", "attn_fwd_local",
                             "attn_bwd_d256", "attn_fwd_d256", "attn_fwd_dropout",
                             "attn_bwd_dropout"],
                    help="launch only this kernel W + K times (profiling); no bench line")
    ap.add_argument("--window-left", type=int, default=1023,
                    help="left bound of the causal sliding window of the *_local kernels")
    ap.add_argument("--p-drop", type=float, default=0.1,
                    help="drop probability of the *_dropout kernels")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = WORKLOADS[args.workload]
    if args.kernel_only:
        print(json.dumps(kernel_only(args, w)), flush=True)
        return
    line = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if line is not None:
        print(json.dumps(line), flush=True)
    _, _, world = dist_env()
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
