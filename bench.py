"""Benchmark of the fused causal attention forwards on GB300.

``python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
[--workload NAME] [--no-secondary]`` prints ONE JSON line.  ``--op`` times one
widened op on its own instead (backward, backward-deterministic, diff,
diff-backward on a TRA workload; fsa on an NSA workload), for per-kernel
measurements and ncu captures.

A step is one pass of the whole threshold-rectified-attention (TRA) path --
tau table, Q K^T, causal mask, threshold and power, W V, store -- fused in one
kernel launch, over one batch of synthetic input of the workload.  Inputs are resident in HBM when the
timed region starts; the inputs plus output (256 MB) are larger than the
129 MB L2, so no flush is done between steps of the headline workload.  The
default workload is the T=8192 one: bf16 B=2 H=32 T=8192 D=64, beta=2 and the
general power p=1.5 on the exp/log path.  The secondary workloads (the
B=4 H=16 T=4096 D=128 p=2 TRA and the NSA selection workloads) are measured
in the same run and reported under ``secondary``.

Multi-GPU (torchrun): the problem is sharded by batch with no collective on
the data path (the work is independent per (batch, head)): with N ranks the
global problem has N times the workload's batches, and rank r draws and
processes its own slice of them (seed r; rank 0's slice is the single-GPU
input), so the work per GPU is fixed ("scaling": "weak"); ``value`` is the
total FLOPs of all ranks over the max elapsed time.
"""

from __future__ import annotations

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

METRIC = "causal fwd TFLOP/s & % of dense BF16 tensor peak (threshold attn; NSA select)"
DEFAULT_WORKLOAD = "tra_bf16_B2_H32_T8192_D64"
SECONDARY = ["tra_bf16_B4_H16_T4096_D128", "nsa_bf16_B2_Hq32_Hkv2_T8192_D128", "nsa_bf16_B1_Hq64_Hkv4_T32768_D128",
             "nsa_bf16_B2_Hq32_Hkv2_T8192_D32_bs32"]
# Shape of the widened rows' lines (training backward, differential forward).
WIDENED_WORKLOAD = "tra_bf16_B4_H16_T4096_D128"
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = {
    "tra": "block_sparse_attention_tra_gb300/csrc/tra_bf16.cu",
    "tra_f32": "block_sparse_attention_tra_gb300/csrc/tra_f32.cu",
    "nsa": "block_sparse_attention_tra_gb300/csrc/nsa_select.cu",
    "nsa_general": "block_sparse_attention_tra_gb300/csrc/nsa_general.cu",
    "fsa": "block_sparse_attention_tra_gb300/csrc/nsa_fsa.cu",
}


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def source_hash(kind: str) -> str:
    with open(os.path.join(ROOT, KERNEL_SOURCES[kind]), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kind: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        tab = json.load(f)
    ent = tab.get(workload)
    if not ent or ent.get("source_sha") != source_hash(kind):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()  # the first sample takes a moment; start the load after it
            while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.02)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def clocks_rejected(c: dict) -> bool:
    """A timed region is not a valid measurement when the GPU throttled for
    hardware or thermal reasons, or when its SM clock sat well below the
    maximum with no reason given (a clock left locked by an earlier user).
    sw_power_cap is normal under a dense tensor load and is kept."""
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    reasons = set(c.get("reasons") or [])
    if bad & reasons:
        return True
    mhz, mx = c.get("sm_mhz"), c.get("sm_max_mhz")
    return bool(mhz and mx and mhz < 0.8 * mx and not (reasons - {"unsampled"}))


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity for a single process)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# --------------------------------------------------------------- our kernels

def make_inputs(name, device, rank=0):
    """The workload and this rank's slice of the batch-sharded problem (host
    tensors and device copies)."""
    from block_sparse_attention_tra_gb300 import workloads

    w = workloads.TRA_WORKLOADS.get(name) or workloads.NSA_WORKLOADS[name]
    tensors = workloads.workload_inputs(w, seed=workloads.shard_seed(rank))
    return w, tensors, [t.to(device) for t in tensors]


def launcher(w, dev_tensors, out, lse=None, stream=None):
    from block_sparse_attention_tra_gb300 import bsa, workloads

    if isinstance(w, workloads.TraWorkload):
        q, k, v = dev_tensors
        return lambda: bsa.tra_forward(q, k, v, w.beta, w.p, out=out, stream=stream)
    q, k, v, idx = dev_tensors
    return lambda: bsa.nsa_select_forward(q, k, v, idx, w.block_size, out=out, lse=lse, stream=stream)


def workload_config(w, world):
    """The `config` object of the JSON line for a TRA or NSA workload."""
    from block_sparse_attention_tra_gb300 import workloads

    par = ("single GPU" if world == 1 else
           f"batch-sharded over {world} GPUs: global batch {w.B * world}, rank r takes batches "
           f"[r*{w.B}, (r+1)*{w.B}) drawn with seed r; no collective")
    if isinstance(w, workloads.TraWorkload):
        return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "D": w.D, "beta": w.beta, "p": w.p,
                "causal": True, "l2": "no flush: q,k,v,out = %d MB > 129 MB L2" % (w.io_bytes // 2**20),
                "parallelism": par}
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T, "D": w.D,
            "block_size": w.block_size, "S": w.S, "causal": True,
            "l2": "no flush (unique K/V stays in L2 by design; gathered bytes counted)", "parallelism": par}


def measure_l2_read_gbs(device, mb: int = 48, reps: int = 40):
    """L2 read bandwidth of this GPU, measured here: the library's streaming-
    read probe (16-byte loads that skip L1, four CTAs per SM) over a buffer of
    `mb` MB that the 129 MB L2 holds, read once to warm it and then `reps`
    times between CUDA events.  Returns (GB/s, description)."""
    import torch

    from block_sparse_attention_tra_gb300 import bsa

    buf = torch.ones(mb * 2**20 // 4, dtype=torch.float32, device=device)
    sink = torch.zeros(1, dtype=torch.int32, device=device)
    best = 0.0
    for _ in range(3):
        bsa.read_probe(buf, 2, sink)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        bsa.read_probe(buf, reps, sink)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, mb * 2**20 * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    how = (f"bsa_read_probe: {mb} MB L2-resident buffer read {reps} times per launch with 16-byte L1-bypassing "
           f"loads, 4 CTAs/SM, best of 3, CUDA events")
    return round(best, 1), how


def roofline_for(w, ms_per_launch, pk, sustained: bool, fsa: bool = False):
    from block_sparse_attention_tra_gb300 import workloads

    if isinstance(w, workloads.TraWorkload):
        achieved = w.flops / (ms_per_launch * 1e-3) / 1e12
        peak = pk["bf16_tflops_sustained"] if sustained and pk.get("bf16_tflops_sustained") else pk["bf16_tflops"]
        if w.dtype == "f32":
            peak = None  # fp32 CUDA-core path: no bf16 tensor roofline applies
        return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4) if peak else None,
                "peak_kind": ("sustained" if sustained else "burst") + " bf16 of " + pk["source"],
                "traffic": ncu_traffic("tra", w.name), "kernel": "tra_bf16_pair_kernel (persistent, tcgen05)",
                "algorithmic_flops_per_launch": w.flops}
    achieved = w.algorithmic_bytes / (ms_per_launch * 1e-3) / 1e9
    general = not (w.block_size == 64 and w.D in (64, 128))  # shapes the general kernel serves
    kind = "fsa" if fsa else "nsa_general" if general else "nsa"
    common = {"traffic": ncu_traffic(kind, ("fsa:" if fsa else "") + w.name),
              "kernel": ("fsa_blockouter_kernel + fsa_combine_kernel" if fsa else
                         "nsa_general_kernel" if general else "nsa_select_kernel"),
              "algorithmic_bytes_per_launch": w.algorithmic_bytes,
              "tflops": round(w.flops / (ms_per_launch * 1e-3) / 1e12, 2),
              "unique_bytes_per_launch": w.unique_bytes,
              "hbm": {"peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                      "peak_kind": "copy bandwidth of " + pk["source"]}}
    if pk.get("l2_read_gbs") and not fsa:
        # The gathered K/V (the bulk of the algorithmic bytes) is served from
        # L2: the unique K/V fits it, and DRAM reads stay near the unique bytes.
        r = {"bound": "l2", "achieved": round(achieved, 1), "peak": pk["l2_read_gbs"], "unit": "GB/s",
             "frac": round(achieved / pk["l2_read_gbs"], 4), "peak_kind": pk["l2_how"]}
    else:
        r = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
             "frac": round(achieved / pk["hbm_gbs"], 4), "peak_kind": "copy bandwidth of " + pk["source"]}
    r.update(common)
    if fsa:
        # The split-K form also writes and re-reads its fp32 partials
        # (m, l and a D-vector per (query, selected block, head)).
        parts = w.B * w.Hq * w.T * w.S * (w.D + 2) * 4
        r["partial_bytes_written_and_read"] = 2 * parts
    return r


# MUFU results per clock per SM on GB300 (sm_103a), measured with a one-CTA-
# per-SM throughput loop: lg2.approx.f32 16, ex2.approx.f32 32, sqrt.approx.f32 16.
MUFU_PER_CLK = {"lg2": 16.0, "ex2": 32.0, "sqrt": 16.0}


def sfu_roofline(w, ms_per_launch, sm_mhz, ops):
    """Special-function roofline of a TRA power class: `ops` maps each MUFU
    operation name to how many it evaluates per causal pair (the general
    power with part of its log2 on the FMA pipe uses 12/16 of an lg2).  The
    time the MUFU units of all SMs need at the sampled SM clock, as a fraction
    of the measured time."""
    if not sm_mhz:
        return None
    import torch

    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    pairs = w.B * w.H * (w.T * (w.T + 1) // 2)
    clk_per_pair = sum(n / MUFU_PER_CLK[o] for o, n in ops.items())
    min_ms = pairs * clk_per_pair / sms / (sm_mhz * 1e6) * 1e3
    return {"bound": "sfu", "ops_per_pair": dict(ops), "results_per_clk_per_sm": {o: MUFU_PER_CLK[o] for o in ops},
            "pairs": pairs, "sm_mhz": sm_mhz, "min_ms": round(min_ms, 4), "frac": round(min_ms / ms_per_launch, 4)}


def sfu_ops(w):
    """MUFU operations per causal pair of the power class tra_forward picks
    for this workload's p (None for p = 1, 2: no MUFU work)."""
    if w.dtype != "bf16" or w.p in (1.0, 2.0):
        return None
    if 1.0 <= w.p <= 64.0:  # part of log2 on the FMA pipe: 10 of every 16 score pairs on MUFU lg2
        return {"lg2": 10 / 16, "ex2": 1.0}
    return {"lg2": 1.0, "ex2": 1.0}


def time_resident(fn, steps, warmup, world, flush=None, soak_s=0.0):
    """Device time (ms) of `steps` launches with inputs resident.  Without a
    flush the launches run back to back between two events; with a flush each
    launch is bracketed by its own events and the flush runs outside them.
    `soak_s` seconds of further untimed launches follow, so that a clock
    sampler running around the call sees the GPU under this load."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        total = e0.elapsed_time(e1)
    else:
        evs = []
        for _ in range(steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            evs.append((a, b))
        torch.cuda.synchronize()
        total = sum(a.elapsed_time(b) for a, b in evs)
    if soak_s > 0:
        t0 = time.time()
        while time.time() - t0 < soak_s:
            for _ in range(8):
                fn()
            torch.cuda.synchronize()
    barrier(world)
    return total


def run_ours(args):
    import torch

    from block_sparse_attention_tra_gb300 import bsa, build, workloads

    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    build.build()
    bsa.load_library()
    pk = peaks()

    w, host, dev = make_inputs(args.workload, device, rank)
    out = torch.empty_like(dev[0])
    fn = launcher(w, dev, out)

    # ---- device-resident timing of the headline workload; a region whose
    # clocks show throttling (on any rank) is measured once more
    with ClockSampler(device.index) as cs:
        total_ms = time_resident(fn, args.steps, args.warmup, world, soak_s=args.clock_soak)
    clocks = cs.summary()
    remeasured = reduce_max(1.0 if clocks_rejected(clocks) else 0.0, world, device) > 0
    if remeasured:
        rejected = clocks
        with ClockSampler(device.index) as cs:
            total_ms = time_resident(fn, args.steps, args.warmup, world, soak_s=args.clock_soak)
        clocks = dict(cs.summary(), remeasured_after=rejected)
    total_ms = reduce_max(total_ms, world, device)
    ms = total_ms / args.steps
    flops_all = w.flops * world
    value = flops_all / (total_ms / args.steps * 1e-3) / 1e12

    # ---- end to end through the public API: pinned host -> device, kernel, device -> host
    pinned = [t.pin_memory() for t in host]
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dev2 = [torch.empty_like(t) for t in dev]
    out2 = torch.empty_like(out)
    fn2 = launcher(w, dev2, out2)

    # One side stream per input so that the host->device copies can use
    # several copy engines at once; the kernel waits for all of them.
    main = torch.cuda.current_stream()
    side = [torch.cuda.Stream() for _ in dev2]

    def e2e_step():
        evs = []
        for d, h, st in zip(dev2, pinned, side):
            st.wait_stream(main)
            with torch.cuda.stream(st):
                d.copy_(h, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(st)
            evs.append(ev)
        for ev in evs:
            main.wait_event(ev)
        fn2()
        out_host.copy_(out2, non_blocking=True)

    if isinstance(w, workloads.TraWorkload):
        # TRA: the library's own host-buffer entry point (tra_forward_host),
        # which streams chunks of heads with the copies overlapping the kernels.
        ws = torch.empty(bsa.tra_forward_host_workspace_size(w.B, w.H, w.T, w.D, 1 if w.dtype == "bf16" else 0),
                         dtype=torch.uint8, device=device)

        def e2e_step():  # noqa: F811
            bsa.tra_forward_host(pinned[0], pinned[1], pinned[2], w.beta, w.p, out=out_host, workspace=ws)

    e2e_ms = reduce_max(time_resident(e2e_step, max(3, args.steps // 2), 2, world), world, device)
    e2e_ms /= max(3, args.steps // 2)
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = out.numel() * out.element_size()

    result = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if getattr(w, "dtype", "bf16") == "bf16" else "f32",  # NSA is bf16 only
        "data": "synthetic (seeded N(0,1) q,k,v; no dataset)",
        "config": workload_config(w, world),
        "roofline": roofline_for(w, ms, pk, sustained=False),
        "e2e": {"value": round(flops_all / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": ("tra_forward_host (C ABI, pinned host q, k, v, out; chunks of heads, copies overlapping "
                         "kernels)" if isinstance(w, workloads.TraWorkload) else
                         "pinned host -> device copies, nsa_select_forward, device -> host copy")},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if isinstance(w, workloads.TraWorkload) and sfu_ops(w):
        # the general power's epilogue is bounded by the MUFU unit, not the tensor pipe
        result["sfu"] = sfu_roofline(w, ms, clocks.get("sm_mhz"), sfu_ops(w))

    # ---- secondary workloads (measured, reported beside the headline)
    if not args.no_secondary:
        flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)

        def flush():
            flush_buf.fill_(1.0)

        sec = []
        sfu_clock = clocks.get("sm_mhz")
        pk["l2_read_gbs"], pk["l2_how"] = measure_l2_read_gbs(device)
        result["l2_read_gbs_measured"] = {"value": pk["l2_read_gbs"], "how": pk["l2_how"]}
        for name in SECONDARY:
            del dev, out
            torch.cuda.empty_cache()
            w2, _, dev = make_inputs(name, device, rank)
            out = torch.empty_like(dev[0])
            lse = None
            if isinstance(w2, workloads.NsaWorkload):
                lse = torch.empty((w2.B, w2.Hq, w2.T), dtype=torch.float32, device=device)
            f = launcher(w2, dev, out, lse)
            n = max(3, args.steps // 2)
            # TRA inputs larger than L2 need no flush (back-to-back launches, as
            # for the headline); the NSA gather's unique K/V fits L2, so those
            # launches are flushed.
            big = isinstance(w2, workloads.TraWorkload) and w2.io_bytes > L2_BYTES
            with ClockSampler(device.index) as cs2:
                t = time_resident(f, n, 3, world, flush=None if big else flush, soak_s=min(args.clock_soak, 1.0))
            t = reduce_max(t, world, device) / n
            entry = {"workload": w2.name, "ms_per_launch": round(t, 4), "clocks": cs2.summary(),
                     "tflops": round(w2.flops * world / (t * 1e-3) / 1e12, 3),
                     "roofline": roofline_for(w2, t, pk, sustained=False),
                     "l2": ("no flush: inputs %d MB > 129 MB L2" % (w2.io_bytes // 2**20)) if big
                     else "flushed between launches"}
            if isinstance(w2, workloads.TraWorkload) and sfu_ops(w2):
                # general power: exp2(p log2 x), an ex2 and (part of) an lg2 per causal pair
                entry["sfu"] = sfu_roofline(w2, t, entry["clocks"]["sm_mhz"], sfu_ops(w2))
            sec.append(entry)
            if isinstance(w2, workloads.NsaWorkload) and w2.block_size == 64 and w2.D in (64, 128):
                # The same selection through the block-outer split-K form
                # (six launches: list build, block pass, combine).
                q2, k2, v2, idx2 = dev
                ws = torch.empty(bsa.nsa_select_fsa_workspace_size(w2.B, w2.Hq, w2.Hkv, w2.T, w2.D,
                                                                   w2.block_size, w2.S),
                                 dtype=torch.uint8, device=device)
                f = lambda: bsa.nsa_select_forward_fsa(q2, k2, v2, idx2, w2.block_size, out=out,  # noqa: E731
                                                       lse=lse, workspace=ws)
                t = reduce_max(time_resident(f, n, 3, world, flush=flush), world, device) / n
                sec.append({"workload": f"nsa_select_forward_fsa on {w2.name}", "ms_per_launch": round(t, 4),
                            "tflops": round(w2.flops * world / (t * 1e-3) / 1e12, 3),
                            "roofline": roofline_for(w2, t, pk, sustained=False, fsa=True),
                            "gpu_launches_per_call": 6, "l2": "flushed between launches"})
                del ws, q2, k2, v2, idx2, f
        # The widened rows on the headline shape: training backward and the
        # fused differential forward (two score streams, with normalisation).
        del dev, out
        torch.cuda.empty_cache()
        wb = workloads.TRA_WORKLOADS[WIDENED_WORKLOAD]
        qb, kb, vb = (t.to(device) for t in workloads.workload_inputs(wb))
        gen = torch.Generator(device="cpu").manual_seed(1)
        dob = torch.randn(qb.shape, generator=gen).to(torch.bfloat16).to(device)
        q2b = torch.randn(qb.shape, generator=gen).to(torch.bfloat16).to(device)
        k2b = torch.randn(qb.shape, generator=gen).to(torch.bfloat16).to(device)
        n = max(3, args.steps // 2)
        extra = [
            ("tra_backward", wb.name, lambda: bsa.tra_backward(qb, kb, vb, dob, wb.beta, wb.p), 10 * wb.flops // 4),
            ("tra_backward(deterministic: two kernels)", wb.name,
             lambda: bsa.tra_backward(qb, kb, vb, dob, wb.beta, wb.p, deterministic=True), 10 * wb.flops // 4),
            ("tra_diff_forward(normalize=1, lambda=0.5)", wb.name,
             lambda: bsa.tra_diff_forward(qb, q2b, kb, k2b, vb, wb.beta, 0.5, wb.p, normalize=True), 2 * wb.flops),
            # gradients of the differential form, dlambda included: two backward passes (10 D FLOPs per pair
            # each) and the normalisation / combination glue (dlambda is summed in the combination)
            ("tra_diff_backward(normalize=1, lambda=0.5, dlambda)", wb.name,
             lambda: bsa.tra_diff_backward(qb, q2b, kb, k2b, vb, dob, wb.beta, 0.5, wb.p, normalize=True,
                                           want_dlam=True),
             2 * 10 * wb.flops // 4),
        ]
        # The half-power variant on the T=8192 general-power workload (p = 1.5
        # as x sqrt(x); a variant of that workload, whose line above is exp/log).
        w3 = workloads.TRA_WORKLOADS["tra_bf16_B2_H32_T8192_D64"]
        q3, k3, v3 = (t.to(device) for t in workloads.workload_inputs(w3))
        o3 = torch.empty_like(q3)
        extra.append(("tra_forward(sqrt_half_powers)", w3.name,
                      lambda: bsa.tra_forward(q3, k3, v3, w3.beta, w3.p, out=o3, sqrt_half_powers=True), w3.flops))
        # Each of these reads and writes four to seven 64-268 MB tensors (more
        # than L2), so the calls run back to back without a flush: a flush
        # before every call would also let each call's host-side work (tensor
        # maps, scratch, marshalling) show up as idle device time.
        for label, wname, f, flops in extra:
            t = reduce_max(time_resident(f, n, 3, world, flush=None), world, device) / n
            sec.append({"workload": f"{label} on {wname}", "ms_per_launch": round(t, 4),
                        "tflops": round(flops * world / (t * 1e-3) / 1e12, 3),
                        "frac_of_bf16_peak": round(flops / (t * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                        "algorithmic_flops": flops, "l2": "no flush: inputs and outputs > 129 MB L2"})
            if label.startswith("tra_forward(sqrt_half_powers)"):
                # p = 1.5 as x sqrt(x): one sqrt per causal pair (clock of the exp/log line's run)
                sec[-1]["sfu"] = sfu_roofline(w3, t, sfu_clock, {"sqrt": 1.0})
        result["secondary"] = sec

    if args.cpu_baseline and rank == 0 and world == 1:
        result["cpu_baseline"] = cpu_baseline(w, host, budget_s=args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return result if rank == 0 else None


# ------------------------------------------------------------ CPU oracle leg

def oracle_units(w, host, n, seed=0):
    """Run the float64 oracle on the first ``n`` units of the workload --
    whole (b, h) heads for TRA, seeded random query groups for NSA -- and
    return the algorithmic FLOPs of that work (4 D per causal pair and head)."""
    import numpy as np

    from block_sparse_attention_tra_gb300 import workloads
    from oracle import nsa as onsa
    from oracle import tra as otra

    if isinstance(w, workloads.TraWorkload):
        q, k, v = host
        flops = 0
        for u in range(n):
            b, h = divmod(u % (w.B * w.H), w.H)
            sl = (slice(b, b + 1), slice(h, h + 1))
            otra.tra_forward(q[sl].double().numpy(), k[sl].double().numpy(), v[sl].double().numpy(), w.beta, w.p)
            flops += otra.tra_flops(1, 1, w.T, w.D)
        return flops
    q, k, v, idx = host
    G = w.G
    rng = np.random.default_rng(seed)
    pairs = 0
    for _ in range(n):
        b, g, i = int(rng.integers(w.B)), int(rng.integers(w.Hkv)), int(rng.integers(w.T))
        toks = onsa.selected_tokens(idx[b, g, i].numpy(), i, w.block_size)
        onsa.softmax_attend(q[b, g * G:(g + 1) * G, i].double().numpy(), k[b, g, toks].double().numpy(),
                            v[b, g, toks].double().numpy(), w.D ** -0.5)
        pairs += toks.size
    return 4 * G * w.D * pairs


def oracle_sample_size(w, host, budget_s):
    """Units of work (heads or query groups) the oracle gets through in about
    ``budget_s`` seconds on this host, from one timed calibration call."""
    from block_sparse_attention_tra_gb300 import workloads

    probe = 1 if isinstance(w, workloads.TraWorkload) else 64
    t0 = time.perf_counter()
    oracle_units(w, host, probe, seed=1)
    dt = max(time.perf_counter() - t0, 1e-6)
    return max(1, int(budget_s / dt * probe))


def unit_name(w, n):
    from block_sparse_attention_tra_gb300 import workloads

    if isinstance(w, workloads.TraWorkload):
        return f"{n} of {w.B * w.H} (b,h) heads of {w.name}"
    return f"{n} seeded random query groups (G={w.G} heads each) of {w.name}"


def cpu_baseline(w, host, budget_s=15.0):
    """Time the float64 oracle on the host cores on a bounded sample of the
    same workload (whole heads for TRA, query groups for NSA), about
    ``budget_s`` seconds of work.  Returns the metric in the same unit."""
    cores = len(os.sched_getaffinity(0))
    n = oracle_sample_size(w, host, budget_s)
    t0 = time.perf_counter()
    flops = oracle_units(w, host, n)
    done = time.perf_counter() - t0
    return {"value": round(flops / done / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{unit_name(w, n)}, float64 numpy/BLAS, {done:.1f} s"}


def run_reference(args):
    """The reference arm: the float64 CPU oracle on the host cores (rank 0
    only).  Every step runs the same bounded sample of the workload (whole
    heads for TRA, query groups for NSA), sized once before the warm-up so
    that the whole run takes a few minutes; ``ms_per_step`` is the measured
    time of that sampled work and ``value`` its FLOPs over that time --
    nothing is scaled up to the full workload."""
    rank, world, _ = dist_info()
    if rank != 0:
        return None
    from block_sparse_attention_tra_gb300 import workloads

    w = workloads.TRA_WORKLOADS.get(args.workload) or workloads.NSA_WORKLOADS[args.workload]
    host = workloads.workload_inputs(w)
    per_step = min(6.0, max(1.0, 150.0 / max(1, args.steps + args.warmup)))
    n = oracle_sample_size(w, host, per_step)
    for _ in range(args.warmup):
        oracle_units(w, host, n)
    times, flops = [], 0
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        flops = oracle_units(w, host, n)
        times.append(time.perf_counter() - t0)
    total_s = time.perf_counter() - t_all
    ms = total_s / args.steps * 1e3
    value = flops / (ms * 1e-3) / 1e12
    cores = len(os.sched_getaffinity(0))
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q,k,v; no dataset)",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": (f"each step: {unit_name(w, n)} ({flops:.4g} FLOP), float64 numpy/BLAS; "
                                    f"median step {statistics.median(times):.2f} s")},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_op(args):
    """Time one of the widened ops (TRA backward or the fused differential
    forward on a TRA workload; the block-outer split-K NSA form on an NSA
    workload); prints a JSON line of the same metric.  Used for the
    per-kernel measurements and ncu captures of those rows."""
    import torch

    from block_sparse_attention_tra_gb300 import bsa, build, workloads

    torch.cuda.set_device(0)
    build.build()
    bsa.load_library()
    pk = peaks()
    if args.op == "fsa":
        w = workloads.NSA_WORKLOADS[args.workload]
        q, k, v, idx = (t.cuda() for t in workloads.workload_inputs(w))
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.T), dtype=torch.float32, device=q.device)
        ws = torch.empty(bsa.nsa_select_fsa_workspace_size(w.B, w.Hq, w.Hkv, w.T, w.D, w.block_size, w.S),
                         dtype=torch.uint8, device=q.device)
        fn = lambda: bsa.nsa_select_forward_fsa(q, k, v, idx, w.block_size, out=out, lse=lse,  # noqa: E731
                                                workspace=ws)
        with ClockSampler(0) as cs:
            total = time_resident(fn, args.steps, args.warmup, 1, soak_s=args.clock_soak)
        ms = total / args.steps
        value = w.flops / (ms * 1e-3) / 1e12
        return {"metric": METRIC, "op": args.op, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
                "higher_is_better": True, "dtype": "bf16", "data": "synthetic", "config": workload_config(w, 1),
                "roofline": roofline_for(w, ms, pk, sustained=False, fsa=True),
                "gpu_launches": 6 * args.steps, "clocks": cs.summary()}
    w = workloads.TRA_WORKLOADS[args.workload]
    q, k, v = (t.cuda() for t in workloads.workload_inputs(w))
    gen = torch.Generator().manual_seed(1)
    extra = [torch.randn(q.shape, generator=gen).to(torch.bfloat16).cuda() for _ in range(2)]
    if args.op == "backward":
        fn = lambda: bsa.tra_backward(q, k, v, extra[0], w.beta, w.p)  # noqa: E731
        flops = 10 * w.flops // 4
        launches = 3  # dq accumulator zeroing, the fused kernel, dq conversion
    elif args.op == "backward-deterministic":
        fn = lambda: bsa.tra_backward(q, k, v, extra[0], w.beta, w.p, deterministic=True)  # noqa: E731
        flops = 10 * w.flops // 4
        launches = 1  # dK/dV and dQ blocks in one grid
    elif args.op == "diff-backward":
        q2, k2 = (torch.randn(q.shape, generator=gen).to(torch.bfloat16).cuda() for _ in range(2))
        fn = lambda: bsa.tra_diff_backward(q, q2, k, k2, v, extra[0], w.beta, 0.5, w.p,  # noqa: E731
                                           normalize=True, want_dlam=True)
        flops = 2 * 10 * w.flops // 4
        launches = 6  # normalisation, two fused backward passes (zeroing + kernel each), combination
    else:
        fn = lambda: bsa.tra_diff_forward(q, extra[0], k, extra[1], v, w.beta, 0.5, w.p, normalize=True)  # noqa: E731
        flops = 2 * w.flops
        launches = 2
    with ClockSampler(0) as cs:
        total = time_resident(fn, args.steps, args.warmup, 1, soak_s=args.clock_soak)
    ms = total / args.steps
    value = flops / (ms * 1e-3) / 1e12
    return {"metric": METRIC, "op": args.op, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic", "config": workload_config(w, 1),
            "roofline": {"bound": "tensor", "achieved": round(value, 2), "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(value / pk["bf16_tflops"], 4),
                         "algorithmic_flops_per_step": flops},
            "gpu_launches": launches * args.steps, "clocks": cs.summary()}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--op", choices=["forward", "backward", "backward-deterministic", "diff", "diff-backward", "fsa"],
                    default="forward",
                    help="forward (the headline path), or one widened op timed on its own")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--clock-soak", type=float, default=1.5,
                    help="seconds of untimed launches after the timed region, under the clock sampler")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        res = run_reference(args)
    elif args.op != "forward":
        res = run_op(args)
    else:
        res = run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
