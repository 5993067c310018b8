"""Benchmark: one block-quantized MoE layer on the T=4 MTP verify batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one full layer forward (router, top-k, permutation, gate/up +
SwiGLU, down, combine) over one synthetic batch, through the library's C ABI.
Prints ONE JSON line (rank 0).  Multi-GPU runs are independent replicas, one
per rank (the layer has no data-path exchange): value = max-over-ranks time /
layers processed by all ranks.

L2 hygiene: the timed loop rotates over ``--copies`` separately allocated
copies of the layer weights (each copy's bytes exceed the 129 MB L2).

--impl reference times the oracle (plain numpy CPU code) on the same
workload, extrapolated from bounded samples; it is a deliberately slow
baseline, not a competitor.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/MoE layer and effective HBM GB/s (T=4 verify, 352×top-8) vs 8 TB/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--workload", default="verify_q8")
    p.add_argument("--copies", type=int, default=None,
                   help="weight copies rotated in the timed loop (default 4 for T <= 8, 1 above: one layer then "
                        "touches every expert, far more than L2)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=2000)
    p.add_argument("--experts", type=int, default=0,
                   help="override the expert count (smaller resident layer for profiler captures)")
    p.add_argument("--tokens", type=int, default=0,
                   help="override the batch size T (with --experts: the same tokens per expert on a smaller layer)")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def replica_max_ms(total_ms, device):
    """The job's time: the longest rank's timed region (every rank ran the same
    steps on its own replica; no data-path exchange)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(total_ms)
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def per_unit_us(total_ms, steps, world):
    """Whole-job µs per unit (layer or round): the job's time over the units
    that all ranks processed."""
    return total_ms * 1e3 / (steps * world)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def cpu_model():
    """The host CPU's model name (from /proc/cpuinfo, else lscpu), for the
    cpu_baseline record."""
    import platform
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def algorithmic_bytes(w, n_unique):
    """Router weight + bias + unique routed experts + shared expert + x + y,
    at the serialised sizes of their formats."""
    def mat(fmt, rows, cols):
        return rows * (cols // 32 * 34 if fmt == 2 else cols // 256 * 144)
    per_expert = 2 * mat(w.routed_fmt, w.I, w.H) + mat(w.routed_fmt, w.H, w.I)
    shared = 2 * mat(w.shared_fmt, w.I_shared, w.H) + mat(w.shared_fmt, w.H, w.I_shared) if w.I_shared else 0
    router = w.E * w.H * 4 + (w.E * 4 if w.bias_std is not None else 0)
    act = 2 * w.T * w.H * 2
    return router + n_unique * per_expert + shared + act


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm = [float(r[1]) for r in self.rows if len(r) >= 8 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 8 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows if len(r) >= 8 for i in range(4)
                          if r[4 + i].lower() in ("active", "1")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sm)}


def measured_tensor_peak():
    """Sustained dense bf16 TFLOP/s from MEASURED_PEAKS.json (a kernel timed inside
    a long step), else the fallback figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if d.get("bf16_tflops_sustained"):
            return float(d["bf16_tflops_sustained"]), "measured sustained cuBLAS bf16 (MEASURED_PEAKS.json)"
    return 1700.0, "fallback sustained bf16 figure"


def expert_load_summary(offsets):
    """Tokens per expert (M_e) from the routing offsets [E+1]: how many experts
    got work, and the spread of their loads (a histogram over power-of-two
    bins: bin b counts experts with 2^b <= M_e < 2^(b+1))."""
    off = np.asarray(offsets, dtype=np.int64)
    m = off[1:] - off[:-1]
    used = m[m > 0]
    if used.size == 0:
        return {"experts_used": 0}
    bins = np.bincount(np.floor(np.log2(used)).astype(np.int64))
    return {"experts_used": int(used.size), "pairs": int(m.sum()), "min": int(used.min()),
            "median": float(np.median(used)), "max": int(used.max()),
            "pow2_hist": [int(b) for b in bins]}


def run_e2e(stream, steps, host_in, dev_in, run, dev_out, host_out):
    """End-to-end steps: each step copies its inputs host -> device (pinned),
    runs, and copies its result device -> host (pinned).  The copies have their
    own streams and the buffers are doubled, so step i+1's input copy and step
    i's result copy overlap the neighbouring steps' kernels, as a serving loop
    would run them.  dev_in[b] / dev_out[b] / host_out[b]: lists of tensors of
    buffer b; run(i, b) launches step i on `stream` reading dev_in[b] and
    writing dev_out[b].  Returns µs per step: events on `stream` from before
    the first input copy to after the last result copy."""
    import torch
    nb = len(dev_in)
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    x_ready = [torch.cuda.Event() for _ in range(nb)]
    ran = [torch.cuda.Event() for _ in range(nb)]
    y_read = [torch.cuda.Event() for _ in range(nb)]
    # a few untimed steps on the same streams and buffers first (warm-up)
    if steps > 0:
        _e2e_loop(stream, min(3, steps), host_in, dev_in, run, dev_out, host_out, h2d, d2h, x_ready, ran, y_read)
    return _e2e_loop(stream, steps, host_in, dev_in, run, dev_out, host_out, h2d, d2h, x_ready, ran, y_read)


def _e2e_loop(stream, steps, host_in, dev_in, run, dev_out, host_out, h2d, d2h, x_ready, ran, y_read):
    import torch
    nb = len(dev_in)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    h2d.wait_event(e0)

    def copy_in(i):
        b = i % nb
        with torch.cuda.stream(h2d):
            if i >= nb:
                h2d.wait_event(ran[b])  # step i - nb has read buffer b
            for d, h in zip(dev_in[b], host_in):
                d.copy_(h, non_blocking=True)
            x_ready[b].record(h2d)

    copy_in(0)
    for i in range(steps):
        b = i % nb
        if i + 1 < steps:
            copy_in(i + 1)
        stream.wait_event(x_ready[b])
        if i >= nb:
            stream.wait_event(y_read[b])  # step i - nb's result has been copied out
        run(i, b)
        ran[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ran[b])
            for h, d in zip(host_out[b], dev_out[b]):
                h.copy_(d, non_blocking=True)
            y_read[b].record(d2h)
    stream.wait_event(y_read[(steps - 1) % nb])
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / steps


E2E_NOTE = ("every step: inputs host->device from pinned memory, the step, result device->host to pinned "
            "memory; copies on their own streams, buffers doubled, so copies overlap neighbouring steps")


KERNEL_SOURCES = {  # the files each path's kernels are compiled from
    "small_t": ("small_t.cu", "gemv.cuh", "layer.cuh", "common.cuh"),
    "large_t": ("gemm_tc.cu", "large_t.cuh", "tc.cuh", "layer.cuh", "common.cuh"),
}


def kernel_hash(path):
    """Hash of the sources the path's dominant kernel is compiled from."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[path]:
        h.update(open(os.path.join(ROOT, "block_quantized_moe_layer_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_record(path, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources for this workload (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    return json.load(open(p)).get(f"{kernel_hash(path)}:{workload}")


def cpu_baseline_sample(w, budget_s=20.0):
    """The oracle on a bounded sample of the workload (one layer forward on a
    T-token batch per repetition), on this host's cores; returns µs/layer."""
    import torch
    from oracle import moe as omoe
    from tests._oracle_layer import synth_oracle_layer
    from block_quantized_moe_layer_gb300 import synth
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    times = []
    variant = 0
    t_end = time.time() + budget_s
    while time.time() < t_end and variant < 8:
        ol = synth_oracle_layer(w, dev)
        x = synth.activations(w, "cpu", variant=variant).float().numpy()
        r = omoe.route(x, ol)
        for e in r["act"]:          # quantise outside the timed part (weight preparation)
            ol.expert(int(e))
        t0 = time.perf_counter()
        omoe.forward(x, ol)
        times.append(time.perf_counter() - t0)
        variant += 1
    return statistics.median(times) * 1e6, len(times)


def run_ours(args):
    import torch
    import block_quantized_moe_layer_gb300 as pkg
    from block_quantized_moe_layer_gb300 import synth
    from block_quantized_moe_layer_gb300.workloads import synthetic_layer

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if args.workload in synth.ROUNDS:
        return run_round(args)
    w = synth.WORKLOADS[args.workload]
    if args.experts or args.tokens:
        import dataclasses
        w = dataclasses.replace(w, E=args.experts or w.E, T=args.tokens or w.T)
    copies = args.copies if args.copies is not None else (4 if w.T <= 8 else 1)
    layers = [synthetic_layer(w, pkg.ACT_BF16, T_max=w.T)[0] for _ in range(copies)]
    x = synth.activations(w, "cuda")
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    # routing of the workload's batch (for the algorithmic bytes), untimed
    layers[0].forward(x, y)
    torch.cuda.synchronize()
    layers[0].status()
    offs = layers[0].routing(w.T)[2]
    n_unique = int((offs[1:] > offs[:-1]).sum().item())
    load = expert_load_summary(offs.cpu().numpy())
    alg = algorithmic_bytes(w, n_unique)

    # The clock sampler starts (and settles) before the warm-up, so the GPU
    # runs the warm-up steps right up to the timed region; the timed region
    # is exactly K back-to-back steps with nothing between the launches.
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for i in range(max(args.warmup, 3)):
        layers[i % len(layers)].forward(x, y)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        layers[i % len(layers)].forward(x, y)
    t_stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    for L in layers:
        L.status()
    # phase timeline of the timed loop's last launch (T <= 8 kernel)
    phases = layers[(args.steps - 1) % len(layers)].timeline() if w.T <= 8 else None
    total_ms = t_start.elapsed_time(t_stop)
    # diagnostic, after the timed region: single launches bracketed by events
    # (an event between two launches removes their programmatic overlap)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(min(16, max(args.steps, 1)))]
    for i, (a, b) in enumerate(evs):
        a.record(stream)
        layers[i % len(layers)].forward(x, y)
        b.record(stream)
    torch.cuda.synchronize()
    launch_us = [a.elapsed_time(b) * 1e3 for (a, b) in evs]
    total_ms = replica_max_ms(total_ms, "cuda")
    us_per_layer = per_unit_us(total_ms, args.steps, world)
    # The roofline's launch duration: a T <= 8 step is one launch, so the
    # average launch duration over the timed region is the step time (events
    # on the launching stream around all K steps).  The event-bracketed
    # launches below are a diagnostic only: an event between two launches
    # removes their programmatic-launch overlap.  A T > 8 forward is eight
    # launches whose grouped GEMMs dominate; its unit is the whole forward.
    kern_us = total_ms * 1e3 / args.steps

    # end to end through the public call: pinned host x -> device, forward,
    # device -> pinned host y, every step
    xh = x.cpu().pin_memory()
    xd = [torch.empty_like(x) for _ in range(2)]
    yd = [torch.empty_like(x) for _ in range(2)]
    yh = [torch.empty_like(xh).pin_memory() for _ in range(2)]
    e2e_steps = max(2, min(args.e2e_steps, args.steps))
    e2e_us = run_e2e(stream, e2e_steps, [xh], [[a] for a in xd],
                     lambda i, b: layers[i % len(layers)].forward(xd[b], yd[b]), [[a] for a in yd],
                     [[a] for a in yh])
    assert torch.equal(yh[(e2e_steps - 1) % 2].cuda(), y)

    peak, peak_src = measured_peaks()
    achieved = alg / (kern_us * 1e-6) / 1e9
    tr = traffic_record("small_t" if w.T <= 8 else "large_t", w.name)
    kname = "moe_small_t_kernel" if w.T <= 8 else "moe_forward (8 launches; the grouped tcgen05 GEMMs dominate)"
    out = {
        "metric": METRIC,
        "value": round(us_per_layer, 3),
        "unit": "us/layer",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "q8_0 weights x bf16 activations (int dp4a, fp32 accumulate)",
        "data": "synthetic (seeded, random-init weights of the workload's shapes)",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "top_k": w.top_k, "I": w.I,
                   "I_shared": w.I_shared, "routed_fmt": ["f32", "bf16", "q8_0", "q4ks"][w.routed_fmt],
                   "unique_experts": n_unique, "algorithmic_bytes": alg, "tokens_per_expert": load,
                   "l2": f"rotating {len(layers)} weight copies of {layers[0].weight_bytes / 1e9:.2f} GB (> L2)",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(w.T / (us_per_layer * 1e-6), 1),
        "effective_gbs": round(alg / (us_per_layer * 1e-6) / 1e9, 1),
        "frac_of_8tbs": round(alg / (us_per_layer * 1e-6) / 8e12, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": tr["bytes_per_launch"] if tr else None,
                     "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": kname, "kernel_us": round(kern_us, 3)},
        "clocks": clk,
        "e2e": {"value": round(e2e_us, 3), "unit": "us/layer", "h2d_bytes_per_step": xh.numel() * xh.element_size(),
                "d2h_bytes_per_step": yh[0].numel() * yh[0].element_size(), "steps": e2e_steps,
                "copies": E2E_NOTE},
        "gpu_launches": args.steps * (1 if w.T <= 8 else 8),
        # µs after the first block passed its dependency wait, last timed launch
        "phases_us": ({k: (None if v is None else round(v, 2)) for k, v in phases.items()} if phases else None),
        # diagnostic: event-bracketed launches (every 8th of the timed loop;
        # the events remove those launches' overlap with their neighbours)
        "launch_us": {"p10": round(float(np.percentile(launch_us, 10)), 3),
                      "p50": round(float(np.percentile(launch_us, 50)), 3),
                      "p90": round(float(np.percentile(launch_us, 90)), 3), "samples": len(launch_us)},
    }
    if w.T > 8:
        # HBM-bound like the T <= 8 path (about 49 flop/B against a ridge of
        # ~257 flop/B at the measured peaks): the roofline is HBM over the
        # forward's algorithmic bytes; the tensor pipe's share is secondary
        flops = 2.0 * w.T * (w.top_k * 3 * w.H * w.I + 3 * w.H * w.I_shared + w.H * w.E)
        tpk, tsrc = measured_tensor_peak()
        got = flops / (kern_us * 1e-6) / 1e12
        out["roofline"]["kernel_us"] = round(kern_us, 3)
        out["tensor"] = {"useful_tflops": round(got, 1), "peak": tpk, "frac": round(got / tpk, 4),
                         "peak_source": tsrc, "flops_per_forward": flops,
                         "note": "useful FLOPs (routed + shared + router) / forward time; secondary to the HBM bound"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        us, n = cpu_baseline_sample(w)
        out["cpu_baseline"] = {"value": round(us, 1), "unit": "us/layer", "cores": os.cpu_count(),
                               "cpu": cpu_model(), "kind": "oracle",
                               "sample": f"{n} full layer forwards (T={w.T}, distinct x), median; numpy fp64, "
                                         f"BLAS on up to {os.cpu_count()} threads"}
    for L in layers:
        L.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


def run_round(args):
    """One MTP draft/verify round per step (8 target layers, 3 draft heads, two
    LM-head passes, acceptance) through the mtp_round C call."""
    import ctypes
    import torch
    import block_quantized_moe_layer_gb300 as pkg
    from block_quantized_moe_layer_gb300 import synth
    from block_quantized_moe_layer_gb300.workloads import synthetic_round
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    r = synth.ROUNDS[args.workload]
    layers, heads, lm = synthetic_round(r, pkg.ACT_BF16)
    x, noise = synth.round_inputs(r, "cuda")
    H, V, k = lm.H, lm.V, r.k
    ws = pkg.round_workspace(H, k, V, pkg.ACT_BF16)
    wp, wn = pkg._aligned(ws)
    logits = torch.empty(k + 1, V, dtype=torch.float32, device="cuda")
    drafts = torch.empty(k, dtype=torch.int32, device="cuda")
    acc = torch.empty(2, dtype=torch.int32, device="cuda")
    tl = (ctypes.c_void_p * len(layers))(*[L.handle.value for L in layers])
    hl = (ctypes.c_void_p * k)(*[L.handle.value for L in heads])
    stream = torch.cuda.current_stream()
    lib = pkg.lib()

    def step(xd, nd, acc=acc, drafts=drafts):
        rc = lib.mtp_round(tl, len(layers), hl, k, lm.handle, xd.data_ptr(), nd.data_ptr(), 1e-6, 0.0, wp, wn,
                           logits.data_ptr(), None, None, drafts.data_ptr(), acc.data_ptr(), acc.data_ptr() + 4,
                           stream.cuda_stream)
        if rc:
            raise RuntimeError(lib.moe_last_error().decode())
    step(x, noise)  # untimed: the routing of every layer, for the algorithmic bytes
    torch.cuda.synchronize()
    for L in layers + heads:
        L.status()
    # algorithmic bytes of one round: each layer's router, unique experts and
    # shared expert at its batch size, plus two LM-head passes
    alg = 0
    for L, wl in list(zip(layers, r.layers)) + list(zip(heads, r.heads)):
        offs = L.routing(wl.T)[2]
        alg += algorithmic_bytes(wl, int((offs[1:] > offs[:-1]).sum().item()))
    alg += 2 * V * (H // 32) * 34
    steps = min(args.steps, 500)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # clock sampler first, then the warm-up right up to the timed region
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(max(args.warmup, 3)):
        step(x, noise)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(steps):
        step(x, noise)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    us = per_unit_us(replica_max_ms(t0.elapsed_time(t1), "cuda"), steps, world)
    xh, nh = x.cpu().pin_memory(), noise.cpu().pin_memory()
    xd = [torch.empty_like(x) for _ in range(2)]
    nd = [torch.empty_like(noise) for _ in range(2)]
    ad = [torch.empty(2, dtype=torch.int32, device="cuda") for _ in range(2)]
    dd = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(2)]
    ah = [torch.empty(2, dtype=torch.int32).pin_memory() for _ in range(2)]
    dh = [torch.empty(k, dtype=torch.int32).pin_memory() for _ in range(2)]
    e2e_steps = max(2, min(args.e2e_steps, steps))
    e2e = run_e2e(stream, e2e_steps, [xh, nh], [[xd[b], nd[b]] for b in range(2)],
                  lambda i, b: step(xd[b], nd[b], ad[b], dd[b]), [[ad[b], dd[b]] for b in range(2)],
                  [[ah[b], dh[b]] for b in range(2)])
    assert ah[(e2e_steps - 1) % 2].tolist() == acc.cpu().tolist()
    peak, peak_src = measured_peaks()
    out = {
        "metric": "µs per MTP draft/verify round (8 target layers T=4, draft heads T=1,2,3, 2 LM-head passes, "
                  "acceptance) and effective HBM GB/s",
        "value": round(us, 2), "unit": "us/round", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "q8_0/q4ks weights x bf16 activations (int dp4a, fp32 accumulate)",
        "data": "synthetic (seeded, random-init weights of the workload's shapes)",
        "config": {"workload": r.name, "k": k, "V": V, "H": H, "target_layers": len(layers),
                   "algorithmic_bytes": alg, "n_accepted_last": int(acc[0].item())},
        "effective_gbs": round(alg / (us * 1e-6) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(alg / (us * 1e-6) / 1e9, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(alg / (us * 1e-6) / 1e9 / peak, 4),
                     "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": "mtp_round (whole round)"},
        "clocks": clk,
        "e2e": {"value": round(e2e, 2), "unit": "us/round",
                "h2d_bytes_per_step": x.numel() * x.element_size() + noise.numel() * noise.element_size(),
                "d2h_bytes_per_step": 4 * (2 + k), "steps": e2e_steps, "copies": E2E_NOTE},
        # per round: a layer launch and a residual/norm launch per target layer, the
        # first norm, two LM-head launches, draft rows, the heads, argmax, acceptance
        "gpu_launches": steps * (2 * len(layers) + len(heads) + 6),
    }
    for L in layers + heads:
        L.close()
    lm.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


def run_reference(args):
    """The oracle on bounded samples of the workload: each step runs the
    oracle's routing for the batch plus the FFN of a slice of the touched
    row blocks; µs/layer is extrapolated from time per row block."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from block_quantized_moe_layer_gb300 import synth as _synth
    if args.workload in _synth.ROUNDS:
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times single-layer workloads only"}))
        return
    import torch
    from oracle import moe as omoe
    from tests._oracle_layer import synth_oracle_layer
    from block_quantized_moe_layer_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    ol = synth_oracle_layer(w, dev)
    x = synth.activations(w, "cpu").float().numpy()
    r = omoe.route(x, ol)
    # work list: 32-row blocks of every touched matrix with the rows they multiply
    def sub(q, r0):
        rb = q.data.shape[1]
        return omoe.QTensor(q.fmt, 32, q.cols, q.data[r0:r0 + 32].reshape(32, rb))
    blocks = []
    items = []
    for e in r["act"]:
        e = int(e)
        sl = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
        items.append((ol.expert(e), x[sl // w.top_k]))
    items.append((ol.shared, x))
    for ex, xr in items:
        u = xr @ ex.gate.dense().T
        h = omoe.silu(u) * (xr @ ex.up.dense().T)
        blocks += [(ex.gate, r0, xr) for r0 in range(0, ex.gate.rows, 32)]
        blocks += [(ex.up, r0, xr) for r0 in range(0, ex.up.rows, 32)]
        blocks += [(ex.down, r0, h) for r0 in range(0, ex.down.rows, 32)]

    def block(i):
        q, r0, inp = blocks[i % len(blocks)]
        return inp @ sub(q, r0).dense().T
    n_blocks = len(blocks)
    t0 = time.perf_counter()
    omoe.route(x, ol)
    t_route = time.perf_counter() - t0
    t0 = time.perf_counter()
    block(0)
    t_blk = max(time.perf_counter() - t0, 1e-5)
    budget = 90.0
    per_step = int(max(1, min(n_blocks, budget / max(1, args.steps + args.warmup) / t_blk)))
    i = 0
    for _ in range(args.warmup):
        for _ in range(per_step):
            block(i)
            i += 1
    samples = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        for _ in range(per_step):
            block(i)
            i += 1
        samples.append((time.perf_counter() - t0) / per_step)
    us = (t_route + statistics.median(samples) * n_blocks) * 1e6
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/layer",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp64 (numpy oracle)", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "top_k": w.top_k, "I": w.I},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/layer", "cores": os.cpu_count(), "cpu": cpu_model(),
                         "kind": "oracle", "sample": f"routing of the batch once + {per_step} of the layer's {n_blocks} "
                                   f"32-row weight blocks (dequantise + multiply) per step; "
                                   f"time per block x blocks per layer"},
        "e2e": {"value": round(us, 1), "unit": "us/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
