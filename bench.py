"""Benchmark: exact attention forward + backward on GB300.

One step = one forward and one backward pass (every kernel of the path) over
the bf16 B=8 H=32 N=4096 d=128 non-causal workload, inputs resident in HBM.
The metric is whole-job TFLOP/s with FLOPs counted as 4*B*H*N^2*d for the
forward and 2.5x that for the backward (halved under a causal mask).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). Multi-GPU runs come from torchrun, one process
per GPU; every (batch, head) is independent, so each rank runs its own copy
of the workload (weak scaling, no collective on the data path).

--impl reference times the fp64 CPU oracle on this machine's host cores on a
bounded sample of the same workload (whole heads, full N), in the same metric.
"""
from __future__ import annotations

import argparse
import ctypes
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

METRIC = "attention fwd/bwd TFLOP/s at B8 H32 N4096 d128 bf16; % of BF16 tensor peak"
METRIC_FWD = "attention forward TFLOP/s (forward-only run of the workload in config); % of BF16 tensor peak"

# DRAM bytes per launch of the dominant kernel at the headline size, from an
# ncu capture of a quarter-size case of the same kernel (the traffic scales
# with the number of heads). Only valid for the kernel source it was measured
# on: reported as null once that file changes.
MEASURED_TRAFFIC = {"workload": "bf16_B8_H32_N4096_d128", "kernel": "bwd_dkdv_kernel<128>",
                    "bytes": 4 * (270.915072e6 + 103.886592e6),
                    "source": "exact_attention_97_gb300/csrc/bwd_tc.cu", "sha256_16": "567d2c49096803e5"}


def _measured_traffic(kernel: str, workload: str):
    import hashlib
    m = MEASURED_TRAFFIC
    if kernel != m["kernel"] or workload != m["workload"]:
        return None
    try:
        with open(os.path.join(ROOT, m["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != m["sha256_16"]:
                return None
    except OSError:
        return None
    return m["bytes"]


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": p["bf16_tflops"], "bf16_tflops_sustained": p.get("bf16_tflops_sustained"),
                "hbm_gbs": p["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _host_info(local: int):
    """Where the host side sits relative to the GPU (for reading e2e copy rates)."""
    info = {"cpus_in_affinity": len(os.sched_getaffinity(0))}
    try:
        bus = subprocess.run(["nvidia-smi", f"--id={local}", "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=10).stdout.strip() or None
        if bus:
            dom = bus.lower()
            if dom.count(":") == 2 and len(dom.split(":")[0]) == 8:
                dom = dom[4:]
            path = f"/sys/bus/pci/devices/{dom}/numa_node"
            if os.path.exists(path):
                info["gpu_numa_node"] = int(open(path).read().strip())
            info["gpu_pci_bus_id"] = bus
    except Exception as exc:  # informational only
        info["error"] = str(exc)[:100]
    return info


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_baseline(w, heads: int):
    """Oracle fwd+bwd on `heads` whole heads of the workload (full N and Nk)."""
    import torch

    import oracle
    from exact_attention_97_gb300.inputs import make_qkv_do

    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    q, _, _, dO = make_qkv_do(1, heads, w.N, w.d, w.seed, dt)
    _, k, v, _ = make_qkv_do(1, heads, w.n_keys, w.d, w.seed, dt)
    f64 = lambda t: t.float().double().numpy()  # noqa: E731
    q, k, v, dO = f64(q), f64(k), f64(v), f64(dO)
    oracle.build()
    t0 = time.perf_counter()
    oracle.attention_fwd_kv(q, k, v, w.scale, w.causal)
    oracle.attention_bwd_kv(q, k, v, dO, w.scale, w.causal)
    dt_s = time.perf_counter() - t0
    flops = (w.flops_fwd() + w.flops_bwd()) / (w.B * w.H) * heads
    return {"value": flops / dt_s / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{heads} whole heads (full N={w.N}, Nk={w.n_keys}, d={w.d}) of the workload, fwd+bwd, "
                      f"fp64, {dt_s:.1f} s wall"}


def cpu_baseline_sampled_rows(w, rows: int = 256):
    """Oracle on `rows` seeded query rows of a workload too large for whole
    heads (the long causal one): O, L and dQ of each sampled row, as the parity
    test computes them. The rate counts the flops those rows execute (S, O, dP
    and dQ: 8 d per visible (query, key) pair); the full problem's time is a
    linear extrapolation of its algorithmic flops at that rate."""
    import torch

    import oracle
    from exact_attention_97_gb300.inputs import make_qkv_do, sample_indices

    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    q, k, v, dO = make_qkv_do(w.B, w.H, w.N, w.d, w.seed, dt)
    flat = sample_indices(w.B * w.H * w.N, rows, seed=5).numpy()
    by_head = {}
    for idx in flat:
        by_head.setdefault(int(idx // w.N), []).append(int(idx % w.N))
    oracle.build()
    f64 = lambda t: t.float().double().numpy()  # noqa: E731
    off = w.n_keys - w.N
    t_total, flops = 0.0, 0.0
    for bh, rr in by_head.items():
        b, h = divmod(bh, w.H)
        qh, kh, vh, doh = (f64(x[b, h]) for x in (q, k, v, dO))
        t0 = time.perf_counter()
        oracle.query_rows(qh, kh, vh, doh, rr, w.scale, w.causal)
        t_total += time.perf_counter() - t0
        flops += sum(8.0 * w.d * (min(w.n_keys, i + 1 + off) if w.causal else w.n_keys) for i in rr)
    rate = flops / t_total
    full = w.flops_fwd() + w.flops_bwd()
    return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{rows} seeded query rows of {w.name} (O, L, dQ at full N={w.N}), fp64, "
                      f"{t_total:.2f} s wall; rate = executed flops (8 d per visible pair) / time",
            "full_problem_s_extrapolated": full / rate,
            "extrapolation": "linear: the workload's fwd+bwd algorithmic flops at the sample's rate"}


def run_reference(args, w):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    times = []
    base = None
    for step in range(args.warmup + args.steps):
        b = cpu_baseline(w, args.ref_heads)
        if step >= args.warmup:
            times.append(b)
        base = b
    vals = [b["value"] for b in times]
    value = statistics.median(vals)
    flops_step = (w.flops_fwd() + w.flops_bwd()) / (w.B * w.H) * args.ref_heads
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": flops_step / (value * 1e12) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "sample_heads_per_step": args.ref_heads},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": base["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import exact_attention_97_gb300 as fa
    from exact_attention_97_gb300.inputs import make_qkv_do
    from exact_attention_97_gb300.shard import head_range, max_over_ranks

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    fa.load()

    # inputs: seeded host tensors, pinned copies for the end-to-end leg, device copies.
    # Weak scaling: the whole job is world x (B x H) independent heads; this
    # rank owns its contiguous block of B x H of them, seeded by the block's
    # offset (rank 0 keeps the workload's own seeds).
    lo, _ = head_range(world * w.B * w.H, rank, world)
    seed = w.seed + 4 * lo
    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    q_h, _, _, do_h = make_qkv_do(w.B, w.H, w.N, w.d, seed, dt)
    _, k_h, v_h, _ = make_qkv_do(w.B, w.H, w.n_keys, w.d, seed, dt)
    q_h, k_h, v_h, do_h = (t.pin_memory() for t in (q_h, k_h, v_h, do_h))
    q, k, v, dO = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d, fa.FA_BF16)
    if args.dropout and not args.dropout_saved:  # room for the keep bits the dK/dV pass hands to the dQ pass
        need = fa.fa_bwd_dropout_workspace_size(w.B, w.H, w.N, w.n_keys, w.d, fa.FA_BF16)
    ws = torch.empty(need, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream()

    drop = {"dropout_p": args.dropout, "seed": 1234, "offset": 0} if args.dropout else {}
    drop_bwd = dict(drop)
    if args.dropout and args.dropout_saved:  # the forward saves its keep bits, the backward reads them
        mask = fa.dropout_mask_buffer(w.B, w.H, w.N, w.n_keys, dev)
        drop["dropout_mask"] = mask
        drop_bwd = {"dropout_p": args.dropout, "dropout_mask": mask}
    launches = [0]
    marks = []  # (fwd start, bwd start, bwd end) events per timed step, on the launch stream

    def step(mark=False):
        if mark:
            m = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            m[0].record(stream)
        fa.attention_forward(q, k, v, w.scale, w.causal, out=o, lse=lse, **drop)
        n = fa.fa_last_launch_count()
        if mark:
            m[1].record(stream)
        if not args.fwd_only:
            fa.attention_backward(q, k, v, o, lse, dO, w.scale, w.causal, workspace=ws, grads=(dq, dk, dv),
                                  **drop_bwd)
        if mark:
            m[2].record(stream)
            marks.append(m)
        launches[0] += n + (0 if args.fwd_only else fa.fa_last_launch_count())

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.fa_device_status() != 0:
        raise RuntimeError("kernel pipeline timeout during warm-up")

    # per-kernel events recorded by the library around each tensor-core kernel:
    # per step, pair 3s = forward, 3s+1 = dK/dV pass, 3s+2 = dQ pass (one pair
    # per step with --fwd-only)
    per = 1 if args.fwd_only else 3
    pairs = per * args.steps
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * pairs)]
    for e in evs:
        e.record(stream)  # creates the underlying CUDA event
    handles = (ctypes.c_void_p * (2 * pairs))(*[e.cuda_event for e in evs])
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    sampler.start()
    time.sleep(0.3)
    fa.fa_set_kernel_timing(handles, pairs)
    launches[0] = 0
    start.record(stream)
    for _ in range(args.steps):
        step(mark=True)
    stop.record(stream)
    torch.cuda.synchronize()
    fa.fa_set_kernel_timing(None, 0)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    if fa.fa_device_status() != 0:
        raise RuntimeError("kernel pipeline timeout in the timed region")
    ms = start.elapsed_time(stop)
    peak_mem = torch.cuda.max_memory_allocated(dev)
    timed_launches = launches[0]  # the graph and end-to-end sections below launch more

    def pair_ms(i):
        return statistics.mean(evs[2 * (per * s + i)].elapsed_time(evs[2 * (per * s + i) + 1])
                               for s in range(args.steps))

    k_fwd = pair_ms(0)
    k_dkdv, k_dq = (None, None) if args.fwd_only else (pair_ms(1), pair_ms(2))
    # per-call windows: the median over steps, so that one host stall in the
    # timed loop (the GPU waiting for a launch) does not stand for every step;
    # the headline value keeps the whole timed region
    fwd_call = statistics.median(m[0].elapsed_time(m[1]) for m in marks)
    bwd_call = None if args.fwd_only else statistics.median(m[1].elapsed_time(m[2]) for m in marks)
    step_ms = sorted(m[0].elapsed_time(m[2]) for m in marks)  # whole step, per timed step
    ms = max_over_ranks(ms, dev)

    flops_step = w.flops_fwd() + (0 if args.fwd_only else w.flops_bwd())
    value = flops_step * world * args.steps / (ms * 1e-3) / 1e12
    peaks = _peaks()
    peak = peaks["bf16_tflops"]
    F = w.flops_fwd()  # two contractions (QK^T, PV) over the pairs in the mask

    def tf(flops, t_ms):
        return flops / (t_ms * 1e-3) / 1e12

    # Algorithmic flops per kernel: the backward's five contractions are split
    # as S, dP, dV, dK in the dK/dV pass (2F) and dQ in the dQ pass (F/2); the
    # dQ pass also recomputes S and dP (executed 3F/2).
    kernels = {"fwd_kernel": {"ms": k_fwd, "algo_tflops": tf(F, k_fwd), "frac": tf(F, k_fwd) / peak}}
    dom = ("fwd_kernel", F, k_fwd)
    if not args.fwd_only:
        kernels["bwd_dkdv_kernel"] = {"ms": k_dkdv, "algo_tflops": tf(2 * F, k_dkdv),
                                      "frac": tf(2 * F, k_dkdv) / peak}
        kernels["bwd_dq_kernel"] = {"ms": k_dq, "algo_tflops": tf(0.5 * F, k_dq),
                                    "executed_tflops": tf(1.5 * F, k_dq), "executed_frac": tf(1.5 * F, k_dq) / peak}
        dom = max(("fwd_kernel", F, k_fwd), ("bwd_dkdv_kernel", 2 * F, k_dkdv),
                  ("bwd_dq_kernel", 0.5 * F, k_dq), key=lambda x: x[2])
    achieved = tf(dom[1], dom[2])
    roofline = {"bound": "tensor", "kernel": f"{dom[0]}<{w.d}>", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": args.traffic if args.traffic is not None else _measured_traffic(f"{dom[0]}<{w.d}>", w.name),
                "peak_source": peaks["source"] + " burst bf16 (cuBLAS), of measured"}
    # Algorithmic HBM bytes per step (each tensor read or written once; L, D
    # and the padded row terms as fp32): the bound of the small, latency-
    # and launch-bound configurations.
    e = 2  # bytes per 16-bit element
    rows_q, rows_k = w.B * w.H * w.N, w.B * w.H * w.n_keys
    bytes_fwd = (rows_q * 2 + rows_k * 2) * w.d * e + rows_q * 4             # Q, K, V in; O, L out
    bytes_bwd = (rows_q * 4 + rows_k * 4) * w.d * e + rows_q * 4 * 3         # Q,K,V,O,dO in; dQ,dK,dV out; L, D
    step_bytes = bytes_fwd + (0 if args.fwd_only else bytes_bwd)
    hbm = {"achieved_gbs": step_bytes * args.steps / (ms * 1e-3) / 1e9, "peak_gbs": peaks["hbm_gbs"],
           "frac": step_bytes * args.steps / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], "bytes_per_step": step_bytes,
           "peak_source": peaks["source"] + " copy bandwidth, of " + peaks["source"]}
    fwd_tf = tf(w.flops_fwd(), fwd_call)
    bwd_tf = None if args.fwd_only else tf(w.flops_bwd(), bwd_call)

    def quantile(xs, p):  # nearest-rank on sorted values
        return xs[min(len(xs) - 1, max(0, int(round(p * (len(xs) - 1)))))]
    spread = {"ms_median": statistics.median(step_ms), "ms_p10": quantile(step_ms, 0.1),
              "ms_p90": quantile(step_ms, 0.9),
              "value_median": tf(flops_step, statistics.median(step_ms)) * world,
              "value_p10": tf(flops_step, quantile(step_ms, 0.9)) * world,
              "value_p90": tf(flops_step, quantile(step_ms, 0.1)) * world,
              "note": "per timed step, fwd start to bwd end on the launch stream (rank 0); value_p10 is "
                      "the 10th-percentile throughput (from the 90th-percentile step time)"}

    # the same step replayed from a CUDA graph (one capture of the forward and
    # backward calls on these buffers): what is left of the step once the
    # host's per-call cost is off the critical path (small shapes)
    graph = None
    if args.graph:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(args.steps, 20)
        ga.record(stream)
        for _ in range(reps):
            g.replay()
        gb.record(stream)
        torch.cuda.synchronize()
        if fa.fa_device_status() != 0:
            raise RuntimeError("kernel pipeline timeout in the graph replays")
        gms = ga.elapsed_time(gb) / reps
        graph = {"ms_per_step": gms, "value": flops_step * world / (gms * 1e-3) / 1e12, "unit": "TFLOP/s",
                 "replays": reps, "note": "one captured step (every kernel of the forward and backward), replayed"}

    # end to end through the public API: pinned host inputs in, results back to pinned host.
    # The training step goes through attention_step_host, which streams chunks of heads
    # through the GPU (copy in, compute, copy out on three streams).
    e2e = None
    if not args.no_e2e:
        if args.fwd_only:
            out_h = [torch.empty_like(q_h).pin_memory(),
                     torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()]
        else:
            out_h = [torch.empty_like(q_h).pin_memory(),
                     torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory(),
                     torch.empty_like(q_h).pin_memory(), torch.empty_like(k_h).pin_memory(),
                     torch.empty_like(v_h).pin_memory()]

        drop_e2e = {k_: v_ for k_, v_ in drop.items() if k_ != "dropout_mask"}  # chunks draw their bits

        def e2e_step():
            if args.fwd_only:
                qd, kd, vd = (t.to(dev, non_blocking=True) for t in (q_h, k_h, v_h))
                od, ld = fa.attention_forward(qd, kd, vd, w.scale, w.causal, **drop_e2e)
                for dst, src in zip(out_h, (od, ld)):
                    dst.copy_(src, non_blocking=True)
            else:
                fa.attention_step_host(q_h, k_h, v_h, do_h, w.scale, w.causal, out=tuple(out_h), **drop_e2e)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e2e_steps = max(3, min(args.steps, 10))
        # every step bracketed by its own events on the caller's stream (the
        # step's streams join it): the median step is the value, so a single
        # host stall does not stand for the run
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
        if world > 1:
            dist.barrier()
        ev[0].record(stream)
        for i in range(e2e_steps):
            e2e_step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        per_step = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(e2e_steps))
        e2e_mean = ev[0].elapsed_time(ev[-1]) / e2e_steps
        ems = statistics.median(per_step) * e2e_steps
        ems = max_over_ranks(ems, dev)
        bytes_in = sum(t.numel() * t.element_size() for t in ((q_h, k_h, v_h) if args.fwd_only else
                                                                (q_h, k_h, v_h, do_h)))
        bytes_out = sum(t.numel() * t.element_size() for t in out_h)
        # the link alone: each direction timed by itself on the same pinned
        # buffers (whole tensors, one copy each), so the e2e time can be read
        # against its copy-bound floor
        ins_h = (q_h, k_h, v_h) if args.fwd_only else (q_h, k_h, v_h, do_h)
        dev_in = [torch.empty_like(t, device=dev) for t in ins_h]
        dev_out = [torch.empty_like(t, device=dev) for t in out_h]

        def timed_copies(pairs, reps=3):
            best = None
            for _ in range(reps):
                a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a2.record(stream)
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
                b2.record(stream)
                torch.cuda.synchronize()
                t = a2.elapsed_time(b2)
                best = t if best is None else min(best, t)
            return best
        h2d_ms = timed_copies(list(zip(dev_in, ins_h)))
        d2h_ms = timed_copies(list(zip(out_h, dev_out)))

        def both_at_once(reps=3):  # inputs in on one stream while outputs go out on another
            sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
            best = None
            for _ in range(reps):
                a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a2.record(stream)
                sa.wait_stream(stream)
                sb.wait_stream(stream)
                with torch.cuda.stream(sa):
                    for dst, src in zip(dev_in, ins_h):
                        dst.copy_(src, non_blocking=True)
                with torch.cuda.stream(sb):
                    for dst, src in zip(out_h, dev_out):
                        dst.copy_(src, non_blocking=True)
                stream.wait_stream(sa)
                stream.wait_stream(sb)
                b2.record(stream)
                torch.cuda.synchronize()
                t = a2.elapsed_time(b2)
                best = t if best is None else min(best, t)
            return best
        both_ms = both_at_once()
        del dev_in, dev_out
        h2d_gbs, d2h_gbs = bytes_in / (h2d_ms * 1e-3) / 1e9, bytes_out / (d2h_ms * 1e-3) / 1e9
        e2e = {"value": flops_step * world * e2e_steps / (ems * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": bytes_in, "d2h_bytes_per_step": bytes_out,
               "ms_per_step": ems / e2e_steps,
               "ms_per_step_min_median_max_mean": [per_step[0], statistics.median(per_step), per_step[-1],
                                                   e2e_mean],
               "h2d_gbs_alone": h2d_gbs, "d2h_gbs_alone": d2h_gbs,
               "copy_ms_alone": {"h2d": h2d_ms, "d2h": d2h_ms},
               "copy_ms_both_directions_at_once": both_ms,
               "floor_ms": max(both_ms, ms / args.steps),
               "floor_note": "the step cannot beat the slower of: all inputs in while all outputs go out (two "
                             "streams at once), the device-resident step; the chunked pipeline overlaps the two",
               "host": _host_info(local)}

    base, base_long = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.fwd_only and not args.dropout:
        base = cpu_baseline(w, args.cpu_heads)
        if not args.shape and not args.workload:
            from exact_attention_97_gb300.inputs import WORKLOADS
            wl = WORKLOADS["bf16_causal_B1_H32_N65536_d128"]
            base_long = {wl.name: cpu_baseline_sampled_rows(wl)}

    if rank == 0:
        line = {
            "metric": METRIC_FWD if args.fwd_only else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "Nk": w.n_keys, "d": w.d,
                       "causal": w.causal, "dropout": args.dropout,
                       "dropout_bits": ("saved by the forward" if args.dropout_saved else "drawn in every pass")
                       if args.dropout else None,
                       "inputs": "i.i.d. N(0,1), seeds Q=0 K=1 V=2 dO=3",
                       "l2": "inputs larger than L2 (each of Q, K, V, dO is "
                             f"{q.numel() * 2 / 1e6:.0f} MB vs 129 MB L2)",
                       "parallelism": f"{world} rank(s), {w.B * w.H} heads each (heads sharded), no collective"},
            "pct_of_peak": value / (peak * world) * 100.0,
            "fwd": {"ms": fwd_call, "tflops": fwd_tf, "frac": fwd_tf / peak},
            "bwd": None if args.fwd_only else {"ms": bwd_call, "tflops": bwd_tf, "frac": bwd_tf / peak},
            "kernels": kernels,
            "roofline": roofline,
            "hbm": hbm,
            "cpu_baseline": base,
            "cpu_baseline_other_workloads": base_long,
            "spread": spread,
            "graph": graph,
            "peak_mem_bytes": peak_mem,
            "peak_mem_note": "torch.cuda.max_memory_allocated over the timed region: inputs, outputs and the "
                             f"backward workspace ({need} bytes); the library allocates nothing itself",
            "e2e": e2e,
            "gpu_launches": timed_launches,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="workload name (default: the headline)")
    ap.add_argument("--shape", default=None,
                    help="B,H,N,d[,causal]: another case of the same kernels (profiling, other shapes)")
    ap.add_argument("--nk", type=int, default=0, help="key/value rows per head for --shape (default N)")
    ap.add_argument("--dtype", choices=["bf16", "f16"], default="bf16", help="16-bit input type for --shape")
    ap.add_argument("--fwd-only", action="store_true",
                    help="time the forward alone (head sizes with no backward kernel, e.g. d = 256)")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="dropout probability on the attention probabilities (Philox mask, seed 1234)")
    ap.add_argument("--dropout-saved", action="store_true",
                    help="with --dropout: the forward saves its keep bits and the backward reads them")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step replayed from a CUDA graph (host launch cost off the critical path)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-heads", type=int, default=8, help="heads in the CPU-baseline sample")
    ap.add_argument("--ref-heads", type=int, default=2, help="heads per step of --impl reference")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args()
    from exact_attention_97_gb300.inputs import HEADLINE, WORKLOADS, Workload
    w = WORKLOADS[args.workload or HEADLINE]
    if args.shape:
        vals = [int(x) for x in args.shape.split(",")]
        B, H, N, d = vals[:4]
        causal = bool(vals[4]) if len(vals) > 4 else False
        kv = f"_Nk{args.nk}" if args.nk else ""
        w = Workload(f"{args.dtype}{'_causal' if causal else ''}_B{B}_H{H}_N{N}{kv}_d{d}", args.dtype, B, H, N, d,
                     causal, Nk=args.nk)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
