"""Benchmark of the W4A16 INT4 MoE expert GEMM pair on one GB300.

Metric (the pages' method: per-layer time of the gate_up GEMM plus the down
GEMM, routing and activation excluded; page "vLLM 宣布 Humming 后端可运行 …
Chord 内核 …", section "六个场景的逐层测量与限定条件"): microseconds per
layer, lower is better, plus achieved HBM GB/s and TFLOP/s against the
measured roofline.

One step = one pass of the whole path over one batch: routing alignment,
gate_up, silu_and_mul, down. The reported value is the mean over the timed
steps of the CUDA-event time of gate_up plus down, with inputs already
resident in HBM; L2 is flushed (a 256 MiB write) before every step and the
weight stream (1.19 GB at the EP8 decode shard) is larger than L2 anyway.

`--impl reference` times the float64 CPU oracle on the host cores instead,
on a bounded sample of the same workload scaled to a whole layer.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload ep8_decode|ep8_decode_e12|tp8_16|tp8_64|tp8_256|ep8_prefill|tiny
                                   |grouped_contig_{128,256,512,1024}|grouped_masked_32]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE W4A16 gate_up+down µs/layer; achieved HBM GB/s or TFLOPS vs roofline"
UNIT = "us/layer"
L2_FLUSH_BYTES = 256 << 20
PROFILES = os.path.join(ROOT, "profiles")


def make_workload(name):
    from w4a16_int4_moe_gb300 import workloads as wl
    if name == "ep8_decode":
        return wl.ep8_decode()
    if name == "ep8_decode_e12":
        # a quarter of the EP8 decode shard (12 experts, 144 rows): the size
        # that detailed profiler captures run on
        return wl.ep8_decode(tokens=144, local_experts=12)
    if name.startswith("tp8_"):
        return wl.tp8(int(name.split("_")[1]))
    if name == "ep8_prefill":
        return wl.ep8_prefill()
    if name == "tiny":
        return wl.tiny()
    raise SystemExit(f"unknown workload {name}")


def algorithmic_work(p):
    """Bytes and flops of each GEMM counted once: 0.5625 B per weight element
    of every expert that has a routed row, activations read once, outputs
    written once; flops 2 * rows * n * k over real rows only."""
    flat = p.topk_ids.reshape(-1)
    local = (flat >= 0) & (flat < p.num_experts)
    active = np.unique(flat[local]).size
    rows = int(local.sum())
    tokens_used = int(np.any((p.topk_ids >= 0) & (p.topk_ids < p.num_experts), axis=1).sum())
    h, i2, i = p.hidden, 2 * p.inter, p.inter
    wb = 0.5 + 2.0 / 32
    gu_bytes = active * i2 * h * wb + tokens_used * h * 2 + rows * i2 * 2
    dn_bytes = active * h * i * wb + rows * i * 2 + p.tokens * h * 4
    return {
        "gate_up": {"bytes": gu_bytes, "flops": 2.0 * rows * i2 * h},
        "down": {"bytes": dn_bytes, "flops": 2.0 * rows * h * i},
        "active_experts": active, "rows": rows,
    }


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


def traffic_record(kernel_file, workload):
    """ncu DRAM bytes per launch, valid only while the kernel source is the
    one the counters were taken on."""
    path = os.path.join(PROFILES, f"traffic_{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    with open(kernel_file, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    if rec.get("kernel_sha256") != sha:
        return None
    return rec


class ClockSampler:
    """nvidia-smi samples every 20 ms; only the samples whose timestamps fall
    inside the timed region are summarised."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        # the raw samples go to W4A16_CLOCKS_CSV when it is set, else to a
        # temporary file that is removed once summarised
        self.keep = "W4A16_CLOCKS_CSV" in os.environ
        self.path = os.environ.get("W4A16_CLOCKS_CSV", "")
        self.window = None

    def start(self):
        try:
            if self.keep:
                os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            else:
                fd, self.path = tempfile.mkstemp(suffix="_clocks.csv")
                os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", os.environ.get("LOCAL_RANK", "0")],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # wait (at most 3 s) for the first sample so that the timed region is covered
        t_end = time.time() + 3.0
        while time.time() < t_end:
            self.fh.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    sm, mx = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                active = [n for n, v in zip(names, parts[6:10]) if v.lower() == "active"]
                samples.append((ts, sm, mx, active))
        if not self.keep:
            os.remove(self.path)
        if not samples:
            return None
        inside = samples
        if self.window is not None:
            t0, t1 = self.window
            sel = [x for x in samples if t0 - 0.025 <= x[0] <= t1 + 0.025]
            if sel:
                inside = sel
        reasons = sorted({r for x in inside for r in x[3]})
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": max(x[2] for x in inside), "reasons": reasons,
                "samples": len(inside), "samples_total": len(samples)}


def cpu_oracle_sample(p, n_experts_sample=None):
    """Time the float64 oracle (as it stands) on a bounded sample: all routed
    rows of a subset of experts through gate_up -> act -> down; scale to a
    whole layer by the fraction of active experts sampled."""
    import oracle
    flat = p.topk_ids.reshape(-1)
    local = (flat >= 0) & (flat < p.num_experts)
    active = np.unique(flat[local])
    if n_experts_sample is None:
        n_experts_sample = active.size
    rng = np.random.default_rng(0)
    chosen = np.sort(rng.choice(active, size=n_experts_sample, replace=False))
    # the tokens routed to the sampled experts, with their other picks masked,
    # so that the per-token work also scales with the sample
    picked = np.isin(p.topk_ids, chosen)
    rows = picked.any(axis=1)
    sub_ids = np.where(picked, p.topk_ids, -1)[rows]
    x_sub, w_sub = p.x[rows], p.topk_weights[rows]
    t0 = time.perf_counter()
    g = oracle.indexed_gate_up(x_sub, sub_ids, p.q_gu, p.s_gu)
    g_bits = oracle.f64_to_bf16_bits(np.nan_to_num(g))
    a_bits = oracle.silu_and_mul(g_bits)
    oracle.indexed_down(a_bits, sub_ids, w_sub, p.q_dn, p.s_dn)
    dt = time.perf_counter() - t0
    scale = active.size / n_experts_sample
    return {"value": dt * scale * 1e6, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n_experts_sample} of {active.size} active experts (all their routed rows, "
                      f"{int(rows.sum())} tokens; gate_up+silu+down, float64 numpy), {dt:.2f} s, "
                      f"scaled x{scale:.2f}"}


def dist_setup(n_gpus):
    import torch
    import torch.distributed as dist
    if n_gpus > 1 or int(os.environ.get("WORLD_SIZE", "1")) > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist.get_rank(), dist.get_world_size(), dist
    return 0, 1, None


def reduce_max(value, dist):
    if dist is None:
        return value
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args):
    rank, world, dist = dist_setup(args.gpus)
    if rank != 0:
        return
    p = make_workload(args.workload)
    for _ in range(args.warmup):
        cpu_oracle_sample(p, n_experts_sample=1)
    vals, samples = [], None
    for _ in range(args.steps):
        rec = cpu_oracle_sample(p, n_experts_sample=args.ref_experts)
        vals.append(rec["value"])
        samples = rec
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": value / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": p.name},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": samples["cores"],
                         "kind": "oracle", "sample": samples["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_ours(args):
    import torch
    from w4a16_int4_moe_gb300 import moe as moe_mod
    from w4a16_int4_moe_gb300 import ops

    rank, world, dist = dist_setup(args.gpus)
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    ops.load_library()

    p = make_workload(args.workload)
    work = algorithmic_work(p)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    gu = moe_mod.PackedExperts.from_checkpoint(to_dev(p.q_gu), to_dev(p.s_gu.view(np.int16)))
    dn = moe_mod.PackedExperts.from_checkpoint(to_dev(p.q_dn), to_dev(p.s_dn.view(np.int16)))
    layer = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, tok_e_hint=p.tok_e_hint(), device=device)
    x = to_dev(p.x.view(np.int16)).view(torch.bfloat16)
    ids = to_dev(p.topk_ids)
    w = to_dev(p.topk_weights)
    out = torch.empty((p.tokens, p.hidden), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        flush.zero_()
        layer.align(ids)
        if ev is not None:
            ev[0].record(stream)
        layer.gate_up_gemm(x, p.tokens)
        if ev is not None:
            ev[1].record(stream)
        layer.activation(p.tokens)
        if ev is not None:
            ev[2].record(stream)
        layer.down_gemm(p.tokens, w, out)
        if ev is not None:
            ev[3].record(stream)

    clocks = ClockSampler()
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, word = ops.w4a16_read_device_status(layer.workspace)
    if st != ops.W4A16_OK:
        raise SystemExit(f"device status {word:#x} after warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(events[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    t_end_wall = time.time()
    clocks.mark(t_end_wall - wall, t_end_wall)
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    gu_us = [events[i][0].elapsed_time(events[i][1]) * 1e3 for i in range(args.steps)]
    dn_us = [events[i][2].elapsed_time(events[i][3]) * 1e3 for i in range(args.steps)]
    st, word = ops.w4a16_read_device_status(layer.workspace)
    if st != ops.W4A16_OK:
        raise SystemExit(f"device status {word:#x} after the timed steps")
    layer_us = statistics.mean(a + b for a, b in zip(gu_us, dn_us))
    layer_us = reduce_max(layer_us, dist)
    wall = reduce_max(wall, dist)
    value = layer_us / world   # replicas: world layers per step

    # ---- the layer with the activation fused into gate_up (reported
    # beside the metric; the metric itself keeps the activation untimed) ----
    fused = None
    if not args.no_fused:
        gu_glu = moe_mod.PackedExperts.from_checkpoint(
            to_dev(p.q_gu), to_dev(p.s_gu.view(np.int16)),
            layout=ops.W4A16_LAYOUT_KTILE64_GLU16)
        layer_f = moe_mod.W4A16MoE(gu_glu, dn, p.topk, p.tokens, tok_e_hint=p.tok_e_hint(),
                                   device=device)
        nf = max(20, args.steps // 4)
        ev_f = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(nf)]
        for i in range(args.warmup + nf):
            e = ev_f[i - args.warmup] if i >= args.warmup else None
            flush.zero_()
            layer_f.align(ids)
            layer.align(ids)
            if e is not None:
                e[0].record(stream)
            layer_f.gate_up_act(x, p.tokens)
            if e is not None:
                e[1].record(stream)
            layer_f.down_gemm(p.tokens, w, out)
            if e is not None:
                e[2].record(stream)
            flush.zero_()
            if e is not None:
                e[3].record(stream)
            layer.gate_up_gemm(x, p.tokens)
            layer.activation(p.tokens)
            layer.down_gemm(p.tokens, w, out)
            if e is not None:
                e[4].record(stream)
        torch.cuda.synchronize()
        st, word = ops.w4a16_read_device_status(layer_f.workspace)
        if st != ops.W4A16_OK:
            raise SystemExit(f"device status {word:#x} in the fused-activation layer")
        fused = {
            "gate_up_silu_us": statistics.mean(e[0].elapsed_time(e[1]) * 1e3 for e in ev_f),
            "down_us": statistics.mean(e[1].elapsed_time(e[2]) * 1e3 for e in ev_f),
            "layer_with_act_us": statistics.mean(e[0].elapsed_time(e[2]) * 1e3 for e in ev_f),
            "unfused_layer_with_act_us": statistics.mean(e[3].elapsed_time(e[4]) * 1e3
                                                         for e in ev_f),
            "steps": nf,
        }

    # ---- end to end through the public call, host buffers: the layer a user
    # builds, with the activation fused into gate_up when measured above ----
    e2e_layer = layer_f if fused is not None else layer
    x_h = torch.from_numpy(p.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    ids_h = torch.from_numpy(p.topk_ids).pin_memory()
    w_h = torch.from_numpy(p.topk_weights).pin_memory()
    out_h = torch.empty((p.tokens, p.hidden), dtype=torch.float32).pin_memory()
    x_d, ids_d, w_d = torch.empty_like(x), torch.empty_like(ids), torch.empty_like(w)

    def e2e_step():
        x_d.copy_(x_h, non_blocking=True)
        ids_d.copy_(ids_h, non_blocking=True)
        w_d.copy_(w_h, non_blocking=True)
        e2e_layer.forward(x_d, ids_d, w_d, out=out)
        out_h.copy_(out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        flush.zero_()
        e2e_step()
    torch.cuda.synchronize()
    e2e_times = []
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e2e_times.append(e0.elapsed_time(e1) * 1e3)
    e2e_us = reduce_max(statistics.mean(e2e_times), dist) / world
    h2d = p.x.nbytes + p.topk_ids.nbytes + p.topk_weights.nbytes
    d2h = p.tokens * p.hidden * 4

    if rank != 0:
        return
    hbm, tflops_peak, peak_src = measured_peaks()
    gu_mean = statistics.mean(gu_us)
    dn_mean = statistics.mean(dn_us)
    gu_gbs = work["gate_up"]["bytes"] / (gu_mean * 1e-6) / 1e9
    dn_gbs = work["down"]["bytes"] / (dn_mean * 1e-6) / 1e9
    total_bytes = work["gate_up"]["bytes"] + work["down"]["bytes"]
    total_flops = work["gate_up"]["flops"] + work["down"]["flops"]
    traffic = traffic_record(os.path.join(ROOT, "w4a16_int4_moe_gb300", "csrc", "moe_gemm.cu"),
                             args.workload)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random uint4 weights, N(0,1) activations)",
        "config": {
            "workload": p.name, "tokens": p.tokens, "hidden": p.hidden, "inter": p.inter,
            "local_experts": p.num_experts, "topk": p.topk, "routed_rows": work["rows"],
            "active_experts": work["active_experts"], "block_m": layer.block_m,
            "l2": "flushed before every step (256 MiB write); the weight stream exceeds L2",
            "parallelism": f"replicas x{world}",
        },
        "gate_up_us": gu_mean, "down_us": dn_mean,
        "achieved": {"hbm_gbs": total_bytes / (layer_us * 1e-6) / 1e9,
                     "tflops": total_flops / (layer_us * 1e-6) / 1e12,
                     "gate_up_gbs": gu_gbs, "down_gbs": dn_gbs},
        "roofline": {
            "bound": "hbm", "kernel": "w4a16_moe_gemm_kernel (gate_up)",
            "achieved": gu_gbs, "peak": hbm, "unit": "GB/s", "frac": gu_gbs / hbm,
            "peak_source": f"{peak_src} hbm_gbs",
            "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
            "algorithmic_bytes": work["gate_up"]["bytes"],
        },
        "gpu_launches": 6 * args.steps,  # align, permute + gate_up, silu, permute + down
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "call": "W4A16MoE.forward (align, gate_up with fused activation, down)"
                        if fused is not None else "W4A16MoE.forward (align, gate_up, act, down)"},
        "clocks": clk,
        "fused_activation": fused,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(p)
    print(json.dumps(line))


def make_grouped(name):
    """Grouped-layout workloads on the EP8 shard: the gate_up-shaped and the
    down-shaped GEMM over the same per-expert rows (random activations)."""
    from w4a16_int4_moe_gb300 import workloads as wl
    if name.startswith("grouped_contig_"):
        m = int(name.split("_")[-1])
        gu = wl.grouped_contiguous_problem(m, 48, 4096, 7168, seed=1)
        dn = wl.grouped_contiguous_problem(m, 48, 7168, 2048, seed=2)
        return gu, dn, f"grouped_contiguous_E48_m{m}_H7168_I2048"
    if name == "grouped_masked_32":
        gu = wl.grouped_masked_problem(48, 32, 4096, 7168, seed=1)
        dn = wl.grouped_masked_problem(48, 32, 7168, 2048, seed=2)
        dn.layout[:] = gu.layout          # the same rows in both GEMMs
        return gu, dn, "grouped_masked_E48_budget32_H7168_I2048"
    raise SystemExit(f"unknown workload {name}")


def run_grouped(args):
    """One step = the grouped gate_up GEMM then the grouped down GEMM (the
    activation between them untimed), L2 flushed before each step."""
    import torch
    from w4a16_int4_moe_gb300 import ops
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    ops.load_library()
    gu, dn, wname = make_grouped(args.workload)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    calls = []
    for gp in (gu, dn):
        pk = ops.w4a16_prepack(to_dev(gp.q), to_dev(gp.s.view(np.int16)))
        a = to_dev(gp.a.view(np.int16)).view(torch.bfloat16)
        lay = to_dev(gp.layout)
        kind = ops.W4A16_GROUPED_CONTIGUOUS if gp.kind == "contiguous" else ops.W4A16_GROUPED_MASKED
        m = gp.a.shape[0] if gp.kind == "contiguous" else gp.a.shape[1]
        shape = (m, gp.n) if gp.kind == "contiguous" else (gp.num_experts, m, gp.n)
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        ws = torch.zeros(256, dtype=torch.uint8, device=device)
        calls.append((gp, kind, pk, a, m, lay, ws, out))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def run(c):
        gp, kind, pk, a, m, lay, ws, out = c
        ops.w4a16_moe_grouped_gemm(kind, pk, gp.num_experts, gp.n, gp.k, a, m, lay, ws,
                                   expected_m=gp.expected_m, out=out)

    for _ in range(args.warmup):
        flush.zero_()
        run(calls[0])
        run(calls[1])
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler()
    clocks.start()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        run(calls[0])
        ev[i][1].record(stream)
        run(calls[1])
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks.mark(time.time() - wall, time.time())
    clk = clocks.stop()
    for c in calls:
        st, word = ops.w4a16_read_device_status(c[6])
        if st != ops.W4A16_OK:
            raise SystemExit(f"device status {word:#x}")
    gu_us = statistics.mean(e[0].elapsed_time(e[1]) * 1e3 for e in ev)
    dn_us = statistics.mean(e[1].elapsed_time(e[2]) * 1e3 for e in ev)
    rows = gu.valid_rows()
    wb = 0.5 + 2.0 / 32
    act_e = 48 if gu.kind == "contiguous" else int((gu.layout > 0).sum())
    gu_bytes = act_e * 4096 * 7168 * wb + rows * 7168 * 2 + rows * 4096 * 2
    dn_bytes = act_e * 7168 * 2048 * wb + rows * 2048 * 2 + rows * 7168 * 2
    gu_flops, dn_flops = 2.0 * rows * 4096 * 7168, 2.0 * rows * 7168 * 2048
    hbm, tflops_peak, peak_src = measured_peaks()
    layer_us = gu_us + dn_us
    tensor = gu.kind == "contiguous"
    if tensor:
        ach = gu_flops / (gu_us * 1e-6) / 1e12
        roof = {"bound": "tensor", "kernel": "w4a16_moe_gemm_kernel (grouped gate_up)",
                "achieved": ach, "peak": tflops_peak, "unit": "TFLOP/s", "frac": ach / tflops_peak,
                "peak_source": f"{peak_src} bf16_tflops", "traffic": None}
    else:
        ach = gu_bytes / (gu_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "kernel": "w4a16_moe_gemm_kernel (grouped gate_up)",
                "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_source": f"{peak_src} hbm_gbs", "traffic": None,
                "algorithmic_bytes": gu_bytes}
    line = {
        "metric": METRIC, "value": layer_us, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random uint4 weights, N(0,1) activations)",
        "config": {"workload": wname, "valid_rows": rows, "experts": 48,
                   "l2": "flushed before every step (256 MiB write)"},
        "gate_up_us": gu_us, "down_us": dn_us,
        "achieved": {"tflops": (gu_flops + dn_flops) / (layer_us * 1e-6) / 1e12,
                     "hbm_gbs": (gu_bytes + dn_bytes) / (layer_us * 1e-6) / 1e9},
        "roofline": roof, "gpu_launches": 2 * args.steps, "clocks": clk,
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ep8_decode")
    ap.add_argument("--ref-experts", type=int, default=2,
                    help="experts per reference step (bounded CPU sample)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fused", action="store_true",
                    help="skip the fused-activation layer measurement")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload.startswith("grouped_"):
        run_grouped(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
